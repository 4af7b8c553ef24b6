"""CPU tests of bench.py's host logic: the algorithmic byte and FLOP counts per
token-head, the state bytes of each workload, the traffic record that stays valid
only while the kernel sources match, and the parsing of the nvidia-smi clock
samples (throttle reasons, one GPU's rows, median clock)."""
import json
import os
import shutil
import types

import torch

import bench
from kda_prefill_gb300 import workloads as wl

PLANE_F32 = 128 * 128 * 4


def _fake(lengths, flags, H, dtype):
    """The fields state_bytes reads, without drawing a full workload."""
    return types.SimpleNamespace(lengths=list(lengths), num_seqs=len(lengths), num_heads=H,
                                 has_initial_state=torch.tensor(flags, dtype=torch.bool),
                                 state_pool=torch.empty(0, dtype=dtype))


def test_per_token_head_counts():
    # q, k, v, out bf16 (256 B each), raw gate fp32 (512 B), raw beta fp32 (4 B)
    assert bench.BYTES_PER_TOKHEAD == 4 * 256 + 512 + 4 == 1540
    assert bench.INTRA_BYTES_PER_TOKHEAD + bench.SCAN_BYTES_PER_TOKHEAD == bench.BYTES_PER_TOKHEAD
    assert bench.RAW_BF16_SAVING == 128 * 2 + 2
    # 2 (5 C^2 d + 3 C d^2) / C at C = 64, d = 128
    assert bench.FLOP_PER_TOKHEAD == 180224


def test_state_bytes_of_the_tiny_case():
    w = wl.tiny_varlen()  # 37, 0, 59 tokens, H = 2, flags 1, 0, 1, fp32 pool
    assert bench.state_bytes(w) == (2 + 3) * 2 * PLANE_F32
    assert bench.BYTES_PER_TOKHEAD * w.total_tokens * w.num_heads == 295680
    assert bench.state_bytes(w, only_long=True) == (2 + 2) * 2 * PLANE_F32  # the empty one is short
    assert bench.long_tokens(w) == 96


def test_state_bytes_of_the_prefills():
    w = _fake([16384], [0], 12, torch.float32)
    assert bench.state_bytes(w) == 786432
    assert bench.BYTES_PER_TOKHEAD * 16384 * 12 + bench.state_bytes(w) == 303562752
    w = _fake([4096], [1], 12, torch.float32)
    assert bench.BYTES_PER_TOKHEAD * 4096 * 12 + bench.state_bytes(w) == 75694080 + 2 * 786432


def test_state_bytes_of_the_mixed_batch():
    lengths = [1] * 512 + [2048] * 4
    w = _fake(lengths, [1] * 512 + [0] * 4, 12, torch.bfloat16)
    plane = 12 * 128 * 128 * 2
    assert plane == 393216
    assert bench.state_bytes(w) == 512 * plane + 516 * plane
    assert bench.BYTES_PER_TOKHEAD * sum(lengths) * 12 == 160849920
    assert bench.state_bytes(w, only_long=True) == 4 * plane
    assert bench.long_tokens(w) == 4 * 2048


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    """A traffic record applies only to the workload it was taken on and only
    while the hash of its kernel sources is the one it records."""
    import hashlib
    srcs = ["kda_prefill_gb300/csrc/kda_intra_tc.cu", "kda_prefill_gb300/csrc/kda_scan_walk.cuh"]
    (tmp_path / "profiles").mkdir()
    h = hashlib.sha256()
    for s in srcs:
        (tmp_path / s).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, s), tmp_path / s)
        h.update(open(tmp_path / s, "rb").read())
    rec = {"kda_fused": {"dram_bytes_per_launch": 123456, "workload": "prefill_16k",
                         "source": srcs, "source_sha": h.hexdigest()[:16]}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("kda_fused", "prefill_16k") == 123456
    assert bench.load_traffic("kda_fused", "another_workload") is None
    assert bench.load_traffic("kda_intra", "prefill_16k") is None
    with open(tmp_path / srcs[-1], "a") as f:
        f.write("\n// changed\n")
    assert bench.load_traffic("kda_fused", "prefill_16k") is None


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, lines, uuid):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(line + "\n" for line in lines))
    s = bench.ClockSampler(uuid)
    s.proc, s.path = _DoneProc(), str(path)
    return s


def test_clock_samples_of_one_gpu_and_their_reasons(tmp_path):
    ok = "Not Active"
    lines = [
        f"0, GPU-a, 2070, 2070, 900.1, 0x0, {ok}, {ok}, {ok}, {ok}",
        f"0, GPU-a, 1950, 2070, 1390.0, 0x4, {ok}, {ok}, {ok}, Active",
        f"0, GPU-a, 2070, 2070, 1200.0, 0x0, {ok}, {ok}, {ok}, {ok}",
        f"1, GPU-b, 900, 2070, 300.0, 0x8, Active, {ok}, {ok}, {ok}",  # another GPU
        "garbled line",
    ]
    got = _sampler_with(tmp_path, lines, "GPU-a").stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    got = _sampler_with(tmp_path, lines, None).stop()  # no uuid: every row counts
    assert got["reasons"] == ["hw_slowdown", "sw_power_cap"] and got["samples"] == 4
