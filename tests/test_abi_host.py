"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every symbol include/kda.h declares, the chunk numbering matches the
repeat_interleave construction, and invalid arguments are rejected before any
CUDA call."""
import ctypes
import os
import re

import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared, "no function found in include/kda.h"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"
    assert sorted(kda.EXPORTED) == declared


def test_only_abi_symbols_exported(lib):
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", kda.LIB_PATH], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm not available")
    ours = [ln.split()[-1] for ln in r.stdout.splitlines() if " T kda_" in ln]
    assert sorted(ours) == _declared_functions()


def test_chunk_size_and_last_error(lib):
    assert kda.chunk_size() in (32, 64, 128)
    assert isinstance(lib.kda_last_error(), bytes)


def _repeat_interleave_reference(cu, C):
    lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    nc = torch.tensor([(x + C - 1) // C for x in lens], dtype=torch.int64)
    seq = torch.repeat_interleave(torch.arange(len(lens)), nc)
    ins = torch.cat([torch.arange(int(n)) for n in nc] + [torch.zeros(0, dtype=torch.int64)])
    off = torch.zeros(len(lens) + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(nc, 0)
    return seq, ins, off


@pytest.mark.parametrize("cu", [
    [0, 37, 37, 96],              # empty sequence in the middle
    [0, 0, 0, 5, 5, 200],          # empty sequences first
    [0, 64, 128, 129],             # chunk-aligned and one-token tails
    [0],                           # no sequences
    [0, 0],                        # one empty sequence
])
@pytest.mark.parametrize("C", [16, 64])
def test_plan_chunks_matches_repeat_interleave(lib, cu, C):
    seq, ins, off = kda.plan_chunks(cu, C)
    rseq, rins, roff = _repeat_interleave_reference(cu, C)
    assert seq.tolist() == rseq.tolist()
    assert ins.tolist() == rins.tolist()
    assert off.tolist() == roff.tolist()


def test_plan_chunks_random(lib):
    g = torch.Generator().manual_seed(0)
    for _ in range(20):
        n = int(torch.randint(1, 40, (1,), generator=g))
        lens = torch.randint(0, 300, (n,), generator=g)
        lens[torch.rand(n, generator=g) < 0.3] = 0
        cu = [0] + torch.cumsum(lens, 0).tolist()
        seq, ins, off = kda.plan_chunks(cu, 64)
        rseq, rins, roff = _repeat_interleave_reference(cu, 64)
        assert seq.tolist() == rseq.tolist() and ins.tolist() == rins.tolist()
        assert off.tolist() == roff.tolist()


def test_plan_chunks_rejects_bad_bounds(lib):
    cu = torch.tensor([0, 5, 3], dtype=torch.int32)
    n = ctypes.c_int64(0)
    rc = lib.kda_plan_chunks(cu.data_ptr(), 2, 64, None, None, None, 0, ctypes.byref(n))
    assert rc == kda.KDA_ERR_INVALID_ARG
    assert b"decreases" in lib.kda_last_error()


def test_debug_wait_timeout_rejects_bad_arguments(lib):
    # checked before any CUDA call: a kind other than 0 or 1, a NULL workspace
    assert lib.kda_debug_wait_timeout(2, 4096, None) == kda.KDA_ERR_INVALID_ARG
    assert b"kind" in lib.kda_last_error()
    assert lib.kda_debug_wait_timeout(0, None, None) == kda.KDA_ERR_INVALID_ARG
    assert b"workspace" in lib.kda_last_error()


def test_workspace_size_is_an_upper_bound(lib):
    C = kda.chunk_size()
    assert kda.workspace_size(0, 0, 12) == 0
    assert kda.workspace_size(-1, 1, 12) == 0
    a = kda.workspace_size(16384, 1, 12)
    b = kda.workspace_size(16384, 4, 12)
    assert 0 < a < b
    # every split of T tokens into N sequences needs at most ceil(T/C) + N chunks
    g = torch.Generator().manual_seed(1)
    for _ in range(10):
        n = int(torch.randint(1, 30, (1,), generator=g))
        lens = torch.randint(0, 500, (n,), generator=g)
        cu = [0] + torch.cumsum(lens, 0).tolist()
        seq, _, _ = kda.plan_chunks(cu, C)
        assert seq.numel() <= (cu[-1] + C - 1) // C + n


# ---------------------------------------------------------------------------
# Argument rejection.  Fake (never dereferenced) device addresses: validation
# runs on the host before any CUDA call.
# ---------------------------------------------------------------------------

T, H, N = 100, 2, 2
ACT = T * H * 128 * 2
BASE = 1 << 40


def _args(**over):
    cu_host = (ctypes.c_int32 * 3)(0, 40, 100)
    a = dict(
        q=BASE, k=BASE + ACT, v=BASE + 2 * ACT, g=BASE + 3 * ACT, b=BASE + 5 * ACT,
        cu=BASE + 6 * ACT, cu_host=ctypes.addressof(cu_host), N=N, T=T, H=H,
        pool=BASE + 10 * ACT, stride0=H * 128 * 128, slots=4, idx=BASE + 7 * ACT,
        hs=BASE + 7 * ACT + 4096, out=BASE + 8 * ACT, lb=-5.0, dtype=0,
        ws=BASE + (1 << 36), wsb=1 << 34, stream=None,
    )
    a.update(over)
    a["_keep"] = cu_host
    return a


def _call(lib, a):
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"], a["cu_host"],
                             a["N"], a["T"], a["H"], a["pool"], a["stride0"], a["slots"],
                             a["idx"], a["hs"], a["out"], a["lb"], a["dtype"], a["ws"],
                             a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code,msg", [
    (dict(H=0), kda.KDA_ERR_INVALID_ARG, b"num_heads"),
    (dict(N=-1), kda.KDA_ERR_INVALID_ARG, b"num_seqs"),
    (dict(T=-5), kda.KDA_ERR_INVALID_ARG, b"total_tokens"),
    (dict(stride0=2 * 128 * 128 - 1), kda.KDA_ERR_INVALID_ARG, b"stride0"),
    (dict(out=BASE + 2 * ACT + 64), kda.KDA_ERR_INVALID_ARG, b"out overlaps v"),
    (dict(pool=BASE + 64), kda.KDA_ERR_INVALID_ARG, b"state_cache overlaps q"),
    (dict(dtype=3), kda.KDA_ERR_UNSUPPORTED, b"state_dtype"),
    (dict(lb=0.5), kda.KDA_ERR_UNSUPPORTED, b"lower_bound"),
    (dict(lb=float("nan")), kda.KDA_ERR_UNSUPPORTED, b"lower_bound"),
    (dict(q=BASE + 8), kda.KDA_ERR_UNSUPPORTED, b"aligned"),
    (dict(wsb=100), kda.KDA_ERR_WORKSPACE, b"workspace"),
    (dict(ws=None), kda.KDA_ERR_WORKSPACE, b"workspace"),
    (dict(pool=None), kda.KDA_ERR_INVALID_ARG, b"required"),
    (dict(idx=None), kda.KDA_ERR_INVALID_ARG, b"required"),
    (dict(slots=1), kda.KDA_ERR_INVALID_ARG, b"num_slots"),
    (dict(cu=None, cu_host=None), kda.KDA_ERR_INVALID_ARG, b"cu_seqlens"),
])
def test_rejects_invalid_arguments(lib, over, code, msg):
    a = _args(**over)
    assert _call(lib, a) == code
    assert msg in lib.kda_last_error(), lib.kda_last_error()


def _call_noalloc(lib, a):
    return lib.kda_chunk_fwd_noalloc(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"],
                                     a["cu_host"], a["N"], a["T"], a["H"], a["pool"],
                                     a["stride0"], a["slots"], a["idx"], a["hs"], a["out"],
                                     a["lb"], a["dtype"], a["stream"])


@pytest.mark.parametrize("over,code,msg", [
    (dict(H=0), kda.KDA_ERR_INVALID_ARG, b"num_heads"),
    (dict(T=-5), kda.KDA_ERR_INVALID_ARG, b"total_tokens"),
    (dict(stride0=2 * 128 * 128 - 1), kda.KDA_ERR_INVALID_ARG, b"stride0"),
    (dict(out=BASE + 2 * ACT + 64), kda.KDA_ERR_INVALID_ARG, b"out overlaps v"),
    (dict(pool=BASE + 64), kda.KDA_ERR_INVALID_ARG, b"state_cache overlaps q"),
    (dict(pool=BASE + 8 * ACT), kda.KDA_ERR_INVALID_ARG, b"state_cache overlaps out"),
    (dict(dtype=3), kda.KDA_ERR_UNSUPPORTED, b"state_dtype"),
    (dict(lb=0.5), kda.KDA_ERR_UNSUPPORTED, b"lower_bound"),
    (dict(q=BASE + 8), kda.KDA_ERR_UNSUPPORTED, b"aligned"),
    (dict(pool=None), kda.KDA_ERR_INVALID_ARG, b"required"),
    (dict(slots=1), kda.KDA_ERR_INVALID_ARG, b"num_slots"),
    (dict(cu_host=None), kda.KDA_ERR_INVALID_ARG, b"cu_seqlens_host"),
    (dict(cu=None), kda.KDA_ERR_INVALID_ARG, b"cu_seqlens"),
])
def test_noalloc_rejects_invalid_arguments(lib, over, code, msg):
    """The allocation-free entry point runs the paged entry point's host checks
    (pool overlaps included) before it touches CUDA."""
    a = _args(**over)
    assert _call_noalloc(lib, a) == code
    assert msg in lib.kda_last_error(), lib.kda_last_error()


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    T_big = 1 << 20  # 16 heads of a 1M-token prefill need far more than the scratch
    cu_host = (ctypes.c_int32 * 2)(0, T_big)
    act = T_big * 16 * 128 * 2
    a = _args(N=1, T=T_big, H=16, cu_host=ctypes.addressof(cu_host), q=BASE, k=BASE + act,
              v=BASE + 2 * act, g=BASE + 3 * act, b=BASE + 5 * act, out=BASE + 6 * act,
              pool=BASE + 8 * act, stride0=16 * 128 * 128)
    assert _call_noalloc(lib, a) == kda.KDA_ERR_WORKSPACE
    assert b"KDA_NOALLOC_SCRATCH_BYTES" in lib.kda_last_error()


@pytest.mark.parametrize("bounds,msg", [
    ((1, 40, 100), b"expected 0"),
    ((0, 50, 40), b"decreases"),
    ((0, 40, 99), b"total_tokens"),
])
def test_rejects_bad_host_bounds(lib, bounds, msg):
    cu_host = (ctypes.c_int32 * 3)(*bounds)
    a = _args(cu_host=ctypes.addressof(cu_host))
    assert _call(lib, a) == kda.KDA_ERR_INVALID_ARG
    assert msg in lib.kda_last_error()


def test_dense_rejects_overlapping_final_state(lib):
    a = _args()
    cu_host = (ctypes.c_int32 * 3)(0, 40, 100)
    rc = lib.kda_chunk_fwd_dense(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"],
                                 ctypes.addressof(cu_host), N, T, H, None, None,
                                 BASE + ACT, 0, a["out"], -5.0, a["ws"], a["wsb"], None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    assert b"final_state overlaps" in lib.kda_last_error()


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        kda.load_library(str(tmp_path / "missing.so"))


def test_status_and_switch_entry_points(lib):
    # kda_check_status rejects a missing output before touching CUDA
    rc = lib.kda_check_status(None, None, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    assert "status" in lib.kda_last_error().decode()
    # the fused-launch switch is host state only
    assert lib.kda_set_fused_launch(0) == kda.KDA_OK
    assert lib.kda_set_fused_launch(1) == kda.KDA_OK
    # four kernels in launch order, the fused launch between the scan and the
    # token-by-token kernel
    names = [lib.kda_kernel_name(i).decode() for i in range(4)]
    assert names == ["kda_intra", "kda_scan", "kda_fused", "kda_decode"]
    assert lib.kda_kernel_name(4) is None
