"""The fused intra-chunk + scan launch against the two kernels in sequence (GPU).

Both schedules run the same arithmetic, so outputs and pool must agree byte for
byte; a hand-off race between the intra-chunk items and the scan walks (a walk
reading a block before it is written) would show as a difference.  The fused
schedule runs several times per case.
"""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun


def _small():
    return wl.make_workload("fused_small", [300, 1, 130, 0, 5, 77], 2, num_slots=10,
                            pool_dtype=torch.float16, seed=41, stride_pad=64)


# case: (workload, fused runs compared with the separate kernels)
CASES = {"prefill_16k": (wl.prefill_16k, 3), "prefill_4k": (wl.prefill_4k, 10),
         "small": (_small, 10)}


def _run(w, fused):
    kda.set_fused_launch(fused)
    kda.set_kernel_timing(True)
    kda.kernel_times()
    try:
        r = DevRun(w)
        ws = torch.empty(kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads),
                         dtype=torch.uint8, device="cuda")
        r.run(workspace=ws)
        torch.cuda.synchronize()
        times, _ = kda.kernel_times()
    finally:
        kda.set_kernel_timing(False)
        kda.set_fused_launch(True)
    return r.out.view(torch.int16).cpu(), r.storage.view(torch.uint8).cpu(), times


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_fused_equals_separate(name):
    assert torch.cuda.is_available(), "GPU test"
    make, runs = CASES[name]
    w = make()
    out_s, pool_s, t_s = _run(w, False)
    assert t_s["kda_fused"] == 0.0 and t_s["kda_scan"] > 0.0
    for _ in range(runs):
        out_f, pool_f, t_f = _run(w, True)
        assert t_f["kda_fused"] > 0.0 and t_f["kda_scan"] == 0.0, t_f
        assert torch.equal(out_f, out_s)
        assert torch.equal(pool_f, pool_s)
