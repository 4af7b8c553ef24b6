"""The kernels' failure path on the GPU, without a fault (GPU).

Every wait in the kernels (mbarrier phases, the fused launch's ready flags) is
bounded: after about a second it gives up, the kernel sets the status word and
leaves.  `kda_debug_wait_timeout` runs that same bounded wait on something that
never happens (an mbarrier nothing arrives on, a flag nothing sets); the test
checks that it gives up in bounded time, that the status word says so, and that
the context stays usable: a normal call right after it matches the oracle and
clears the status.
"""
import time

import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun, TOL, compare


@pytest.mark.gpu
@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "ready_flag"])
def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable(kind):
    assert torch.cuda.is_available(), "GPU test"
    w = wl.tiny_varlen()
    ws = torch.zeros(kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kda.debug_wait_timeout(kind, ws)
    status = kda.check_status(ws)  # waits for the stream
    elapsed = time.perf_counter() - t0
    print(f"kind {kind}: gave up after {elapsed:.3f} s, status {status}")
    assert status == kda.STATUS_WAIT_TIMEOUT
    # the wait's limit is one second of GPU time; allow launch and host slack
    assert 0.5 <= elapsed <= 30.0, elapsed

    r = DevRun(w)
    r.run(workspace=ws)
    compare(r, tol=TOL[torch.float32])
    assert kda.check_status(ws) == 0

