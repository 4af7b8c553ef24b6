"""Exact check of the 2-byte pool store.  Without initial states nothing the
kernels compute depends on the pool dtype: only the final store differs.  So on
the same inputs a bf16 or fp16 pool must receive exactly the round-to-nearest-even
cast of what an fp32 pool receives, and `out` must be bit-identical.  The batch
mixes long sequences (chunked kernels), short ones (token-by-token kernel) and an
empty one (its slot receives zeros)."""
import pytest
import torch

from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun

pytestmark = pytest.mark.gpu

LENGTHS = [300, 5, 0, 130, 1]


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_two_byte_pool_store_is_rne_of_the_fp32_state(dt):
    assert torch.cuda.is_available(), "GPU test"
    flags = [0] * len(LENGTHS)
    w32 = wl.make_workload("rne_f32", LENGTHS, 2, num_slots=8, pool_dtype=torch.float32,
                           has_initial_state=flags, seed=21)
    w16 = wl.make_workload("rne_16", LENGTHS, 2, num_slots=8, pool_dtype=dt,
                           has_initial_state=flags, seed=21)
    # same seed and draw order: the same inputs and slots, only the pool dtype differs
    assert torch.equal(w32.q, w16.q) and torch.equal(w32.state_indices, w16.state_indices)
    r32 = DevRun(w32).run()
    r16 = DevRun(w16).run()
    torch.cuda.synchronize()
    assert torch.equal(r32.out.view(torch.int16), r16.out.view(torch.int16))
    for s in w32.state_indices.tolist():
        want = r32.pool[s].cpu().to(dt)  # round to nearest even
        got = r16.pool[s].cpu()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), s
