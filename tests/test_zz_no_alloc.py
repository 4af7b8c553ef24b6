"""GPU test of the allocation-free entry point, kda_chunk_fwd_noalloc.

That entry point serves callers that may not allocate device memory (for
example a serving runtime that owns all device memory in its own fixed arena,
or a plain-C caller with no device allocator).  It runs the same kernels as
kda_chunk_fwd with its scratch in a fixed array inside the library, so its
results must match kda_chunk_fwd's.  Two calls in a row are checked, which also
covers the array keeping the previous call's contents.

Kept in a file of its own, collected last, so that a run that stops at the
first failure has run every other test before this one.
"""

import numpy as np
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun, TOL, rel_l2

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, r: DevRun, cu_host):
    w = r.w
    rc = lib.kda_chunk_fwd_noalloc(
        r.q.data_ptr(), r.k.data_ptr(), r.v.data_ptr(), r.g.data_ptr(), r.b.data_ptr(),
        r.cu.data_ptr(), cu_host.data_ptr(), w.num_seqs, w.total_tokens, w.num_heads,
        r.pool.data_ptr(), r.pool.stride(0), r.pool.shape[0], r.idx.data_ptr(),
        r.hs.view(torch.uint8).data_ptr(), r.out.data_ptr(), float(w.lower_bound),
        kda.STATE_DTYPES[r.pool.dtype], torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.kda_last_error().decode()


@pytest.mark.parametrize("lengths,H,dt", [
    ([37, 0, 59], 2, torch.float32),
    ([300, 1, 0, 130], 3, torch.bfloat16),
])
def test_noalloc_matches_chunk_fwd_two_calls(lengths, H, dt):
    assert torch.cuda.is_available(), "GPU test"
    lib = kda.load_library()
    w = wl.make_workload("noalloc", lengths, H, num_slots=len(lengths) + 3, pool_dtype=dt,
                         stride_pad=128, seed=77 + H)
    ref = DevRun(w)
    new = DevRun(w)
    cu_host = w.cu_seqlens.clone()
    for call in range(2):  # the second call continues from the updated slots
        ref.run()
        _call_noalloc(lib, new, cu_host)
        torch.cuda.synchronize()
        eo = rel_l2(new.out.float().cpu().numpy(), ref.out.float().cpu().numpy())
        idx = w.state_indices.long().tolist()
        es = rel_l2(np.stack([new.pool[i].float().cpu().numpy() for i in idx]),
                    np.stack([ref.pool[i].float().cpu().numpy() for i in idx]))
        assert eo <= TOL[dt] and es <= TOL[dt], (call, eo, es)
        # unselected slots and the stride padding keep their bytes
        assert torch.equal(new.storage.cpu().view(torch.uint8), ref.storage.cpu().view(torch.uint8))

