"""GPU test of the allocation-free entry point, kda_chunk_fwd_noalloc.

That entry point serves callers that may not allocate device memory (for
example a serving runtime that owns all device memory in its own fixed arena,
or a plain-C caller with no device allocator).  It runs the same kernels as
kda_chunk_fwd with its scratch in a fixed array inside the library and its
chunk table built on the device, so its results must equal kda_chunk_fwd's
byte for byte.  Two calls in a row are checked, which also covers the array
keeping the previous call's contents.  The cases run the fused launch (small
ragged batch), the separate kernels with the token-by-token kernel (more than
1024 sequences, so the device table builder carries across its 1024-sequence
tiles), and the segmented scan (one long sequence, two heads).

Device bounds that disagree with the host bounds must not be trusted: the call
then computes nothing and reports the disagreement in the status word.

Kept in a file of its own, collected last, so that a run that stops at the
first failure has run every other test before this one.
"""

import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, r: DevRun, cu_host, cu_dev=None):
    w = r.w
    cu = r.cu if cu_dev is None else cu_dev
    rc = lib.kda_chunk_fwd_noalloc(
        r.q.data_ptr(), r.k.data_ptr(), r.v.data_ptr(), r.g.data_ptr(), r.b.data_ptr(),
        cu.data_ptr(), cu_host.data_ptr(), w.num_seqs, w.total_tokens, w.num_heads,
        r.pool.data_ptr(), r.pool.stride(0), r.pool.shape[0], r.idx.data_ptr(),
        r.hs.view(torch.uint8).data_ptr(), r.out.data_ptr(), float(w.lower_bound),
        kda.STATE_DTYPES[r.pool.dtype], torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.kda_last_error().decode()


def _many_sequences():
    """1200 sequences: one-token decode steps, empty ones, short ones up to the
    token-by-token limit and a few long ones, in a seeded order."""
    g = torch.Generator().manual_seed(5)
    lengths = []
    for i in range(1200):
        u = float(torch.rand(1, generator=g))
        if u < 0.05:
            lengths.append(0)
        elif u < 0.80:
            lengths.append(1)
        elif u < 0.99:
            lengths.append(int(torch.randint(2, 9, (1,), generator=g)))
        else:
            lengths.append(int(torch.randint(65, 200, (1,), generator=g)))
    return lengths


CASES = {
    "fused_small": ([37, 0, 59], 2, torch.float32),
    "ragged_bf16": ([300, 1, 0, 130], 3, torch.bfloat16),
    "segmented_1x1024_h2": ([1024], 2, torch.float32),
    "many_1200_seqs": (_many_sequences(), 2, torch.bfloat16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_equals_chunk_fwd_two_calls(case):
    assert torch.cuda.is_available(), "GPU test"
    lengths, H, dt = CASES[case]
    lib = kda.load_library()
    w = wl.make_workload("noalloc_" + case, lengths, H, num_slots=len(lengths) + 3,
                         pool_dtype=dt, stride_pad=128, seed=77 + H)
    ref = DevRun(w)
    new = DevRun(w)
    cu_host = w.cu_seqlens.clone()
    for call in range(2):  # the second call continues from the updated slots
        ref.run()
        _call_noalloc(lib, new, cu_host)
        torch.cuda.synchronize()
        assert kda.check_status(None) == 0
        assert torch.equal(new.out.view(torch.int16), ref.out.view(torch.int16)), (case, call)
        # every byte of the pool: the selected slots, the unselected ones and
        # the stride padding
        assert torch.equal(new.storage.view(torch.uint8), ref.storage.view(torch.uint8)), \
            (case, call)


@pytest.mark.parametrize("device_bounds", [
    [0, 37, 40, 96],    # same totals as the host bounds: only the checksum differs
    [0, 500, 20, 96],   # out of range and decreasing
    [0, 37, 37, 90],    # ends before total_tokens
    [5, 37, 37, 96],    # does not start at 0
])
def test_noalloc_refuses_device_bounds_that_disagree(device_bounds):
    assert torch.cuda.is_available(), "GPU test"
    lib = kda.load_library()
    w = wl.make_workload("noalloc_mismatch", [37, 0, 59], 2, num_slots=6, seed=91)
    r = DevRun(w)
    r.out.fill_(7.0)
    out_before = r.out.clone()
    pool_before = r.storage.clone()
    cu_dev = torch.tensor(device_bounds, dtype=torch.int32, device="cuda")
    _call_noalloc(lib, r, w.cu_seqlens.clone(), cu_dev)
    torch.cuda.synchronize()
    assert kda.check_status(None) & kda.STATUS_BOUNDS_MISMATCH
    assert torch.equal(r.out.view(torch.int16), out_before.view(torch.int16))
    assert torch.equal(r.storage.view(torch.uint8), pool_before.view(torch.uint8))
    # the next call with agreeing bounds runs normally and equals kda_chunk_fwd
    ref = DevRun(w)
    ref.run()
    _call_noalloc(lib, r, w.cu_seqlens.clone())
    torch.cuda.synchronize()
    assert kda.check_status(None) == 0
    assert torch.equal(r.out.view(torch.int16), ref.out.view(torch.int16))
