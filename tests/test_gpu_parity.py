"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, on
small cases that span several chunks with ragged tails, on the named serving
workloads (sampled heads at full size), and on the edge cases of the method."""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun, TOL, compare, oracle_paged, unselected_untouched, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kda.load_library()


def test_tiny_varlen_workload():
    """3 sequences (37, 0, 59 tokens), H=2, fp32 pool; slot 2 (empty sequence,
    no initial state) is NaN-poisoned and must come back as zeros."""
    w = wl.tiny_varlen()
    wl.poison_unread_slots(w)
    r = DevRun(w)
    before = r.storage.cpu().clone()
    r.run()
    compare(r, tol=TOL[torch.float32])
    assert unselected_untouched(r, before)
    assert torch.equal(r.pool[2].cpu(), torch.zeros_like(r.pool[2].cpu()))


CASES = [
    # lengths, H, pool dtype, stride pad
    ([1, 63, 64, 65, 130, 0, 200], 3, torch.float32, 0),
    ([129, 1, 0, 0, 257], 2, torch.float32, 256),
    ([300, 5, 64], 2, torch.bfloat16, 64),
    ([77, 0, 191, 2], 2, torch.float16, 0),
    ([1] * 17 + [90], 2, torch.bfloat16, 0),
    # around the token-by-token / chunked split (at most 8 tokens: token by token)
    ([8, 9, 1, 0, 7, 2, 64, 3], 2, torch.float32, 32),
    ([3] * 5 + [1] * 5 + [8], 3, torch.float16, 0),
    # more than 2 * SMs / 8 (sequence, head) pairs on a 152-SM GPU: the scan's
    # large-batch form, each warp owning 16 value rows of the state (64 value rows
    # per CTA while those fit one wave, 128 beyond)
    ([70, 9, 128, 200, 65, 150, 33, 99, 64, 300] * 2, 2, torch.float32, 0),
    ([130, 65, 10, 257, 64] * 4, 2, torch.bfloat16, 64),
    ([70, 9, 128, 200, 65, 150, 33, 99, 64, 300] * 4, 2, torch.float32, 0),
    ([130, 65, 10, 257, 64] * 8, 2, torch.bfloat16, 64),
    # 64 value rows per CTA with a few token-by-token pairs beside the scan (fp16
    # pool, padded slot stride); 128 rows chosen because a wave of token-by-token
    # pairs runs beside a scan whose 64-row walks would fit one wave
    ([130, 65, 257] * 7 + [1] * 10, 2, torch.float16, 128),
    ([100] * 30 + [1] * 80, 2, torch.bfloat16, 0),
    # many short sequences: each persistent token-by-token CTA takes several items,
    # so its ring of state stages wraps around more than once
    ([1] * 300 + [2, 0, 5, 8] * 20, 2, torch.bfloat16, 0),
    ([1, 3, 0, 7] * 100 + [70], 2, torch.float32, 32),
]


@pytest.mark.parametrize("lengths,H,dt,pad", CASES)
def test_small_parity(lengths, H, dt, pad):
    w = wl.make_workload("small", lengths, H, num_slots=len(lengths) + 5, pool_dtype=dt,
                         stride_pad=pad, seed=sum(lengths) + H)
    wl.poison_unread_slots(w)
    r = DevRun(w)
    before = r.storage.cpu().clone()
    r.run()
    compare(r, tol=TOL[dt])
    assert unselected_untouched(r, before)


RAW_BF16_CASES = [
    # lengths, H, pool dtype, lower_bound
    ([1, 63, 64, 65, 130, 0, 200], 3, torch.float32, -5.0),
    ([300, 5, 64, 1, 1], 2, torch.bfloat16, -5.0),
    ([150, 2], 2, torch.float32, -40.0),  # the exact intra-chunk kernel
]


@pytest.mark.parametrize("lengths,H,dt,lb", RAW_BF16_CASES)
def test_raw_bf16_gate_and_beta(lengths, H, dt, lb):
    """Raw gate and beta in bf16 (kda_chunk_fwd_raw_bf16): parity with the
    oracle on the same bf16 values, through the chunked, the exact and the
    token-by-token kernels; unselected slots untouched."""
    w = wl.make_workload("raw16", lengths, H, num_slots=len(lengths) + 3, pool_dtype=dt,
                         lower_bound=lb, seed=40 + sum(lengths), raw_bf16=True)
    assert w.g_raw.dtype == torch.bfloat16 and w.beta_raw.dtype == torch.bfloat16
    wl.poison_unread_slots(w)
    r = DevRun(w)
    before = r.storage.cpu().clone()
    r.run()
    compare(r, tol=TOL[dt])
    assert unselected_untouched(r, before)


def test_saturated_gates_and_strong_bound():
    """Raw gate +8 everywhere (about 5 nats of decay per token and channel at
    lower_bound -5; 160+ nats per chunk) and, separately, lower_bound -40: no
    overflow, parity holds."""
    w = wl.make_workload("sat", [200, 70], 2, num_slots=4, seed=5)
    w.g_raw.fill_(8.0)
    compare(DevRun(w).run(), tol=TOL[torch.float32])
    w2 = wl.make_workload("strong", [150], 2, num_slots=2, lower_bound=-40.0, seed=6,
                          has_initial_state=[1])
    compare(DevRun(w2).run(), tol=TOL[torch.float32])


def test_no_decay():
    """lower_bound 0: no decay at all, the state only accumulates delta writes."""
    w = wl.make_workload("nodecay", [180, 33], 2, num_slots=3, lower_bound=0.0, seed=7)
    compare(DevRun(w).run(), tol=TOL[torch.float32])


def test_paged_equals_dense_bit_for_bit():
    """The paged call and the dense call give identical bytes for out and the
    selected states (same kernels, same schedule)."""
    w = wl.make_workload("pd", [100, 0, 65, 3], 2, num_slots=9, stride_pad=128, seed=8,
                         has_initial_state=[1, 0, 1, 0])
    r = DevRun(w).run()
    N, H = w.num_seqs, w.num_heads
    init = torch.zeros(N, H, 128, 128, dtype=w.state_pool.dtype)
    for n in range(N):
        if bool(w.has_initial_state[n]):
            init[n] = w.state_pool[int(w.state_indices[n])]
    init = init.cuda()
    fin = torch.empty_like(init)
    out = torch.empty_like(r.v)
    kda.chunk_fwd_dense(r.q, r.k, r.v, r.g, r.b, r.cu, initial_state=init,
                        has_initial_state=r.hs, final_state=fin, out=out,
                        lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(out, r.out)
    for n in range(N):
        assert torch.equal(fin[n], r.pool[int(w.state_indices[n])])
    # zero initial state via NULL equals has_initial_state = 0 everywhere
    fin0 = torch.empty_like(init)
    out0 = torch.empty_like(r.v)
    kda.chunk_fwd_dense(r.q, r.k, r.v, r.g, r.b, r.cu, final_state=fin0, out=out0,
                        lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    r0 = DevRun(w)
    r0.hs.zero_()
    r0.run()
    torch.cuda.synchronize()
    assert torch.equal(out0, r0.out)


def test_has_initial_state_false_never_reads_slot():
    """A NaN-filled slot whose flag is false gives the same bytes as a
    zero-filled one."""
    w = wl.make_workload("nan", [90, 40], 2, num_slots=4, seed=9, has_initial_state=[0, 1])
    a = DevRun(w)
    a.pool[int(w.state_indices[0])] = float("nan")
    a.run()
    b = DevRun(w)
    b.pool[int(w.state_indices[0])] = 0.0
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert torch.isfinite(a.out.float()).all()
    for i in w.state_indices.tolist():
        assert torch.equal(a.pool[i], b.pool[i])


def test_all_sequences_empty():
    """No tokens at all: flagged slots keep their value (bit-exact round trip
    through fp32), unflagged slots become zeros."""
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        w = wl.make_workload("empty", [0, 0, 0], 2, num_slots=5, pool_dtype=dt, seed=10,
                             has_initial_state=[1, 0, 1])
        r = DevRun(w)
        before = r.pool.clone()
        r.run()
        torch.cuda.synchronize()
        idx = w.state_indices.tolist()
        assert torch.equal(r.pool[idx[0]], before[idx[0]])
        assert torch.equal(r.pool[idx[2]], before[idx[2]])
        assert torch.equal(r.pool[idx[1]], torch.zeros_like(before[idx[1]]))


def test_deterministic():
    w = wl.make_workload("det", [333, 0, 17], 3, num_slots=6, seed=11)
    a = DevRun(w).run()
    b = DevRun(w).run()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out) and torch.equal(a.storage, b.storage)


def test_device_bounds_equal_host_bounds():
    """Without host bounds the call reads cu_seqlens back once; results are
    bit-identical to the call with host bounds."""
    w = wl.make_workload("dev", [70, 0, 130], 2, num_slots=4, seed=12)
    a = DevRun(w).run(host_bounds=True)
    b = DevRun(w).run(host_bounds=False)
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out) and torch.equal(a.storage, b.storage)


def test_split_call_matches_single_call():
    """A sequence run in two calls that hand the state over through its slot
    equals one call (within tolerance: chunk boundaries differ)."""
    w = wl.make_workload("split", [230], 2, num_slots=3, seed=13, has_initial_state=[1],
                         state_indices=[1])
    full = DevRun(w).run()
    s = 97
    first = wl.make_workload("a", [s], 2, num_slots=3, seed=13, has_initial_state=[1],
                             state_indices=[1])
    for name in ("q", "k", "v", "g_raw", "beta_raw"):
        getattr(first, name).copy_(getattr(w, name)[:, :s])
    first.pool_storage.copy_(w.pool_storage)
    a = DevRun(first).run()
    second = wl.make_workload("b", [230 - s], 2, num_slots=3, seed=13, has_initial_state=[1],
                              state_indices=[1])
    for name in ("q", "k", "v", "g_raw", "beta_raw"):
        getattr(second, name).copy_(getattr(w, name)[:, s:])
    b = DevRun(second)
    b.storage.copy_(a.storage)
    b.run()
    torch.cuda.synchronize()
    out2 = torch.cat([a.out, b.out], dim=1).float().cpu()
    assert rel_l2(out2.numpy(), full.out.float().cpu().numpy()) < 2e-3
    assert rel_l2(b.pool[1].cpu().numpy(), full.pool[1].cpu().numpy()) < 2e-3


# ---------------------------------------------------------------------------
# Named serving workloads at full size; the oracle checks sampled heads.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,heads", [
    ("prefill_4k", [0, 7]),
    ("prefill_16k", [3]),
    ("varlen_batch", [5]),
    ("mixed_bf16_pool", [0, 11]),
])
def test_serving_workload_sampled_heads(name, heads):
    w = wl.WORKLOADS[name]()
    r = DevRun(w)
    before = r.storage.cpu().clone()
    r.run()
    tol = TOL[w.state_pool.dtype]
    eo, es = compare(r, heads=heads, tol=tol)
    print(f"{name}: out rel-L2 {eo:.3e}, state rel-L2 {es:.3e}")
    assert unselected_untouched(r, before)
    assert torch.isfinite(r.out.float()).all()


@pytest.mark.gpu
@pytest.mark.parametrize("fused", [True, False])
def test_bad_state_index_is_skipped_and_reported(fused):
    """A slot outside [0, num_slots) is neither read nor written and shows in the
    status word; the other sequences are unaffected (the walks check the long
    sequences' slots, the token-by-token kernel the short one's)."""
    import copy
    lengths = [130, 70, 3, 90]
    w = wl.make_workload("bad_slot", lengths, 2, num_slots=6, state_indices=[1, 6, -3, 4],
                         has_initial_state=[1, 1, 1, 0], seed=51)
    # the oracle on the same inputs with harmless slots for the two bad sequences
    ref = copy.copy(w)
    ref.state_indices = torch.tensor([1, 2, 3, 4], dtype=torch.int32)
    ref.has_initial_state = torch.tensor([True, False, False, False])
    o_ref, f_ref = oracle_paged(ref)
    r = DevRun(w)
    before = r.storage.cpu().clone()
    ws = torch.empty(kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    kda.set_fused_launch(fused)
    try:
        r.run(workspace=ws)
        status = kda.check_status(ws)
    finally:
        kda.set_fused_launch(True)
    assert status == kda.STATUS_BAD_SLOT
    after = r.storage.cpu()
    for slot in (0, 2, 3, 5):  # no valid sequence writes them, the bad ones must not
        assert torch.equal(after[slot].view(torch.int32), before[slot].view(torch.int32))
    cu = w.cu_seqlens.tolist()
    for n, slot in ((0, 1), (3, 4)):
        o_gpu = r.out[0, cu[n]:cu[n + 1]].double().cpu().numpy()
        assert rel_l2(o_gpu, o_ref[cu[n]:cu[n + 1]]) <= TOL[torch.float32]
        f_gpu = r.pool[slot].double().cpu().numpy()
        assert rel_l2(f_gpu, f_ref[n]) <= TOL[torch.float32]


@pytest.mark.gpu
def test_status_is_clear_after_a_normal_call():
    w = wl.tiny_varlen()
    r = DevRun(w)
    ws = torch.empty(kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    r.run(workspace=ws)
    assert kda.check_status(ws) == 0


SEGMENTED_CASES = [
    # at most 4 (sequence, head) pairs with long sequences: the scan runs
    # segmented (pass A, combine, pass B)
    ([3000], 1, torch.float32, 0, [1]),                 # one pair, 10 segments of 5 chunks
    ([1000, 700, 5], 2, torch.float16, 32, [1, 0, 1]),  # 4 pairs, 3 and 2 segments, one short
]


@pytest.mark.gpu
@pytest.mark.parametrize("lengths,H,dt,pad,flags", SEGMENTED_CASES)
def test_segmented_scan(lengths, H, dt, pad, flags):
    w = wl.make_workload("segmented", lengths, H, num_slots=len(lengths) + 3, pool_dtype=dt,
                         stride_pad=pad, has_initial_state=flags, seed=sum(lengths) + H)
    wl.poison_unread_slots(w)
    r = DevRun(w)
    before = r.storage.cpu().clone()
    kda.set_kernel_timing(True)
    kda.kernel_times()
    try:
        r.run()
        torch.cuda.synchronize()
        times, _ = kda.kernel_times()
    finally:
        kda.set_kernel_timing(False)
    assert times["kda_fused"] == 0.0 and times["kda_scan"] > 0.0, times
    compare(r, tol=TOL[dt])
    assert unselected_untouched(r, before)
