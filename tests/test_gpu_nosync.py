"""Streams: with host bounds a call makes no synchronising CUDA call; without
them it reads the bounds back once, which waits for the stream (ROCm/aiter PR
#6912, "Changes": one pinned non-blocking upload of the chunk metadata on a
cache miss, no blocking copy).  A bounded spin kernel queued ahead of the call
shows which: a host-bounds call returns while the stream is still busy (on a
metadata-cache hit and on a miss, including misses that fill the pinned
staging memory while every earlier upload is still queued behind the spin),
the device-bounds call only after the spin has ended."""
import time

import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 400_000_000  # ~0.2 s at 2 GHz


def _call(r: DevRun, cu_host, cu_dev):
    """The workload's call with other bounds (same tensors)."""
    kda.chunk_fwd(r.q, r.k, r.v, r.g, r.b, cu_dev, state_cache=r.pool,
                  state_indices=r.idx, has_initial_state=r.hs, out=r.out,
                  lower_bound=r.w.lower_bound, cu_seqlens_cpu=cu_host)


def test_host_bounds_call_does_not_wait_for_the_gpu():
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("nosync", [300, 5, 0, 70], 2, num_slots=6, seed=31)
    r = DevRun(w)
    r.run()  # the metadata for these bounds is cached from here on
    r.run(host_bounds=False)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    torch.cuda._sleep(SPIN_CYCLES)
    t0 = time.perf_counter()
    r.run(host_bounds=True)
    t_host = time.perf_counter() - t0
    still_busy = not stream.query()
    torch.cuda.synchronize()

    torch.cuda._sleep(SPIN_CYCLES)
    t0 = time.perf_counter()
    r.run(host_bounds=False)
    t_dev = time.perf_counter() - t0
    torch.cuda.synchronize()

    assert still_busy, "the stream finished before the host-bounds call returned"
    assert t_host < 0.05, t_host
    assert t_dev > 0.1 and t_dev > 4 * t_host, (t_dev, t_host)


def test_metadata_miss_does_not_wait_for_the_gpu():
    """Bounds never seen before: the chunk table is built on the host and
    uploaded behind the busy stream without waiting for it."""
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("nosync_miss", [300, 5, 0, 70], 2, num_slots=6, seed=32)
    r = DevRun(w)
    r.run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # a permutation of the lengths: the same tokens, bounds new to the cache
    new_bounds = torch.tensor([0, 70, 70, 75, 375], dtype=torch.int32)
    new_dev = new_bounds.to("cuda")  # copied before the spin, not behind it
    torch.cuda.synchronize()
    entries = kda.cache_entries()
    torch.cuda._sleep(SPIN_CYCLES)
    t0 = time.perf_counter()
    _call(r, new_bounds, new_dev)
    t_miss = time.perf_counter() - t0
    still_busy = not stream.query()
    torch.cuda.synchronize()
    assert kda.cache_entries() == entries + 1, "the call was not a cache miss"
    assert still_busy, "the stream finished before the call returned"
    assert t_miss < 0.01, t_miss  # < 5 % of the ~0.2 s spin


def test_metadata_misses_never_wait_when_the_staging_fills():
    """Twenty misses with ~0.5 MB of chunk metadata each (30,000 decode
    sequences) behind one busy stream: their uploads all wait for the spin, so
    the first pinned staging block (8 MB) fills and the next miss needs more.
    Every call must still return without waiting for the GPU."""
    assert torch.cuda.is_available(), "GPU test"
    dev = torch.device("cuda")
    N, H = 30000, 1
    gen = torch.Generator(device="cpu").manual_seed(7)
    q = torch.randn(1, N, H, 128, generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn(1, N, H, 128, generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn(1, N, H, 128, generator=gen).to(torch.bfloat16).to(dev)
    g = torch.randn(1, N, H, 128, generator=gen).to(dev)
    b = torch.randn(1, N, H, generator=gen).to(dev)
    pool = torch.zeros(N, H, 128, 128, dtype=torch.bfloat16, device=dev)
    idx = torch.arange(N, dtype=torch.int32, device=dev)
    hs = torch.zeros(N, dtype=torch.uint8, device=dev)
    out = torch.empty_like(v)

    def bounds(i):
        # one-token sequences, except sequence i empty and i + 1 with two tokens
        lens = torch.ones(N, dtype=torch.int64)
        lens[i], lens[i + 1] = 0, 2
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
        return cu

    sets = [bounds(i) for i in range(21)]
    devs = [c.to(dev) for c in sets]

    def call(j):
        kda.chunk_fwd(q, k, v, g, b, devs[j], state_cache=pool, state_indices=idx,
                      has_initial_state=hs, out=out, lower_bound=-5.0,
                      cu_seqlens_cpu=sets[j])

    call(0)  # library, first staging block and metadata pool set up
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    torch.cuda._sleep(2 * SPIN_CYCLES)
    times = []
    for j in range(1, 21):
        t0 = time.perf_counter()
        call(j)
        times.append(time.perf_counter() - t0)
    still_busy = not stream.query()
    torch.cuda.synchronize()
    assert still_busy, "the stream finished before the last call returned"
    assert max(times) < 0.02, times  # < 5 % of the ~0.4 s spin, every call
