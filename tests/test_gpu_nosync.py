"""Streams: with host bounds a call makes no synchronising CUDA call; without
them it reads the bounds back once, which waits for the stream (ROCm/aiter PR
#6912, "Changes").  A bounded spin kernel (about 0.2 s) queued ahead of the call
shows which: the host-bounds call returns while the stream is still busy, the
device-bounds call only after the spin has ended."""
import time

import pytest
import torch

from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun

pytestmark = pytest.mark.gpu

SPIN_CYCLES = 400_000_000  # ~0.2 s at 2 GHz


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
