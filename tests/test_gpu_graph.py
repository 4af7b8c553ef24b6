"""CUDA graph capture of the forward (GPU).

After one call has cached the metadata of a set of bounds, a call with host
bounds makes no synchronising CUDA call and can be captured; replaying the graph
does what the call does.  A metadata miss, or device-only bounds, while the
stream captures is an error (KDA_ERR_CAPTURE_MISS) returned before anything is
enqueued.
"""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun


def _workspace(w):
    return torch.empty(kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads),
                       dtype=torch.uint8, device="cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("fused", [True, False])
def test_captured_call_replays_like_eager_calls(fused):
    """fused=False: the intra-chunk kernel, the scan and the token-by-token
    kernel as separate launches."""
    assert torch.cuda.is_available(), "GPU test"
    kda.set_fused_launch(fused)
    try:
        _captured_call_replays_like_eager_calls()
    finally:
        kda.set_fused_launch(True)


def _captured_call_replays_like_eager_calls():
    # long, short (token by token) and empty sequences in one batch
    w = wl.make_workload("graph", [300, 1, 130, 0, 5], 2, num_slots=8, seed=31,
                         has_initial_state=[1, 1, 0, 1, 0], stride_pad=64)
    eager, twin, warm = DevRun(w), DevRun(w), DevRun(w)
    ws_e, ws_t = _workspace(w), _workspace(w)
    eager.run(workspace=ws_e)
    eager.run(workspace=ws_e)
    warm.run(workspace=_workspace(w))  # caches the metadata of these bounds
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        twin.run(workspace=ws_t)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(twin.out, eager.out)
    assert torch.equal(twin.storage.view(torch.uint8), eager.storage.view(torch.uint8))


@pytest.mark.gpu
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_capture_without_cached_metadata_is_refused():
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("graph_miss", [77, 3, 191], 2, num_slots=4, seed=32)
    r = DevRun(w)
    ws = _workspace(w)
    kda.release_cache()
    s = torch.cuda.Stream()
    for host_bounds in (True, False):
        with pytest.raises(kda.KDAError) as e:
            with torch.cuda.graph(torch.cuda.CUDAGraph(), stream=s):
                r.run(host_bounds=host_bounds, workspace=ws)
        assert e.value.code == kda.KDA_ERR_CAPTURE_MISS
    torch.cuda.synchronize()
    # the same call outside capture still works afterwards
    r.run(workspace=ws)
    torch.cuda.synchronize()
