"""GPU tests of the Python binding's argument checks: tensors whose sizes or
layout disagree with the batch are rejected in Python, before the C ABI is
called, instead of reaching the kernels as out-of-range reads."""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import DevRun

pytestmark = pytest.mark.gpu


def _paged(r: DevRun, **over):
    a = dict(state_cache=r.pool, state_indices=r.idx, has_initial_state=r.hs, out=r.out,
             lower_bound=r.w.lower_bound, cu_seqlens_cpu=r.w.cu_seqlens)
    a.update(over)
    return kda.chunk_fwd(r.q, r.k, r.v, r.g, r.b, r.cu, **a)


def test_paged_binding_rejects_inconsistent_arguments():
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("binding", [37, 0, 59], 2, num_slots=5, seed=3)
    r = DevRun(w)
    _paged(r)  # the consistent call goes through
    torch.cuda.synchronize()
    need = kda.workspace_size(w.total_tokens, w.num_seqs, w.num_heads)
    cases = [
        (dict(state_indices=r.idx[:2]), "state_indices"),
        (dict(state_indices=torch.stack([r.idx, r.idx], 1)[:, 0]), "state_indices"),
        (dict(has_initial_state=r.hs[:2]), "has_initial_state"),
        (dict(cu_seqlens_cpu=w.cu_seqlens[:3]), "cu_seqlens_cpu"),
        (dict(workspace=torch.empty(need, dtype=torch.uint8)), "workspace"),
        (dict(workspace=torch.empty(2 * need, dtype=torch.uint8, device="cuda")[::2]),
         "workspace"),
    ]
    for over, name in cases:
        with pytest.raises(ValueError, match=name):
            _paged(r, **over)


def test_dense_binding_rejects_inconsistent_flags():
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("binding_dense", [37, 0, 59], 2, num_slots=5, seed=4)
    r = DevRun(w)
    N, H = w.num_seqs, w.num_heads
    init = torch.zeros(N, H, 128, 128, device="cuda")
    fin = torch.empty_like(init)
    out = torch.empty_like(r.v)
    with pytest.raises(ValueError, match="has_initial_state"):
        kda.chunk_fwd_dense(r.q, r.k, r.v, r.g, r.b, r.cu, initial_state=init,
                            has_initial_state=r.hs[:1], final_state=fin, out=out,
                            lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    kda.chunk_fwd_dense(r.q, r.k, r.v, r.g, r.b, r.cu, initial_state=init,
                        has_initial_state=r.hs, final_state=fin, out=out,
                        lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
