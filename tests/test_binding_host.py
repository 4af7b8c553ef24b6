"""CPU tests of the Python binding's argument checks.  The checks run before the
binding touches CUDA, so CPU tensors that report themselves as CUDA tensors
reach them; every call here must stop at a ValueError or TypeError."""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl


class _AsCuda(torch.Tensor):
    """A CPU tensor that passes the binding's `is_cuda` test."""

    @property
    def is_cuda(self):
        return True


def _c(x):
    return x.as_subclass(_AsCuda)


@pytest.fixture(scope="module")
def args():
    w = wl.make_workload("binding_host", [37, 0, 59], 2, num_slots=5, seed=3)
    S, stride0 = w.pool_storage.shape
    pool = w.pool_storage.as_strided((S, 2, 128, 128), (stride0, 128 * 128, 128, 1))
    return w, dict(q=_c(w.q), k=_c(w.k), v=_c(w.v), g=_c(w.g_raw), b=_c(w.beta_raw),
                   cu=_c(w.cu_seqlens), pool=_c(pool), idx=_c(w.state_indices),
                   hs=_c(w.has_initial_state), out=_c(torch.empty_like(w.v)))


def _paged(w, a, **over):
    kw = dict(state_cache=a["pool"], state_indices=a["idx"], has_initial_state=a["hs"],
              out=a["out"], lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    kw.update(over)
    return kda.chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"], **kw)


@pytest.mark.parametrize("case,message", [
    ("indices_short", "state_indices must be a contiguous tensor of 3"),
    ("indices_strided", "state_indices must be a contiguous tensor of 3"),
    ("flags_short", "has_initial_state must be a contiguous tensor of 3"),
    ("host_bounds_short", "cu_seqlens_cpu has 3 bounds"),
    ("pool_plane", r"state_cache must be \[slots, H, 128, 128\]"),
    ("pool_padded_plane", "only stride\\(0\\) may pad"),
    ("out_shape", "out must have the shape of v"),
    ("q_dtype", "q must be torch.bfloat16"),
    ("raw_dtypes_differ", "g_raw and beta_raw must share a dtype"),
    ("pool_dtype", "state_cache dtype"),
    ("flags_dtype", "has_initial_state must be a bool/uint8"),
])
def test_paged_binding_rejects_before_cuda(args, case, message):
    w, a = args
    idx, hs, pool = a["idx"], a["hs"], a["pool"]
    over, call_args = {}, dict(a)
    if case == "indices_short":
        over["state_indices"] = idx[:2]
    elif case == "indices_strided":
        over["state_indices"] = _c(torch.stack([w.state_indices] * 2, 1)[:, 0])
    elif case == "flags_short":
        over["has_initial_state"] = hs[:2]
    elif case == "host_bounds_short":
        over["cu_seqlens_cpu"] = w.cu_seqlens[:3]
    elif case == "pool_plane":
        over["state_cache"] = _c(torch.zeros(5, 2, 128, 64))
    elif case == "pool_padded_plane":
        over["state_cache"] = _c(torch.zeros(5, 2, 128, 130)[..., :128])
    elif case == "out_shape":
        over["out"] = _c(torch.empty(1, 96, 2, 64, dtype=torch.bfloat16))
    elif case == "q_dtype":
        call_args["q"] = _c(w.q.float())
    elif case == "raw_dtypes_differ":
        call_args["b"] = _c(w.beta_raw.bfloat16())
    elif case == "pool_dtype":
        over["state_cache"] = _c(torch.zeros(5, 2, 128, 128, dtype=torch.float64))
    elif case == "flags_dtype":
        over["has_initial_state"] = _c(w.has_initial_state.int())
    with pytest.raises((ValueError, TypeError), match=message):
        _paged(w, call_args, **over)


def test_dense_binding_rejects_before_cuda(args):
    w, a = args
    fin = _c(torch.empty(3, 2, 128, 128))
    with pytest.raises(ValueError, match="has_initial_state"):
        kda.chunk_fwd_dense(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"],
                            initial_state=_c(torch.zeros(3, 2, 128, 128)),
                            has_initial_state=a["hs"][:1], final_state=fin, out=a["out"],
                            lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    with pytest.raises(ValueError, match="final_state"):
        kda.chunk_fwd_dense(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"],
                            final_state=_c(torch.empty(2, 2, 128, 128)), out=a["out"],
                            lower_bound=w.lower_bound, cu_seqlens_cpu=w.cu_seqlens)
    with pytest.raises(TypeError, match="initial_state"):
        kda.chunk_fwd_dense(a["q"], a["k"], a["v"], a["g"], a["b"], a["cu"],
                            initial_state=_c(torch.zeros(3, 2, 128, 128, dtype=torch.float16)),
                            final_state=fin, out=a["out"], lower_bound=w.lower_bound,
                            cu_seqlens_cpu=w.cu_seqlens)
