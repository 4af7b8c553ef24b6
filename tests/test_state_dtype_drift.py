"""Long-sequence numerics of the 2-byte state pools (GPU).

One sequence is served as a prefill call followed by one-token decode calls,
each call reading its initial state from the pool slot and writing the final
state back rounded to the pool's element type, as a serving loop does.  The
outputs of every call are compared with the fp64 oracle run over the whole
sequence in one pass (no rounding anywhere), window by window of decode steps,
and the final state likewise.  This is the study the state-dtype option of the
pages leaves to offline numerics (ROCm/aiter PR #5249, description: fp16 versus
bf16 storage of an fp32-accumulated state, and whether the error grows with
sequence length); here it also pins that the drift stays inside the forward's
tolerance for each pool type.
"""
import pytest
import torch

import kda_prefill_gb300 as kda
from kda_prefill_gb300 import workloads as wl
from tests.gpu_helpers import TOL, oracle_paged, rel_l2

PREFILL, DECODE, WINDOW, H = 1024, 512, 128, 2


def _serve(w, dt):
    """Prefill then one-token calls; returns (out [T, H, V] fp64, final state [H, V, K])."""
    dev = "cuda"
    T = w.total_tokens
    q, k, v = w.q[0].to(dev), w.k[0].to(dev), w.v[0].to(dev)
    g, b = w.g_raw[0].to(dev), w.beta_raw[0].to(dev)
    pool = torch.zeros((1, H, 128, 128), dtype=dt, device=dev)
    idx = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((1, T, H, 128), dtype=torch.bfloat16, device=dev)
    bounds = [(0, PREFILL)] + [(PREFILL + s, PREFILL + s + 1) for s in range(DECODE)]
    for c, (t0, t1) in enumerate(bounds):
        n = t1 - t0
        cu_h = torch.tensor([0, n], dtype=torch.int32)
        hs = torch.tensor([0 if c == 0 else 1], dtype=torch.uint8, device=dev)
        o = torch.empty((1, n, H, 128), dtype=torch.bfloat16, device=dev)
        kda.chunk_fwd(q[None, t0:t1].contiguous(), k[None, t0:t1].contiguous(),
                      v[None, t0:t1].contiguous(), g[None, t0:t1].contiguous(),
                      b[None, t0:t1].contiguous(), cu_h.to(dev), state_cache=pool,
                      state_indices=idx, has_initial_state=hs, out=o,
                      lower_bound=w.lower_bound, cu_seqlens_cpu=cu_h)
        out[:, t0:t1] = o
    torch.cuda.synchronize()
    return out[0].double().cpu().numpy(), pool[0].double().cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_state_dtype_drift_over_decode_steps(dt):
    assert torch.cuda.is_available(), "GPU test"
    w = wl.make_workload("drift", [PREFILL + DECODE], H, num_slots=1, seed=21,
                         has_initial_state=[0])
    ref_out, ref_fin = oracle_paged(w)
    got_out, got_fin = _serve(w, dt)
    errs = [rel_l2(got_out[PREFILL + s:PREFILL + s + WINDOW], ref_out[PREFILL + s:PREFILL + s + WINDOW])
            for s in range(0, DECODE, WINDOW)]
    e_pre = rel_l2(got_out[:PREFILL], ref_out[:PREFILL])
    e_fin = rel_l2(got_fin, ref_fin[0])
    name = str(dt).replace("torch.", "")
    print(f"\n{name} pool: prefill out {e_pre:.3e}; decode windows of {WINDOW} steps "
          + " ".join(f"{e:.3e}" for e in errs) + f"; final state {e_fin:.3e}")
    tol = TOL[dt]
    assert e_pre <= tol and e_fin <= tol and max(errs) <= tol, (e_pre, errs, e_fin)
