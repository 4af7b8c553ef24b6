"""Helpers shared by the GPU tests: move a workload to the device, run the
CUDA path through the binding, run the oracle on the same bytes (optionally on
a subset of heads), and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import kda_prefill_gb300 as kda
from kda_prefill_gb300.workloads import Workload

# Tolerances of the forward (rel-L2 against the fp64 oracle), by pool dtype.
TOL = {torch.float32: 5e-3, torch.bfloat16: 2e-2, torch.float16: 2e-2}


def rel_l2(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    d = np.linalg.norm(x - y)
    n = np.linalg.norm(y)
    return float(d / n) if n > 0 else float(d)


class DevRun:
    """Device copies of a workload plus the outputs of one call."""

    def __init__(self, w: Workload, device="cuda"):
        self.w = w
        self.q = w.q.to(device)
        self.k = w.k.to(device)
        self.v = w.v.to(device)
        self.g = w.g_raw.to(device)
        self.b = w.beta_raw.to(device)
        self.cu = w.cu_seqlens.to(device)
        self.storage = w.pool_storage.to(device)
        S, stride0 = w.pool_storage.shape
        H = w.num_heads
        self.pool = self.storage.as_strided((S, H, 128, 128), (stride0, 128 * 128, 128, 1))
        self.idx = w.state_indices.to(device)
        self.hs = w.has_initial_state.to(device)
        self.out = torch.empty_like(self.v)

    def run(self, host_bounds=True, workspace=None):
        kda.chunk_fwd(self.q, self.k, self.v, self.g, self.b, self.cu,
                      state_cache=self.pool, state_indices=self.idx,
                      has_initial_state=self.hs, out=self.out,
                      lower_bound=self.w.lower_bound,
                      cu_seqlens_cpu=self.w.cu_seqlens if host_bounds else None,
                      workspace=workspace)
        return self


def oracle_paged(w: Workload, heads=None):
    """fp64 oracle on the workload (restricted to `heads` if given).

    Returns (out [T, Hs, V], final [N, Hs, V, K]) for the selected heads."""
    hsel = list(range(w.num_heads)) if heads is None else list(heads)
    q = w.q[0][:, hsel].double().numpy()
    k = w.k[0][:, hsel].double().numpy()
    v = w.v[0][:, hsel].double().numpy()
    g = w.g_raw[0][:, hsel].double().numpy()
    b = w.beta_raw[0][:, hsel].double().numpy()
    idx = w.state_indices.long().numpy()
    flags = w.has_initial_state.numpy().astype(np.uint8)
    N = w.num_seqs
    init = np.zeros((N, len(hsel), 128, 128))
    for n in range(N):
        if flags[n]:
            init[n] = w.state_pool[idx[n]][hsel].double().numpy()
    out, fin = oracle.forward(q, k, v, g, b, w.cu_seqlens.numpy(), init, flags,
                              lower_bound=w.lower_bound)
    return out, fin


def per_sequence_rel_l2(o_gpu, o_ref, f_gpu, f_ref, cu):
    """Worst rel-L2 over the sequences of a packed batch: of each sequence's
    output rows (sequences with tokens) and of its final state.  A global rel-L2
    over a whole pack could hide a wrong result confined to a few short
    sequences; this cannot."""
    worst_o, worst_s = 0.0, 0.0
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            worst_o = max(worst_o, rel_l2(o_gpu[a:b], o_ref[a:b]))
        if f_ref.size:
            worst_s = max(worst_s, rel_l2(f_gpu[n], f_ref[n]))
    return worst_o, worst_s


def compare(run: DevRun, heads=None, tol=None):
    """Compares a finished GPU run with the oracle; returns (out_err, state_err),
    the rel-L2 over the whole batch.  With `tol`, it also asserts that the
    worst sequence of the batch (output rows and final state separately) is
    within the same tolerance; both figures are printed."""
    w = run.w
    hsel = list(range(w.num_heads)) if heads is None else list(heads)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle_paged(w, hsel)
    o_gpu = run.out[0][:, hsel].double().cpu().numpy()
    idx = w.state_indices.long().tolist()
    f_gpu = np.stack([run.pool[i][hsel].double().cpu().numpy() for i in idx]) if idx else \
        np.zeros((0, len(hsel), 128, 128))
    eo = rel_l2(o_gpu, o_ref) if o_ref.size else 0.0
    es = rel_l2(f_gpu, f_ref) if f_ref.size else 0.0
    wo, ws = per_sequence_rel_l2(o_gpu, o_ref, f_gpu, f_ref, w.cu_seqlens.numpy())
    print(f"{w.name}: out rel-L2 {eo:.3e} (worst sequence {wo:.3e}), "
          f"state rel-L2 {es:.3e} (worst sequence {ws:.3e})")
    if tol is not None:
        assert np.isfinite(o_gpu).all() and np.isfinite(f_gpu).all()
        assert eo <= tol, f"out rel-L2 {eo:.3e} > {tol}"
        assert es <= tol, f"state rel-L2 {es:.3e} > {tol}"
        assert wo <= tol, f"worst sequence's out rel-L2 {wo:.3e} > {tol}"
        assert ws <= tol, f"worst sequence's state rel-L2 {ws:.3e} > {tol}"
    return eo, es


def unselected_untouched(run: DevRun, before: torch.Tensor) -> bool:
    """True when every byte of the pool storage outside the selected slot
    planes (unselected slots and the stride padding) is unchanged."""
    after = run.storage.cpu()
    plane = run.w.num_heads * 128 * 128
    mask = torch.ones_like(after, dtype=torch.bool)
    for i in run.w.state_indices.tolist():
        mask[i, :plane] = False
    a = after.view(torch.uint8 if after.element_size() == 1 else
                   {4: torch.int32, 2: torch.int16}[after.element_size()])
    b = before.view(a.dtype)
    return bool(torch.equal(a[mask], b[mask]))
