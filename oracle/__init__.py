"""Plain CPU oracle for the KDA forward — test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library and its
Python binding) never does, and the two share no code.

The arithmetic lives in ``kda_oracle.c`` (fp64, token by token).  This module
compiles it with gcc, loads it with ctypes and adds the paged-pool semantics
around it:

* ``state_indices[n]`` names the pool slot of sequence ``n``; the slot is read
  only when ``has_initial_state[n]`` is set (ROCm/aiter PR #5754, "Technical
  Details": a false flag starts from zero and does not read a dirty slot);
* the final state of every sequence, empty ones included, is written back to the
  same slot (same section: the last segment writes the final state to the same
  row); slots that no sequence selects are returned unchanged.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# eps inside the square root of the L2 norm (the pages do not state it; 1e-6 is
# the plainest reading, and it only matters for all-zero rows).
L2_EPS = 1e-6


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library; returns its path."""
    cmd = [
        "gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c11",
        "-shared", "-fPIC", *extra_flags, src, "-o", out, "-lm",
    ]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _needs_build() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    return os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib):
    f = lib.kda_oracle_forward
    f.restype = ctypes.c_int
    f.argtypes = [
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int32, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_double, ctypes.c_double,
        ctypes.c_void_p, ctypes.c_void_p,
    ]
    lib.kda_oracle_num_threads.restype = ctypes.c_int
    lib.kda_oracle_num_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def num_threads() -> int:
    return int(load().kda_oracle_num_threads())


def _f64(x) -> np.ndarray:
    try:
        import torch  # noqa: F401  (only to accept CPU tensors)
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(q, k, v, g_raw, beta_raw, cu_seqlens, initial_state=None,
            has_initial_state=None, lower_bound: float = -5.0,
            eps: float = L2_EPS, lib=None):
    """Dense-state oracle.

    q, k, g_raw: [T, H, K] (a leading batch dim of 1 is accepted);
    v: [T, H, V]; beta_raw: [T, H]; cu_seqlens: [N+1];
    initial_state: [N, H, V, K] or None; has_initial_state: [N] or None
    (None means "set" when an initial state is given, "clear" otherwise).

    Returns (out [T, H, V], final_state [N, H, V, K]) as fp64 numpy arrays.
    """
    lib = lib or load()
    q, k, v, g_raw, beta_raw = (_f64(t) for t in (q, k, v, g_raw, beta_raw))
    if q.ndim == 4:
        q, k, v, g_raw = q[0], k[0], v[0], g_raw[0]
    if beta_raw.ndim == 3:
        beta_raw = beta_raw[0]
    q, k, v, g_raw, beta_raw = (np.ascontiguousarray(t) for t in (q, k, v, g_raw, beta_raw))
    T, H, K = q.shape
    V = v.shape[2]
    assert k.shape == (T, H, K) and g_raw.shape == (T, H, K)
    assert v.shape == (T, H, V) and beta_raw.shape == (T, H)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
        dtype=np.int64))
    N = cu.shape[0] - 1
    if has_initial_state is None:
        flags = np.full(N, 1 if initial_state is not None else 0, dtype=np.uint8)
    else:
        hs = has_initial_state
        hs = hs.cpu().numpy() if hasattr(hs, "cpu") else hs
        flags = np.ascontiguousarray(np.asarray(hs).astype(np.uint8))
    init = None if initial_state is None else _f64(initial_state)
    if init is not None:
        assert init.shape == (N, H, V, K)
    out = np.empty((T, H, V), dtype=np.float64)
    fin = np.empty((N, H, V, K), dtype=np.float64)
    rc = lib.kda_oracle_forward(
        T, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
        N, _ptr(cu), _ptr(init), _ptr(flags), float(lower_bound), float(eps),
        _ptr(out), _ptr(fin))
    if rc != 0:
        raise ValueError(f"kda_oracle_forward rejected its arguments (rc={rc})")
    return out, fin


def forward_paged(q, k, v, g_raw, beta_raw, cu_seqlens, state_pool,
                  state_indices, has_initial_state, lower_bound: float = -5.0,
                  eps: float = L2_EPS, lib=None):
    """Paged-pool oracle.

    state_pool: [slots, H, V, K] (any float dtype; read exactly as fp64);
    state_indices: [N] distinct slots; has_initial_state: [N].

    Returns (out [T, H, V] fp64, new_pool [slots, H, V, K] fp64) where
    new_pool equals the input pool except on the selected slots, which hold the
    unrounded final states.
    """
    pool = _f64(state_pool)
    idx = np.asarray(state_indices.cpu().numpy() if hasattr(state_indices, "cpu")
                     else state_indices, dtype=np.int64)
    hs = has_initial_state
    hs = np.asarray(hs.cpu().numpy() if hasattr(hs, "cpu") else hs).astype(bool)
    assert len(np.unique(idx)) == len(idx), "state_indices must be distinct"
    N = idx.shape[0]
    init = np.zeros((N,) + pool.shape[1:], dtype=np.float64)
    for n in range(N):
        if hs[n]:
            init[n] = pool[idx[n]]
    out, fin = forward(q, k, v, g_raw, beta_raw, cu_seqlens, init, hs,
                       lower_bound, eps, lib)
    new_pool = pool.copy()
    for n in range(N):
        new_pool[idx[n]] = fin[n]
    return out, new_pool
