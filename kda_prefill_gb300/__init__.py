"""Python binding of the GB300 chunkwise KDA forward library (``libkda.so``).

Argument marshalling only: every step of the forward runs in the CUDA kernels
behind the C ABI declared in ``include/kda.h``.  PyTorch provides device
memory and the current stream.  There is no fallback: if the library is
missing or was not built, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "chunk_fwd", "chunk_fwd_dense", "workspace_size", "chunk_size", "plan_chunks",
    "release_cache", "cache_entries", "load_library", "KDAError", "STATE_DTYPES",
    "set_kernel_timing", "kernel_times", "set_fused_launch", "check_status",
    "debug_wait_timeout", "STATUS_WAIT_TIMEOUT", "STATUS_SMEM_ALIGN", "STATUS_BAD_SLOT", "STATUS_BOUNDS_MISMATCH",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_CAPTURE_MISS = -3
KDA_ERR_CUDA = -4
KDA_ERR_WORKSPACE = -5

STATE_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}

# Every symbol include/kda.h declares (tests check the library exports them).
EXPORTED = (
    "kda_chunk_size", "kda_workspace_size", "kda_chunk_fwd", "kda_chunk_fwd_dense",
    "kda_plan_chunks", "kda_last_error", "kda_release_cache", "kda_cache_entries",
    "kda_set_kernel_timing", "kda_kernel_times", "kda_kernel_name", "kda_chunk_fwd_raw_bf16",
    "kda_chunk_fwd_noalloc", "kda_set_fused_launch", "kda_check_status",
    "kda_debug_wait_timeout",
)


class KDAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"KDA error {code}: {msg}")
        self.code = code


_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


def load_library(path: str = LIB_PATH):
    """Loads libkda.so (built by ``kda_prefill_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m kda_prefill_gb300.build` "
            "(or __graft_entry__.build()); there is no non-CUDA fallback")
    lib = ctypes.CDLL(path)
    lib.kda_chunk_size.restype = ctypes.c_int
    lib.kda_chunk_size.argtypes = []
    lib.kda_workspace_size.restype = ctypes.c_size_t
    lib.kda_workspace_size.argtypes = [_i64, _i32, _i32]
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_release_cache.restype = ctypes.c_int
    lib.kda_release_cache.argtypes = []
    lib.kda_cache_entries.restype = ctypes.c_int
    lib.kda_cache_entries.argtypes = []
    lib.kda_plan_chunks.restype = ctypes.c_int
    lib.kda_plan_chunks.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _i64, _vp]
    lib.kda_chunk_fwd.restype = ctypes.c_int
    lib.kda_chunk_fwd.argtypes = [
        _vp, _vp, _vp, _vp, _vp,        # q k v g_raw beta_raw
        _vp, _vp, _i32, _i64, _i32,     # cu_seqlens cu_seqlens_host N T H
        _vp, _i64, _i32, _vp, _vp,      # state_cache stride0 slots indices has_init
        _vp, ctypes.c_float, ctypes.c_int,  # out lower_bound state_dtype
        _vp, ctypes.c_size_t, _vp,      # workspace bytes stream
    ]
    lib.kda_chunk_fwd_raw_bf16.restype = ctypes.c_int
    lib.kda_chunk_fwd_raw_bf16.argtypes = list(lib.kda_chunk_fwd.argtypes)
    lib.kda_chunk_fwd_dense.restype = ctypes.c_int
    lib.kda_chunk_fwd_dense.argtypes = [
        _vp, _vp, _vp, _vp, _vp,
        _vp, _vp, _i32, _i64, _i32,
        _vp, _vp, _vp, ctypes.c_int,    # initial_state has_init final_state state_dtype
        _vp, ctypes.c_float,            # out lower_bound
        _vp, ctypes.c_size_t, _vp,
    ]
    lib.kda_set_kernel_timing.restype = ctypes.c_int
    lib.kda_set_kernel_timing.argtypes = [ctypes.c_int]
    lib.kda_set_fused_launch.restype = ctypes.c_int
    lib.kda_set_fused_launch.argtypes = [ctypes.c_int]
    lib.kda_check_status.restype = ctypes.c_int
    lib.kda_check_status.argtypes = [_vp, _vp, _vp]
    lib.kda_debug_wait_timeout.restype = ctypes.c_int
    lib.kda_debug_wait_timeout.argtypes = [ctypes.c_int, _vp, _vp]
    lib.kda_kernel_times.restype = ctypes.c_int
    lib.kda_kernel_times.argtypes = [_vp, ctypes.c_int, _vp, _vp]
    lib.kda_kernel_name.restype = ctypes.c_char_p
    lib.kda_kernel_name.argtypes = [ctypes.c_int]
    lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
    lib.kda_chunk_fwd_noalloc.argtypes = [
        _vp, _vp, _vp, _vp, _vp,        # q k v g_raw beta_raw
        _vp, _vp, _i32, _i64, _i32,     # cu_seqlens cu_seqlens_host N T H
        _vp, _i64, _i32, _vp, _vp,      # state_cache stride0 slots indices has_init
        _vp, ctypes.c_float, ctypes.c_int,  # out lower_bound state_dtype
        _vp,                            # stream
    ]
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(rc: int, lib) -> None:
    if rc != KDA_OK:
        raise KDAError(rc, lib.kda_last_error().decode(errors="replace"))


def chunk_size() -> int:
    return int(load_library().kda_chunk_size())


def workspace_size(total_tokens: int, num_seqs: int, num_heads: int) -> int:
    return int(load_library().kda_workspace_size(total_tokens, num_seqs, num_heads))


def release_cache() -> None:
    lib = load_library()
    _check(lib.kda_release_cache(), lib)


def cache_entries() -> int:
    return int(load_library().kda_cache_entries())


def set_kernel_timing(enable: bool) -> None:
    lib = load_library()
    _check(lib.kda_set_kernel_timing(1 if enable else 0), lib)


STATUS_WAIT_TIMEOUT = 1
STATUS_SMEM_ALIGN = 2
STATUS_BAD_SLOT = 4
STATUS_BOUNDS_MISMATCH = 8


def check_status(workspace: Optional[torch.Tensor] = None, stream=None) -> int:
    """Status word of the last call that used `workspace` (None: the scratch of
    the allocation-free entry point), after waiting for `stream` (default: the
    current stream).  0 when it completed normally, else STATUS_* bits."""
    lib = load_library()
    s = stream if stream is not None else torch.cuda.current_stream()
    v = ctypes.c_int(0)
    _check(lib.kda_check_status(_ptr(workspace), s.cuda_stream, ctypes.byref(v)), lib)
    return int(v.value)


def debug_wait_timeout(kind: int, workspace: torch.Tensor, stream=None) -> None:
    """Enqueues the failure-path diagnostic: a bounded wait on something that
    never happens (kind 0: an mbarrier, 1: a ready flag) gives up after about a
    second and sets STATUS_WAIT_TIMEOUT in `workspace`'s status word."""
    lib = load_library()
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.kda_debug_wait_timeout(int(kind), _ptr(workspace), s.cuda_stream), lib)


def set_fused_launch(enable: bool) -> None:
    """Enables (default) or disables the fused intra + scan launch."""
    lib = load_library()
    _check(lib.kda_set_fused_launch(1 if enable else 0), lib)


def kernel_times():
    """Per-kernel elapsed ms summed over the calls since the last read:
    ({name: ms}, calls)."""
    lib = load_library()
    ms = (ctypes.c_float * 16)()
    count = ctypes.c_int(0)
    calls = ctypes.c_int(0)
    _check(lib.kda_kernel_times(ctypes.addressof(ms), 16, ctypes.byref(count),
                                ctypes.byref(calls)), lib)
    names = [lib.kda_kernel_name(i).decode() for i in range(count.value)]
    return {n: float(ms[i]) for i, n in enumerate(names)}, calls.value


def plan_chunks(cu_seqlens_host, chunk: Optional[int] = None):
    """Host-only chunk numbering: (chunk_seq, chunk_in_seq, seq_chunk_offset)."""
    lib = load_library()
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    N = cu.numel() - 1
    c = chunk or chunk_size()
    n = ctypes.c_int64(0)
    rc = lib.kda_plan_chunks(cu.data_ptr(), N, c, None, None, None, 0, ctypes.byref(n))
    if rc not in (KDA_OK, KDA_ERR_WORKSPACE):
        _check(rc, lib)
    cap = n.value
    seq = torch.empty(cap, dtype=torch.int32)
    ins = torch.empty(cap, dtype=torch.int32)
    off = torch.empty(N + 1, dtype=torch.int32)
    _check(lib.kda_plan_chunks(cu.data_ptr(), N, c, seq.data_ptr(), ins.data_ptr(),
                               off.data_ptr(), cap, ctypes.byref(n)), lib)
    return seq, ins, off


def _flat(x: torch.Tensor, name: str, dtype, D: int = 128) -> torch.Tensor:
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x


def _ptr(x: Optional[torch.Tensor]):
    return None if x is None else x.data_ptr()


def _host_bounds(cu_seqlens_cpu, N: int):
    if cu_seqlens_cpu is None:
        return None
    h = torch.as_tensor(cu_seqlens_cpu)
    if h.device.type != "cpu":
        raise ValueError("cu_seqlens_cpu must be a CPU tensor")
    if h.numel() != N + 1:
        raise ValueError(f"cu_seqlens_cpu has {h.numel()} bounds, cu_seqlens {N + 1}")
    return h.to(torch.int32).contiguous()


def _workspace(workspace, T, N, H, device):
    need = workspace_size(T, N, H)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    if workspace.device != device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace too small: {need} bytes needed")
    return workspace


def _same_device(device, **tensors) -> None:
    """Every given tensor lives on `device` (the kernels read them all there)."""
    for name, x in tensors.items():
        if x is not None and x.device != device:
            raise ValueError(f"{name} is on {x.device}, q on {device}")


def _per_sequence(x: torch.Tensor, name: str, N: int) -> None:
    """One entry per sequence, contiguous (the kernels index it by sequence)."""
    if x.numel() != N or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of {N} entries, one per "
                         f"sequence; got shape {tuple(x.shape)}")


def _common(q, k, v, g_raw, beta_raw, cu_seqlens, raw_dtypes=(torch.float32,)):
    if q.dim() == 4:
        if q.shape[0] != 1:
            raise ValueError("packed varlen input must have batch dim 1")
    _flat(q, "q", torch.bfloat16)
    _flat(k, "k", torch.bfloat16)
    _flat(v, "v", torch.bfloat16)
    if g_raw.dtype not in raw_dtypes or beta_raw.dtype != g_raw.dtype:
        raise TypeError(f"g_raw and beta_raw must share a dtype among {raw_dtypes}")
    _flat(g_raw, "g_raw", g_raw.dtype)
    _flat(beta_raw, "beta_raw", beta_raw.dtype)
    T, H, D = q.shape[-3], q.shape[-2], q.shape[-1]
    if D != 128 or tuple(k.shape[-3:]) != (T, H, D) or tuple(v.shape[-3:]) != (T, H, D):
        raise ValueError("q, k, v must be [1, T, H, 128]")
    if tuple(g_raw.shape[-3:]) != (T, H, D) or tuple(beta_raw.shape[-2:]) != (T, H):
        raise ValueError("g_raw must be [1, T, H, 128] and beta_raw [1, T, H]")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise TypeError("cu_seqlens must be an int32 CUDA tensor")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous 1-D tensor of N + 1 bounds")
    _same_device(q.device, k=k, v=v, g_raw=g_raw, beta_raw=beta_raw, cu_seqlens=cu_seqlens)
    return T, H, cu_seqlens.numel() - 1


def chunk_fwd(q, k, v, g_raw, beta_raw, cu_seqlens, *, state_cache, state_indices,
              has_initial_state, out, lower_bound: float = -5.0, cu_seqlens_cpu=None,
              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged-pool forward (``kda_chunk_fwd``, or ``kda_chunk_fwd_raw_bf16`` when
    g_raw and beta_raw are bf16).  Writes ``out`` and the selected pool slots in
    place and returns ``out``."""
    lib = load_library()
    T, H, N = _common(q, k, v, g_raw, beta_raw, cu_seqlens,
                      raw_dtypes=(torch.float32, torch.bfloat16))
    _flat(out, "out", torch.bfloat16)
    if tuple(out.shape) != tuple(v.shape):
        raise ValueError("out must have the shape of v")
    if state_cache.dtype not in STATE_DTYPES:
        raise TypeError(f"state_cache dtype {state_cache.dtype} not supported")
    if state_cache.dim() != 4 or tuple(state_cache.shape[1:]) != (H, 128, 128):
        raise ValueError("state_cache must be [slots, H, 128, 128]")
    if tuple(state_cache.stride()[1:]) != (128 * 128, 128, 1):
        raise ValueError("each slot plane of state_cache must be dense (only stride(0) may pad)")
    if state_indices.dtype != torch.int32 or not state_indices.is_cuda:
        raise TypeError("state_indices must be an int32 CUDA tensor")
    hs = has_initial_state
    if hs.dtype == torch.bool:
        hs = hs.view(torch.uint8)
    if hs.dtype != torch.uint8 or not hs.is_cuda:
        raise TypeError("has_initial_state must be a bool/uint8 CUDA tensor")
    _per_sequence(state_indices, "state_indices", N)
    _per_sequence(hs, "has_initial_state", N)
    _same_device(q.device, out=out, state_cache=state_cache, state_indices=state_indices,
                 has_initial_state=hs)
    host = _host_bounds(cu_seqlens_cpu, N)
    ws = _workspace(workspace, T, N, H, q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    fn = lib.kda_chunk_fwd_raw_bf16 if g_raw.dtype == torch.bfloat16 else lib.kda_chunk_fwd
    rc = fn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
        _ptr(cu_seqlens), _ptr(host), N, T, H,
        _ptr(state_cache), state_cache.stride(0), state_cache.shape[0],
        _ptr(state_indices), _ptr(hs),
        _ptr(out), float(lower_bound), STATE_DTYPES[state_cache.dtype],
        _ptr(ws), ws.numel() * ws.element_size(), s.cuda_stream)
    _check(rc, lib)
    return out


def chunk_fwd_dense(q, k, v, g_raw, beta_raw, cu_seqlens, *, final_state, out,
                    initial_state: Optional[torch.Tensor] = None,
                    has_initial_state: Optional[torch.Tensor] = None,
                    lower_bound: float = -5.0, cu_seqlens_cpu=None,
                    workspace: Optional[torch.Tensor] = None, stream=None):
    """Dense-state forward (``kda_chunk_fwd_dense``): writes ``out`` and
    ``final_state`` [N, H, 128, 128]; returns (out, final_state)."""
    lib = load_library()
    T, H, N = _common(q, k, v, g_raw, beta_raw, cu_seqlens)
    _flat(out, "out", torch.bfloat16)
    if final_state.dtype not in STATE_DTYPES or not final_state.is_contiguous():
        raise TypeError("final_state must be a contiguous fp32/bf16/fp16 tensor")
    if tuple(final_state.shape) != (N, H, 128, 128):
        raise ValueError("final_state must be [N, H, 128, 128]")
    if initial_state is not None:
        if initial_state.dtype != final_state.dtype or not initial_state.is_contiguous():
            raise TypeError("initial_state must be contiguous with final_state's dtype")
        if tuple(initial_state.shape) != (N, H, 128, 128):
            raise ValueError("initial_state must be [N, H, 128, 128]")
    hs = has_initial_state
    if hs is not None:
        if hs.dtype == torch.bool:
            hs = hs.view(torch.uint8)
        if hs.dtype != torch.uint8 or not hs.is_cuda:
            raise TypeError("has_initial_state must be a bool/uint8 CUDA tensor")
        _per_sequence(hs, "has_initial_state", N)
    _same_device(q.device, out=out, final_state=final_state, initial_state=initial_state,
                 has_initial_state=hs)
    host = _host_bounds(cu_seqlens_cpu, N)
    ws = _workspace(workspace, T, N, H, q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    rc = lib.kda_chunk_fwd_dense(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
        _ptr(cu_seqlens), _ptr(host), N, T, H,
        _ptr(initial_state), _ptr(hs), _ptr(final_state), STATE_DTYPES[final_state.dtype],
        _ptr(out), float(lower_bound),
        _ptr(ws), ws.numel() * ws.element_size(), s.cuda_stream)
    _check(rc, lib)
    return out, final_state
