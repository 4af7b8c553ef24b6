"""Seeded synthetic inputs for the KDA forward.

This module draws random numbers and lays them out; it contains none of the
method's arithmetic, so that the oracle and the CUDA path can both take their
inputs from it without sharing any computation.

Every tensor is drawn on the CPU from one ``torch.Generator`` in a fixed order:
sequence lengths (when drawn), q, k, v, raw gate, raw beta, state pool, state
indices, has-initial-state flags.  q, k and v are drawn in fp32 and rounded to
bf16 (round to nearest even), so the oracle and the GPU see the same bytes.

The named workloads follow the serving shapes of the KDA prefill pages
(ROCm/aiter PR #5754, "Serving-shaped A/B" and "Test Result": K3 H=12, D=128,
lower_bound = -5, varlen cu_seqlens, fp32 V-first pool; PR #5249 for the 2-byte
pool).  The pages measure on serving traffic only; these synthetic draws stand
in for it.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

D = 128  # head dimension K = V of the serving shapes

# Canary written into the padding of a pool whose slot stride is padded, and
# into slots the call must not touch.  A quiet-NaN bit pattern for fp32 pools.
CANARY_F32_BITS = 0x7FC0DEAD
CANARY_16_BITS = 0x7E5A


@dataclass
class Workload:
    name: str
    q: torch.Tensor            # [1, T, H, K] bf16
    k: torch.Tensor            # [1, T, H, K] bf16
    v: torch.Tensor            # [1, T, H, V] bf16
    g_raw: torch.Tensor        # [1, T, H, K] fp32 raw gate
    beta_raw: torch.Tensor     # [1, T, H]    fp32 raw beta
    cu_seqlens: torch.Tensor   # [N+1] int32
    state_pool: torch.Tensor   # [slots, H, V, K] view, stride(0) may be padded
    pool_storage: torch.Tensor # [slots, stride0] backing storage of the pool
    state_indices: torch.Tensor      # [N] int32
    has_initial_state: torch.Tensor  # [N] bool
    lower_bound: float = -5.0
    meta: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def lengths(self) -> list:
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _canary(dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.float32:
        return torch.tensor([CANARY_F32_BITS], dtype=torch.int32).view(torch.float32)
    if dtype in (torch.bfloat16, torch.float16):
        return torch.tensor([CANARY_16_BITS], dtype=torch.int16).view(dtype)
    raise ValueError(dtype)


def make_workload(name: str, lengths: Sequence[int], num_heads: int, *,
                  num_slots: int, pool_dtype=torch.float32, stride_pad: int = 0,
                  pool_std: float = 0.1, state_indices: Optional[Sequence[int]] = None,
                  has_initial_state: Optional[Sequence[int]] = None,
                  init_prob: float = 0.5, lower_bound: float = -5.0, seed: int = 0,
                  draw_lengths=None, gate_scale: float = 1.0, raw_bf16: bool = False) -> Workload:
    """Draws one workload.

    ``lengths`` fixes the sequence lengths unless ``draw_lengths`` is given, in
    which case it is called with the generator first (so the lengths are part
    of the seeded stream).  ``state_indices`` defaults to a random choice of
    distinct slots, ``has_initial_state`` to Bernoulli(``init_prob``).
    ``raw_bf16`` rounds the raw gate and beta to bf16 (RNE) after drawing them,
    so both paths read the same values.
    """
    g = torch.Generator().manual_seed(seed)
    if draw_lengths is not None:
        lengths = draw_lengths(g)
    lengths = [int(x) for x in lengths]
    N = len(lengths)
    H = num_heads
    T = sum(lengths)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)

    q = _bf16(torch.randn(1, T, H, D, generator=g))
    k = _bf16(torch.randn(1, T, H, D, generator=g))
    v = _bf16(torch.randn(1, T, H, D, generator=g))
    g_raw = torch.randn(1, T, H, D, generator=g) * gate_scale
    beta_raw = torch.randn(1, T, H, generator=g)
    if raw_bf16:
        g_raw, beta_raw = g_raw.to(torch.bfloat16), beta_raw.to(torch.bfloat16)

    plane = H * D * D
    stride0 = plane + stride_pad
    storage = torch.empty(num_slots, stride0, dtype=pool_dtype)
    storage[:, :] = _canary(pool_dtype)
    live = (torch.randn(num_slots, plane, generator=g) * pool_std).to(pool_dtype)
    storage[:, :plane] = live
    pool = storage.as_strided((num_slots, H, D, D), (stride0, D * D, D, 1))

    if state_indices is None:
        idx = torch.randperm(num_slots, generator=g)[:N].to(torch.int32)
    else:
        idx = torch.tensor(list(state_indices), dtype=torch.int32)
    if has_initial_state is None:
        flags = torch.rand(N, generator=g) < init_prob
    else:
        flags = torch.tensor([bool(x) for x in has_initial_state], dtype=torch.bool)
    assert idx.numel() == N and flags.numel() == N

    return Workload(name=name, q=q, k=k, v=v, g_raw=g_raw, beta_raw=beta_raw,
                    cu_seqlens=cu, state_pool=pool, pool_storage=storage,
                    state_indices=idx, has_initial_state=flags,
                    lower_bound=lower_bound,
                    meta=dict(seed=seed, stride_pad=stride_pad, pool_std=pool_std))


def poison_unread_slots(w: Workload) -> None:
    """Fills the slots of sequences without an initial state with NaN: a
    correct kernel never reads them."""
    for n in range(w.num_seqs):
        if not bool(w.has_initial_state[n]):
            w.state_pool[int(w.state_indices[n])] = float("nan")


# ---------------------------------------------------------------------------
# The named serving workloads.
# ---------------------------------------------------------------------------

def tiny_varlen() -> Workload:
    """3 sequences of 37, 0 and 59 tokens, H=2, fp32 pool of 8 slots."""
    return make_workload("tiny_varlen", [37, 0, 59], 2, num_slots=8,
                         state_indices=[5, 2, 7], has_initial_state=[1, 0, 1],
                         seed=0)


def prefill_4k() -> Workload:
    """1 x 4096 tokens, H=12, fp32 pool of 64 slots with stride(0) padded by
    256 elements, one slot with an initial state."""
    return make_workload("prefill_1x4096_h12", [4096], 12, num_slots=64,
                         stride_pad=256, state_indices=[13],
                         has_initial_state=[1], seed=1)


def prefill_16k() -> Workload:
    """1 x 16384 tokens, H=12, contiguous fp32 pool of 64 slots, no initial
    state (the slot is poisoned with NaN)."""
    w = make_workload("prefill_1x16384_h12", [16384], 12, num_slots=64,
                      state_indices=[0], has_initial_state=[0], seed=2)
    poison_unread_slots(w)
    return w


def prefill_16k_raw_bf16() -> Workload:
    """The 1 x 16384, H=12 prefill with the raw gate and beta in bf16."""
    w = make_workload("prefill_1x16384_h12_rawbf16", [16384], 12, num_slots=64,
                      state_indices=[0], has_initial_state=[0], seed=2, raw_bf16=True)
    poison_unread_slots(w)
    return w


def prefill_16k_h2() -> Workload:
    """1 x 16384 tokens with 2 heads (a few-head shard of the long prefill),
    contiguous fp32 pool of 8 slots, no initial state."""
    w = make_workload("prefill_1x16384_h2", [16384], 2, num_slots=8,
                      state_indices=[0], has_initial_state=[0], seed=6)
    poison_unread_slots(w)
    return w


def _varlen_lengths(g: torch.Generator, n: int = 128, max_len: int = 2048,
                    p_empty: float = 0.05):
    empty = torch.rand(n, generator=g) < p_empty
    lens = torch.randint(1, max_len + 1, (n,), generator=g)
    lens[empty] = 0
    return lens.tolist()


def varlen_batch() -> Workload:
    """128 sequences, lengths 0 with probability 0.05 else uniform on
    [1, 2048], H=12, fp32 pool of 256 slots, random distinct slots,
    has_initial_state ~ Bernoulli(0.5)."""
    return make_workload("varlen_128seq_h12", [], 12, num_slots=256,
                         draw_lengths=_varlen_lengths, init_prob=0.5, seed=3)


def mixed_bf16_pool() -> Workload:
    """512 one-token (decode) sequences followed by 4 sequences of 2048 tokens,
    H=12, bf16 pool of 1024 slots; decode sequences carry a state, the prefill
    ones start from zero."""
    lengths = [1] * 512 + [2048] * 4
    flags = [1] * 512 + [0] * 4
    return make_workload("mixed_512x1_4x2048_bf16pool_h12", lengths, 12,
                         num_slots=1024, pool_dtype=torch.bfloat16,
                         has_initial_state=flags, seed=4)


WORKLOADS = {
    "tiny_varlen": tiny_varlen,
    "prefill_4k": prefill_4k,
    "prefill_16k": prefill_16k,
    "prefill_16k_raw_bf16": prefill_16k_raw_bf16,
    "prefill_16k_h2": prefill_16k_h2,
    "varlen_batch": varlen_batch,
    "mixed_bf16_pool": mixed_bf16_pool,
}
