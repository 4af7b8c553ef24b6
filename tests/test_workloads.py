"""CPU tests of the seeded input generators (kda_prefill_gb300/workloads.py):
they are deterministic, hold the sizes, bounds, slots, flags, canaries and
poisoned slots each named workload states, and share nothing with either side
of the parity comparison."""
import ast
import math
import os

import torch

from kda_prefill_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PLANE = 128 * 128


def _fields(w):
    return [w.q, w.k, w.v, w.g_raw, w.beta_raw, w.cu_seqlens, w.pool_storage,
            w.state_indices, w.has_initial_state]


def _same_bytes(a, b):
    return a.dtype == b.dtype and a.shape == b.shape and torch.equal(
        a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def test_same_seed_same_bytes_other_seed_other_values():
    a = wl.make_workload("a", [37, 0, 59], 2, num_slots=8, seed=5)
    b = wl.make_workload("b", [37, 0, 59], 2, num_slots=8, seed=5)
    c = wl.make_workload("c", [37, 0, 59], 2, num_slots=8, seed=6)
    assert all(_same_bytes(x, y) for x, y in zip(_fields(a), _fields(b)))
    assert not torch.equal(a.q, c.q)


def test_tiny_varlen_recipe():
    w = wl.tiny_varlen()
    assert w.cu_seqlens.tolist() == [0, 37, 37, 96]
    assert w.num_heads == 2 and w.total_tokens == 96
    assert w.state_indices.tolist() == [5, 2, 7]
    assert w.has_initial_state.tolist() == [True, False, True]
    assert tuple(w.state_pool.shape) == (8, 2, 128, 128)
    assert w.state_pool.dtype == torch.float32 and w.lower_bound == -5.0
    assert w.q.dtype == torch.bfloat16 and w.g_raw.dtype == torch.float32
    assert tuple(w.beta_raw.shape) == (1, 96, 2)
    # pool drawn with standard deviation 0.1
    assert 0.08 < float(w.state_pool.std()) < 0.12


def test_prefill_4k_padded_stride_holds_canaries():
    w = wl.prefill_4k()
    S, stride0 = w.pool_storage.shape
    assert (S, stride0) == (64, 12 * PLANE + 256)
    assert w.state_pool.stride(0) == stride0
    canary = w.pool_storage[:, 12 * PLANE:].view(torch.int32)
    assert bool((canary == wl.CANARY_F32_BITS).all())
    assert w.state_indices.tolist() == [13] and w.has_initial_state.tolist() == [True]
    assert torch.isfinite(w.state_pool[13]).all()


def test_prefill_16k_poisons_the_unread_slot():
    w = wl.prefill_16k()
    assert w.total_tokens == 16384 and w.num_heads == 12 and w.num_seqs == 1
    assert w.state_indices.tolist() == [0] and w.has_initial_state.tolist() == [False]
    assert bool(torch.isnan(w.state_pool[0]).all())
    assert torch.isfinite(w.state_pool[1:]).all()


def test_q_k_v_are_bf16_draws_of_unit_normals():
    w = wl.make_workload("stats", [4096], 4, num_slots=2, seed=9)
    for x in (w.q, w.k, w.v, w.g_raw):
        f = x.float()
        assert abs(float(f.mean())) < 0.01 and abs(float(f.std()) - 1.0) < 0.01


def test_varlen_length_draw():
    """Length 0 with probability 0.05, else uniform on [1, 2048]: the draw of
    the varlen batch (seed 3, lengths first in the stream)."""
    g = torch.Generator().manual_seed(3)
    lens = wl._varlen_lengths(g)
    assert len(lens) == 128
    assert all(0 <= x <= 2048 for x in lens)
    n_empty = sum(1 for x in lens if x == 0)
    assert n_empty <= 20  # binomial(128, 0.05): mean 6.4
    # the draw itself (its mean would be 128 * 0.95 * 1024.5, about 124.6K tokens)
    assert (sum(lens), n_empty) == (113251, 8)
    # a larger draw of the same rule shows its two parts
    big = wl._varlen_lengths(torch.Generator().manual_seed(11), n=20000)
    frac_empty = sum(1 for x in big if x == 0) / len(big)
    assert abs(frac_empty - 0.05) < 4 * math.sqrt(0.05 * 0.95 / len(big))
    nz = torch.tensor([x for x in big if x > 0], dtype=torch.float64)
    assert int(nz.min()) == 1 and int(nz.max()) == 2048
    assert abs(float(nz.mean()) - 1024.5) < 20


def test_default_slots_are_distinct_and_flags_follow_the_rule():
    w = wl.make_workload("slots", [3] * 40, 1, num_slots=64, seed=12, init_prob=0.5)
    idx = w.state_indices.tolist()
    assert len(set(idx)) == 40 and all(0 <= s < 64 for s in idx)
    assert w.has_initial_state.dtype == torch.bool
    assert 5 < int(w.has_initial_state.sum()) < 35


def test_mixed_pool_shape_rule_on_a_small_copy():
    """The mixed batch's rule (one-token sequences with a state first, then
    prefills without) on fewer sequences, with the 2-byte pool's canary."""
    lengths = [1] * 6 + [70] * 2
    w = wl.make_workload("mixed_small", lengths, 2, num_slots=16, pool_dtype=torch.bfloat16,
                         stride_pad=8, has_initial_state=[1] * 6 + [0] * 2, seed=4)
    assert w.total_tokens == 146 and w.state_pool.dtype == torch.bfloat16
    assert len(set(w.state_indices.tolist())) == 8
    assert bool((w.pool_storage[:, 2 * PLANE:].view(torch.int16) == wl.CANARY_16_BITS).all())
    assert w.has_initial_state.tolist() == [True] * 6 + [False] * 2


def test_raw_bf16_rounds_after_the_same_draw():
    a = wl.make_workload("a", [50], 2, num_slots=2, seed=8)
    b = wl.make_workload("b", [50], 2, num_slots=2, seed=8, raw_bf16=True)
    assert b.g_raw.dtype == torch.bfloat16 and b.beta_raw.dtype == torch.bfloat16
    assert torch.equal(a.g_raw.to(torch.bfloat16), b.g_raw)
    assert torch.equal(a.beta_raw.to(torch.bfloat16), b.beta_raw)
    assert torch.equal(a.q, b.q) and torch.equal(a.pool_storage, b.pool_storage)


def test_generator_module_imports_neither_side():
    """The inputs module may serve both sides only if it depends on neither."""
    src = open(os.path.join(ROOT, "kda_prefill_gb300", "workloads.py")).read()
    mods = set()
    for node in ast.walk(ast.parse(src)):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            mods.add((node.module or "").split(".")[0] if node.level == 0 else ".")
    assert mods <= {"__future__", "dataclasses", "typing", "torch"}, mods
