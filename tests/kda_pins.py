"""Independent checks that pin the oracle (used by test_oracle_pins.py and by the
mutation test, which re-runs them against deliberately broken oracle builds).

Every check here is computed without the oracle's own code path:

* ``brute_force`` evaluates the recurrence as products of explicit K x K
  transition matrices, S_t = S_0 M_1..M_t + sum_s b_s v_s k_s^T M_{s+1}..M_t,
  instead of the oracle's in-place rank-1 updates;
* the closed forms follow from the definition of the gated delta rule by hand
  (no decay and no write, pure decay, one token, the delta-rule write that
  makes S k = v when b = 1).

The recurrence (V-first state, per-channel decay):
    S_t = S_{t-1} Diag(exp g_t) (I - b_t k_t k_t^T) + b_t v_t k_t^T,
    o_t = S_t q_t / sqrt(K),  q, k L2-normalised, g = lb*sigmoid(g_raw),
    b = sigmoid(beta_raw).
Sources: ROCm/aiter PR #4741 (Summary; "Optimizations Applied": L2 norm,
lower-bounded-sigmoid gate, beta sigmoid, zero padding is a no-op) and PR #5754
("Technical Details": has_initial_state = false starts from zero).
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def brute_force(q, k, v, g_raw, beta_raw, cu, init, flags, lb, eps=EPS):
    T, H, K = q.shape
    V = v.shape[2]
    N = len(cu) - 1
    out = np.zeros((T, H, V))
    fin = np.zeros((N, H, V, K))
    I = np.eye(K)
    for n in range(N):
        for h in range(H):
            S0 = init[n, h].copy() if flags[n] else np.zeros((V, K))
            toks = list(range(cu[n], cu[n + 1]))
            Ms, Ws, Qs = [], [], []
            for t in toks:
                kn = k[t, h] / np.sqrt(np.dot(k[t, h], k[t, h]) + eps)
                qn = q[t, h] / np.sqrt(np.dot(q[t, h], q[t, h]) + eps) / np.sqrt(K)
                a = np.exp(lb * _sig(g_raw[t, h]))
                b = _sig(beta_raw[t, h])
                Ms.append(np.diag(a) @ (I - b * np.outer(kn, kn)))
                Ws.append(b * np.outer(v[t, h], kn))
                Qs.append(qn)
            S = S0
            for i, t in enumerate(toks):
                P = np.eye(K)
                for s in range(i + 1):
                    P = P @ Ms[s]
                S = S0 @ P
                for s in range(i + 1):
                    R = np.eye(K)
                    for r in range(s + 1, i + 1):
                        R = R @ Ms[r]
                    S = S + Ws[s] @ R
                out[t, h] = S @ Qs[i]
            fin[n, h] = S
    return out, fin


def rand_case(rng, lengths, H, K, V, init_scale=0.3, gate_scale=1.0):
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = rng.standard_normal((T, H, K)) * gate_scale
    b = rng.standard_normal((T, H))
    N = len(lengths)
    init = rng.standard_normal((N, H, V, K)) * init_scale
    flags = (rng.random(N) < 0.6).astype(np.uint8)
    return dict(q=q, k=k, v=v, g_raw=g, beta_raw=b, cu=cu, init=init, flags=flags)


def rel(x, y):
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


# ---------------------------------------------------------------------------
# The checks.  Each returns None on success and raises AssertionError on a
# mismatch.  ``fwd`` is the oracle's dense forward with the signature of
# ``oracle.forward``.
# ---------------------------------------------------------------------------

def check_brute_force(fwd, seed=0, K=6, V=4, H=2, lb=-5.0):
    rng = np.random.default_rng(seed)
    c = rand_case(rng, [5, 0, 9, 1], H, K, V)
    out, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                   c["init"], c["flags"], lb)
    bo, bfin = brute_force(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"],
                           c["cu"], c["init"], c["flags"], lb)
    assert rel(out, bo) < 1e-12, rel(out, bo)
    assert rel(fin, bfin) < 1e-12, rel(fin, bfin)


def check_brute_force_wide(fwd, seed=7, K=24, V=40, H=2, lb=-5.0):
    """The unrolled form with more value rows than one work block of the oracle
    holds (16), and a ragged last block: every row's inputs, initial state,
    output and final state land at its own index."""
    rng = np.random.default_rng(seed)
    c = rand_case(rng, [4, 0, 3], H, K, V)
    flags = np.array([1, 0, 1], np.uint8)
    out, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                   c["init"], flags, lb)
    bo, bfin = brute_force(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"],
                           c["cu"], c["init"], flags, lb)
    assert rel(out, bo) < 1e-12, rel(out, bo)
    assert rel(fin, bfin) < 1e-12, rel(fin, bfin)


def check_noop_tokens(fwd, K=6, V=4, H=2, lb=-5.0):
    """raw gate = raw beta = -inf gives g = 0 and b = 0: the state is carried
    unchanged and every output is S_0 q^."""
    rng = np.random.default_rng(1)
    c = rand_case(rng, [7], H, K, V)
    c["g_raw"][:] = -np.inf
    c["beta_raw"][:] = -np.inf
    flags = np.ones(1, np.uint8)
    out, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                   c["init"], flags, lb)
    assert np.array_equal(fin[0], c["init"][0])
    for t in range(7):
        for h in range(H):
            qn = c["q"][t, h] / np.sqrt(np.dot(c["q"][t, h], c["q"][t, h]) + EPS) / np.sqrt(K)
            assert np.allclose(out[t, h], c["init"][0, h] @ qn, rtol=1e-13, atol=1e-15)


def check_pure_decay(fwd, K=6, V=4, H=2, lb=-3.0):
    """b = 0: S_T = S_0 Diag(exp(sum_t lb*sigmoid(g_raw_t)))."""
    rng = np.random.default_rng(2)
    c = rand_case(rng, [6], H, K, V)
    c["beta_raw"][:] = -np.inf
    flags = np.ones(1, np.uint8)
    _, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                 c["init"], flags, lb)
    for h in range(H):
        G = (lb * _sig(c["g_raw"][:, h, :])).sum(axis=0)
        want = c["init"][0, h] * np.exp(G)[None, :]
        assert np.allclose(fin[0, h], want, rtol=1e-12, atol=0)


def check_single_token(fwd, K=6, V=4, H=2, lb=-5.0):
    """S_0 = 0, one token: S_1 = b v k^T and o = b (k^.q^) v = b cos(q,k) v / sqrt(K)."""
    rng = np.random.default_rng(3)
    c = rand_case(rng, [1], H, K, V)
    flags = np.zeros(1, np.uint8)
    out, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                   None, flags, lb)
    for h in range(H):
        q, k, v = c["q"][0, h], c["k"][0, h], c["v"][0, h]
        b = _sig(c["beta_raw"][0, h])
        cos = np.dot(q, k) / np.sqrt(np.dot(q, q) + EPS) / np.sqrt(np.dot(k, k) + EPS)
        assert np.allclose(out[0, h], b * cos * v / np.sqrt(K), rtol=1e-12, atol=1e-15)
        kn = k / np.sqrt(np.dot(k, k) + EPS)
        assert np.allclose(fin[0, h], b * np.outer(v, kn), rtol=1e-12, atol=1e-15)


def check_delta_write(fwd, K=6, V=4, H=2, lb=-5.0):
    """b = 1 (raw beta = 40 rounds sigmoid to exactly 1 in fp64) and eps = 0
    (so |k^| = 1): after every token S_t k^_t = v_t, whatever came before."""
    rng = np.random.default_rng(4)
    c = rand_case(rng, [5], H, K, V)
    c["beta_raw"][:] = 40.0
    flags = np.ones(1, np.uint8)
    # Recover S_t from the per-prefix final states by calling on each prefix.
    for t in range(1, 6):
        cu = np.array([0, t], np.int64)
        _, fin = fwd(c["q"][:t], c["k"][:t], c["v"][:t], c["g_raw"][:t],
                     c["beta_raw"][:t], cu, c["init"], flags, lb, 0.0)
        for h in range(H):
            kk = c["k"][t - 1, h]
            kn = kk / np.linalg.norm(kk)
            assert np.allclose(fin[0, h] @ kn, c["v"][t - 1, h], rtol=1e-12, atol=1e-13)


def check_zero_init_flag(fwd, K=6, V=4, H=2, lb=-5.0):
    """has_initial_state = 0 equals a zero initial state, even when the given
    initial state is NaN (it must not be read)."""
    rng = np.random.default_rng(5)
    c = rand_case(rng, [4, 3], H, K, V)
    nan_init = np.full_like(c["init"], np.nan)
    zeros = np.zeros_like(c["init"])
    flags0 = np.zeros(2, np.uint8)
    flags1 = np.ones(2, np.uint8)
    o1, f1 = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], nan_init, flags0, lb)
    o2, f2 = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], zeros, flags1, lb)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)
    assert np.isfinite(o1).all() and np.isfinite(f1).all()


def check_empty_sequence(fwd, K=6, V=4, H=2, lb=-5.0):
    """An empty sequence returns its initial state (zeros without one)."""
    rng = np.random.default_rng(6)
    c = rand_case(rng, [0, 3, 0], H, K, V)
    flags = np.array([1, 1, 0], np.uint8)
    _, fin = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], c["init"], flags, lb)
    assert np.array_equal(fin[0], c["init"][0])
    assert np.array_equal(fin[2], np.zeros_like(fin[2]))


def check_row_permutation(fwd, K=6, V=5, H=1, lb=-5.0):
    """V rows are independent: permuting the rows of v and of S_0 permutes the
    output channels and the final-state rows the same way."""
    rng = np.random.default_rng(7)
    c = rand_case(rng, [6], H, K, V)
    flags = np.ones(1, np.uint8)
    perm = rng.permutation(V)
    o1, f1 = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], c["init"], flags, lb)
    o2, f2 = fwd(c["q"], c["k"], c["v"][:, :, perm], c["g_raw"], c["beta_raw"], c["cu"],
                 c["init"][:, :, perm, :], flags, lb)
    assert np.allclose(o2, o1[:, :, perm], rtol=1e-13, atol=1e-15)
    assert np.allclose(f2, f1[:, :, perm, :], rtol=1e-13, atol=1e-15)


def check_scale_invariance(fwd, K=6, V=4, H=2, lb=-5.0):
    """q and k enter only through their directions (up to the norm's eps)."""
    rng = np.random.default_rng(8)
    c = rand_case(rng, [5], H, K, V)
    flags = np.ones(1, np.uint8)
    o1, f1 = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], c["init"], flags, lb, 0.0)
    o2, f2 = fwd(c["q"] * 7.0, c["k"] * 0.25, c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                 c["init"], flags, lb, 0.0)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(f1, f2, rtol=1e-12, atol=1e-14)


def check_split_call(fwd, K=6, V=4, H=2, lb=-5.0):
    """Running a sequence in one call equals running it in two calls that hand
    the state over (fp64 state: bit-equal)."""
    rng = np.random.default_rng(9)
    c = rand_case(rng, [9], H, K, V)
    flags = np.ones(1, np.uint8)
    o, f = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], c["init"], flags, lb)
    s = 4
    oa, fa = fwd(c["q"][:s], c["k"][:s], c["v"][:s], c["g_raw"][:s], c["beta_raw"][:s],
                 np.array([0, s]), c["init"], flags, lb)
    ob, fb = fwd(c["q"][s:], c["k"][s:], c["v"][s:], c["g_raw"][s:], c["beta_raw"][s:],
                 np.array([0, 9 - s]), fa, flags, lb)
    assert np.array_equal(np.concatenate([oa, ob]), o)
    assert np.array_equal(fb, f)


def check_sequence_independence(fwd, K=6, V=4, H=2, lb=-5.0):
    """Sequences packed together do not interact."""
    rng = np.random.default_rng(10)
    c = rand_case(rng, [3, 5], H, K, V)
    o, f = fwd(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"], c["init"], c["flags"], lb)
    o2, f2 = fwd(c["q"][3:], c["k"][3:], c["v"][3:], c["g_raw"][3:], c["beta_raw"][3:],
                 np.array([0, 5]), c["init"][1:], c["flags"][1:], lb)
    assert np.array_equal(o[3:], o2) and np.array_equal(f[1], f2[0])


ALL_CHECKS = [
    check_brute_force,
    check_brute_force_wide, check_noop_tokens, check_pure_decay, check_single_token,
    check_delta_write, check_zero_init_flag, check_empty_sequence,
    check_row_permutation, check_scale_invariance, check_split_call,
    check_sequence_independence,
]
