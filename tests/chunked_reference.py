"""Chunked fp64 staging reference (tests only).

Evaluates the chunkwise form of the gated delta rule that the CUDA kernels
implement, step by step, in fp64 numpy: the per-chunk decay-weighted tiles,
the unit-lower-triangular solve, w and u, then the serial walk over chunks.
It is checked against the token-by-token oracle, which pins the chunk algebra
independently of the GPU; the GPU tests can diff intermediate tiles with it.

Inside a chunk with cumulative log-decay G_i (per channel) and incoming S_0:
  A_kk[i,j] = b_i sum_c k_ic k_jc e^{G_ic-G_jc} (j<i),  A_qk[i,j] (j<=i) alike with q_i
  T = (I + A_kk)^{-1},  w = T (b k e^G),  u = T (b v)
  U = u - w S_0^T,  o = (q e^G) S_0^T + A_qk U,  S_C = S_0 Diag(e^{G_C}) + U^T (k e^{G_C-G})
"""
import numpy as np


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def chunk_tiles(q, k, v, g_raw, beta_raw, lb, eps=1e-6):
    """One chunk of one head (rows already padded with zeros / beta 0 / g 0)."""
    C, K = q.shape
    qn = q / np.sqrt((q * q).sum(1, keepdims=True) + eps) / np.sqrt(K)
    kn = k / np.sqrt((k * k).sum(1, keepdims=True) + eps)
    g = lb * _sig(g_raw)
    b = _sig(beta_raw)
    G = np.cumsum(g, axis=0)
    diff = G[:, None, :] - G[None, :, :]               # [i, j, c]
    mask_l = np.tril(np.ones((C, C), bool), -1)
    mask_le = np.tril(np.ones((C, C), bool), 0)
    E = np.exp(np.where(mask_le[:, :, None], diff, -np.inf))
    Akk = b[:, None] * np.einsum("ic,jc,ijc->ij", kn, kn, E) * mask_l
    Aqk = np.einsum("ic,jc,ijc->ij", qn, kn, E) * mask_le
    Tm = np.linalg.inv(np.eye(C) + Akk)
    w = Tm @ (b[:, None] * kn * np.exp(G))
    u = Tm @ (b[:, None] * v)
    qg = qn * np.exp(G)
    kg = kn * np.exp(G[-1][None, :] - G)
    gamma = np.exp(G[-1])
    return dict(Akk=Akk, Aqk=Aqk, T=Tm, w=w, u=u, qg=qg, kg=kg, gamma=gamma)


def forward(q, k, v, g_raw, beta_raw, cu, init, flags, lb, C=64, eps=1e-6):
    T_, H, K = q.shape
    V = v.shape[2]
    N = len(cu) - 1
    out = np.zeros((T_, H, V))
    fin = np.zeros((N, H, V, K))
    for n in range(N):
        for h in range(H):
            S = init[n, h].copy() if flags[n] else np.zeros((V, K))
            for t0 in range(cu[n], cu[n + 1], C):
                L = min(C, cu[n + 1] - t0)
                pad = lambda x, fill=0.0: np.concatenate(
                    [x, np.full((C - L,) + x.shape[1:], fill)]) if L < C else x
                qq = pad(q[t0:t0 + L, h])
                kk = pad(k[t0:t0 + L, h])
                vv = pad(v[t0:t0 + L, h])
                gg = pad(g_raw[t0:t0 + L, h], -np.inf)   # g = 0 on padded rows
                bb = pad(beta_raw[t0:t0 + L, h], -np.inf)  # beta = 0 on padded rows
                tl = chunk_tiles(qq, kk, vv, gg, bb, lb, eps)
                U = tl["u"] - tl["w"] @ S.T
                o = tl["qg"] @ S.T + tl["Aqk"] @ U
                out[t0:t0 + L, h] = o[:L]
                S = S * tl["gamma"][None, :] + U.T @ tl["kg"]
            fin[n, h] = S
    return out, fin


# ---------------------------------------------------------------------------
# Segmented walk.  Each chunk maps the state affinely, S -> S M_c + N_c with
# M_c = Diag(gamma) - w^T kg and N_c = u^T kg, so a run of chunks maps its start
# state S to S Phi + N: Phi is the walk of the K identity rows with u = 0, N the
# walk of a zero state.  The segments' (Phi, N) are independent of one another
# and of the incoming state; chaining S_start(s + 1) = S_start(s) Phi_s + N_s and
# walking each segment from its start state gives the serial walk's outputs and
# final state.  (ROCm/aiter PR #4741, "Optimizations Applied", splits the state
# walk of long sequences into segments; the page does not give the composition,
# which follows from each chunk's affine map of the state.)
# ---------------------------------------------------------------------------

def _padded_tiles(q, k, v, g_raw, beta_raw, lb, t_begin, t_end, h, C, eps):
    """(first token, valid rows, tiles) of the chunks of tokens t_begin..t_end-1."""
    tiles = []
    for t0 in range(t_begin, t_end, C):
        L = min(C, t_end - t0)

        def pad(x, fill=0.0):
            return np.concatenate([x, np.full((C - L,) + x.shape[1:], fill)]) if L < C else x

        tl = chunk_tiles(pad(q[t0:t0 + L, h]), pad(k[t0:t0 + L, h]), pad(v[t0:t0 + L, h]),
                         pad(g_raw[t0:t0 + L, h], -np.inf), pad(beta_raw[t0:t0 + L, h], -np.inf),
                         lb, eps)
        tiles.append((t0, L, tl))
    return tiles


def _walk(S, tiles, zero_u=False, out=None, h=None):
    """The serial walk over `tiles` from state S (rows of any count); with
    zero_u the chunks' u are taken as 0; with `out` the outputs are written."""
    for t0, L, tl in tiles:
        u = np.zeros((tl["w"].shape[0], S.shape[0])) if zero_u else tl["u"]
        U = u - tl["w"] @ S.T
        if out is not None:
            out[t0:t0 + L, h] = (tl["qg"] @ S.T + tl["Aqk"] @ U)[:L]
        S = S * tl["gamma"][None, :] + U.T @ tl["kg"]
    return S


def forward_segmented(q, k, v, g_raw, beta_raw, cu, init, flags, lb, C=64, seg_chunks=2,
                      eps=1e-6):
    """The chunkwise forward with each sequence's walk cut into segments of
    seg_chunks chunks: pass A (Phi, N of every segment but the last), the chain of
    segment start states, pass B (every segment from its start state)."""
    T_, H, K = q.shape
    V = v.shape[2]
    N = len(cu) - 1
    out = np.zeros((T_, H, V))
    fin = np.zeros((N, H, V, K))
    for n in range(N):
        for h in range(H):
            tiles = _padded_tiles(q, k, v, g_raw, beta_raw, lb, cu[n], cu[n + 1], h, C, eps)
            segs = [tiles[i:i + seg_chunks] for i in range(0, len(tiles), seg_chunks)] or [[]]
            phi = [_walk(np.eye(K), sg, zero_u=True) for sg in segs[:-1]]
            nst = [_walk(np.zeros((V, K)), sg) for sg in segs[:-1]]
            starts = [init[n, h].copy() if flags[n] else np.zeros((V, K))]
            for s in range(len(segs) - 1):
                starts.append(starts[s] @ phi[s] + nst[s])
            for s, sg in enumerate(segs):
                S = _walk(starts[s], sg, out=out, h=h)
            fin[n, h] = S
    return out, fin


# ---------------------------------------------------------------------------
# Bounded construction of the decay factors e^{G_i - G_j} (j <= i) of one chunk,
# as the tensor-core intra kernel forms them: the chunk is cut into 16-row
# blocks; with a = e^g per token and channel, P_i the product of a over block
# rows up to i and E_B a block's total, a pair in blocks J < I is
# P_i * (E_{J+1} ... E_{I-1}) * (E_J / P_j) and a pair inside one block P_i / P_j.
# Every factor of the off-diagonal form is <= 1, so nothing overflows whatever
# the decay; the diagonal quotient needs P >= ~e^-87 in fp32, which holds while
# a block's 16 tokens decay by at most 80 nats (lower_bound >= -5).
# ---------------------------------------------------------------------------

def bounded_decay_pairs(g_raw, lb, dtype=np.float32, block=16):
    """[C, C, K] factors e^{G_i - G_j} for j <= i (0 above the diagonal),
    evaluated in `dtype` by the bounded construction."""
    C, K = g_raw.shape
    a = np.exp((lb * _sig(g_raw.astype(np.float64))).astype(dtype)).astype(dtype)
    nb = C // block
    P = np.empty_like(a)
    E = np.empty((nb, K), dtype)
    for B in range(nb):
        acc = np.ones(K, dtype)
        for r in range(block):
            acc = (acc * a[B * block + r]).astype(dtype)
            P[B * block + r] = acc
        E[B] = acc
    out = np.zeros((C, C, K), dtype)
    for i in range(C):
        I = i // block
        for j in range(i + 1):
            J = j // block
            if I == J:
                out[i, j] = P[i] / P[j]
            else:
                mid = np.ones(K, dtype)
                for B in range(J + 1, I):
                    mid = (mid * E[B]).astype(dtype)
                out[i, j] = P[i] * mid * (E[J] / P[j])
    return out


# ---------------------------------------------------------------------------
# Operand-rounding model of the kernels' precision choices.  Every tensor-core
# operand is rounded to the type it is stored in; sums are exact (fp64), since
# fp32 accumulation adds far less error than 10- or 7-bit operand mantissas.
#   "kernel": diagonal 16-row blocks of A_qk / A_kk from tf32 operands, every
#             other operand fp16 (off-diagonal factors, the middle-block decay
#             table, T's off-diagonal blocks, w, u, qg, kg, A_qk, U and the
#             state operand), the state master copy and gamma unrounded, out bf16;
#   "bf16":   the same with every one of those operands in bf16;
#   "diag_bf16": the kernel's choice except for bf16 diagonal blocks.
# ---------------------------------------------------------------------------

def _round_bits(x, drop):
    """Round-to-nearest-even of fp32 values to (23 - drop) mantissa bits."""
    f = np.asarray(x, np.float32).copy()
    u = f.view(np.uint32)
    bias = np.uint32((1 << (drop - 1)) - 1) + ((u >> np.uint32(drop)) & np.uint32(1))
    u[:] = (u + bias) & ~np.uint32((1 << drop) - 1)
    return f.astype(np.float64)


def rnd(x, kind):
    if kind == "fp16":
        return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)
    if kind == "tf32":
        return _round_bits(x, 13)
    if kind == "bf16":
        return _round_bits(x, 16)
    return np.asarray(x, np.float64)


def forward_rounded(q, k, v, g_raw, beta_raw, cu, lb, prec="kernel", C=64, block=16,
                    eps=1e-6):
    """Outputs [T, H, V] of zero-initial-state sequences under the rounding model."""
    diag_t, op_t = {"kernel": ("tf32", "fp16"), "bf16": ("bf16", "bf16"),
                    "diag_bf16": ("bf16", "fp16")}[prec]
    T_, H, K = q.shape
    V = v.shape[2]
    out = np.zeros((T_, H, V))
    nb = C // block
    blk = np.arange(C) // block
    for n in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((V, K))
            for t0 in range(cu[n], cu[n + 1], C):
                L = min(C, cu[n + 1] - t0)
                qq, kk, vv = (np.zeros((C, K)), np.zeros((C, K)), np.zeros((C, V)))
                gg = np.full((C, K), -np.inf)
                bb = np.full(C, -np.inf)
                qq[:L], kk[:L], vv[:L] = q[t0:t0 + L, h], k[t0:t0 + L, h], v[t0:t0 + L, h]
                gg[:L], bb[:L] = g_raw[t0:t0 + L, h], beta_raw[t0:t0 + L, h]
                qn = qq / np.sqrt((qq * qq).sum(1, keepdims=True) + eps) / np.sqrt(K)
                kn = kk / np.sqrt((kk * kk).sum(1, keepdims=True) + eps)
                g = lb * _sig(gg)
                b = _sig(bb)
                G = np.cumsum(g, axis=0)
                a = np.exp(g)
                P = np.empty_like(a)
                E = np.empty((nb, K))
                for B in range(nb):
                    P[B * block:(B + 1) * block] = np.cumprod(a[B * block:(B + 1) * block], axis=0)
                    E[B] = P[(B + 1) * block - 1]
                R = E[blk] / P                      # E_J / P_j
                Aqk = np.zeros((C, C))
                Akk = np.zeros((C, C))
                for I in range(nb):
                    ri = slice(I * block, (I + 1) * block)
                    for J in range(I + 1):
                        rj = slice(J * block, (J + 1) * block)
                        if I == J:
                            right = rnd(kn[rj] / P[rj], diag_t)
                            lq, lk = rnd(qn[ri] * P[ri], diag_t), rnd(kn[ri] * P[ri], diag_t)
                        else:
                            mid = rnd(np.prod(E[J + 1:I], axis=0), op_t)
                            right = rnd(kn[rj] * R[rj], op_t)
                            lq = rnd(rnd(qn[ri] * P[ri], op_t) * mid, op_t)
                            lk = rnd(rnd(kn[ri] * P[ri], op_t) * mid, op_t)
                        Aqk[ri, rj] = lq @ right.T
                        Akk[ri, rj] = b[ri, None] * (lk @ right.T)
                Aqk = np.tril(Aqk)
                Akk = np.tril(Akk, -1)
                off = blk[:, None] != blk[None, :]
                Akk_r = np.where(off, rnd(Akk, op_t), Akk)   # diagonal blocks solved in fp32
                Tm = np.linalg.inv(np.eye(C) + Akk_r)
                w = rnd(Tm @ rnd(b[:, None] * kn * np.exp(G), op_t), op_t)
                u = rnd(Tm @ rnd(b[:, None] * vv, op_t), op_t)
                qg = rnd(qn * np.exp(G), op_t)
                kg = rnd(kn * np.exp(G[-1][None, :] - G), op_t)
                Aqk = rnd(Aqk, op_t)
                gamma = np.exp(G[-1])
                Sr = rnd(S, op_t)
                U = rnd(u - w @ Sr.T, op_t)
                out[t0:t0 + L, h] = rnd(qg @ Sr.T + Aqk @ U, "bf16")[:L]
                S = S * gamma[None, :] + U.T @ kg
    return out
