"""Writes the oracle regression fixtures in this folder.

It calls only ``oracle/`` on inputs drawn here with a fixed seed, and stores the
inputs with the outputs as text.  The fixture anchors the oracle's arithmetic:
a later change that moves these numbers has to say which reading of the
recurrence justifies it.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(2024)
    lengths = [3, 0, 4]
    H, K, V = 1, 4, 3
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    q = np.round(rng.standard_normal((T, H, K)), 3)
    k = np.round(rng.standard_normal((T, H, K)), 3)
    v = np.round(rng.standard_normal((T, H, V)), 3)
    g = np.round(rng.standard_normal((T, H, K)), 3)
    b = np.round(rng.standard_normal((T, H)), 3)
    init = np.round(rng.standard_normal((3, H, V, K)) * 0.1, 3)
    flags = np.array([1, 0, 1], np.uint8)
    out, fin = oracle.forward(q, k, v, g, b, cu, init, flags, lower_bound=-5.0)
    fx = dict(
        what="KDA forward, fp64 oracle, lower_bound=-5, eps=1e-6, K=4, V=3, H=1",
        lower_bound=-5.0, eps=oracle.L2_EPS, cu_seqlens=cu.tolist(),
        has_initial_state=flags.tolist(), q=q.tolist(), k=k.tolist(), v=v.tolist(),
        g_raw=g.tolist(), beta_raw=b.tolist(), initial_state=init.tolist(),
        out=[[[float(repr_) for repr_ in row] for row in t] for t in out.tolist()],
        final_state=fin.tolist(),
    )
    with open(os.path.join(HERE, "oracle_small_varlen.json"), "w") as f:
        json.dump(fx, f, indent=1)


if __name__ == "__main__":
    main()
