"""Pins the CPU oracle to things other than itself (brute force, closed forms,
invariants), and shows that plausible mistakes planted in a copy of it are
caught by those pins."""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from tests import kda_pins as pins


def _fwd(lib):
    def f(q, k, v, g_raw, beta_raw, cu, init, flags, lb, eps=pins.EPS):
        return oracle.forward(q, k, v, g_raw, beta_raw, cu, initial_state=init,
                              has_initial_state=flags, lower_bound=lb, eps=eps, lib=lib)
    return f


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check, oracle_lib):
    check(_fwd(oracle_lib))


@pytest.mark.parametrize("seed", [11, 12])
def test_brute_force_full_width(seed, oracle_lib):
    """K = V = 128 (the serving head size) against the unrolled form, with an
    empty sequence and a one-token sequence in the pack."""
    rng = np.random.default_rng(seed)
    c = pins.rand_case(rng, [3, 0, 1, 4], 2, 128, 128, init_scale=0.1)
    out, fin = oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                              c["init"], c["flags"], -5.0, lib=oracle_lib)
    bo, bf = pins.brute_force(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                              c["init"], c["flags"], -5.0)
    assert pins.rel(out, bo) < 1e-12
    assert pins.rel(fin, bf) < 1e-12


def test_brute_force_long_decay(oracle_lib):
    """Saturated decay (raw gate +8: ~5 nats per token and channel) over 40
    tokens, far past fp32 range for exp(-G): the token recurrence has no
    overflow and matches the unrolled form."""
    rng = np.random.default_rng(13)
    c = pins.rand_case(rng, [40], 1, 8, 3)
    c["g_raw"][:] = 8.0
    out, fin = oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                              c["init"], c["flags"], -5.0, lib=oracle_lib)
    bo, bf = pins.brute_force(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                              c["init"], c["flags"], -5.0)
    assert np.isfinite(out).all()
    assert pins.rel(out, bo) < 1e-12 and pins.rel(fin, bf) < 1e-11


def test_paged_wrapper_semantics(oracle_lib):
    """Pool semantics of the oracle: selected slots get the final states
    (empty sequences included), unselected slots are returned bit-identical,
    a slot without has_initial_state is never read."""
    rng = np.random.default_rng(14)
    c = pins.rand_case(rng, [3, 0, 2], 2, 6, 4)
    pool = rng.standard_normal((6, 2, 4, 6))
    idx = np.array([4, 1, 2])
    flags = np.array([1, 0, 0], bool)
    pool[1] = np.nan
    pool[2] = np.nan
    out, newpool = oracle.forward_paged(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"],
                                        c["cu"], pool, idx, flags, lower_bound=-5.0,
                                        lib=oracle_lib)
    assert np.isfinite(out).all()
    for s in (0, 3, 5):
        assert np.array_equal(newpool[s], pool[s])
    assert np.array_equal(newpool[1], np.zeros_like(pool[1]))  # empty, no init -> zeros
    init = np.stack([pool[4], np.zeros_like(pool[4]), np.zeros_like(pool[4])])
    o2, f2 = oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                            init, flags.astype(np.uint8), -5.0, lib=oracle_lib)
    assert np.array_equal(out, o2)
    assert np.array_equal(newpool[4], f2[0]) and np.array_equal(newpool[2], f2[2])


def test_rejects_bad_bounds(oracle_lib):
    rng = np.random.default_rng(15)
    c = pins.rand_case(rng, [2, 2], 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], np.array([0, 3, 2]),
                       None, np.zeros(2, np.uint8), -5.0, lib=oracle_lib)


# ---------------------------------------------------------------------------
# Mutation check: each plausible mistake, planted in a temporary copy of the
# oracle source, must make at least one pin fail.
# ---------------------------------------------------------------------------

MUTANTS = {
    "decay_sign": ("decay[c] = exp(lower_bound * sigmoid(g_raw[c]));",
                   "decay[c] = exp(-lower_bound * sigmoid(g_raw[c]));"),
    "no_decay": ("for (int c = 0; c < K; ++c) s[c] *= dec[c];",
                 "(void)dec;"),
    "decay_on_rows": ("for (int c = 0; c < K; ++c) s[c] *= dec[c];",
                      "for (int c = 0; c < K; ++c) s[c] *= dec[v0 + r];"),
    "no_beta": ("const double d = beta * (v[tv + v0 + r] - sk);",
                "const double d = (v[tv + v0 + r] - sk);"),
    "beta_not_sigmoid": ("*beta = sigmoid(beta_raw);", "*beta = beta_raw;"),
    "no_sqrt_k": ("double rq = 1.0 / sqrt(sq + eps) / sqrt((double)K);",
                  "double rq = 1.0 / sqrt(sq + eps);"),
    "k_not_normalised": ("double rk = 1.0 / sqrt(sk + eps);", "double rk = 1.0;"),
    "output_uses_k": ("for (int c = 0; c < K; ++c) o += s[c] * qn[c];",
                      "for (int c = 0; c < K; ++c) o += s[c] * kn[c];"),
    "gate_not_sigmoid": ("decay[c] = exp(lower_bound * sigmoid(g_raw[c]));",
                         "decay[c] = exp(lower_bound * g_raw[c]);"),
    "reads_unflagged_init": ("if (has_init && has_init[n]) {", "if (init) {"),
    "write_uses_q": ("for (int c = 0; c < K; ++c) s[c] += d * kn[c];",
                     "for (int c = 0; c < K; ++c) s[c] += d * qn[c] * sqrt((double)K);"),
    "decay_after_write": [
        ("for (int c = 0; c < K; ++c) s[c] *= dec[c];", "/* no decay before the write */"),
        ("for (int c = 0; c < K; ++c) s[c] += d * kn[c];",
         "for (int c = 0; c < K; ++c) s[c] += d * kn[c];\n"
         "for (int c = 0; c < K; ++c) s[c] *= dec[c];")],
    "output_before_write": [
        ("const double d = beta * (v[tv + v0 + r] - sk);",
         "double o0 = 0.0; for (int c = 0; c < K; ++c) o0 += s[c] * qn[c];\n"
         "const double d = beta * (v[tv + v0 + r] - sk);"),
        ("out[tv + v0 + r] = o;", "out[tv + v0 + r] = o0; (void)o;")],
    "beta_on_erase_only": ("const double d = beta * (v[tv + v0 + r] - sk);",
                           "const double d = v[tv + v0 + r] - beta * sk;"),
    "lower_bound_ignored": ("decay[c] = exp(lower_bound * sigmoid(g_raw[c]));",
                            "decay[c] = exp(-sigmoid(g_raw[c]));"),
    "last_token_skipped": ("for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {",
                           "for (int64_t t = cu[n]; t + 1 < cu[n + 1]; ++t) {"),
    "init_ignored": ("if (has_init && has_init[n]) {", "if (0 && has_init && has_init[n]) {"),
    "row_block_offset_dropped": [
        ("v[tv + v0 + r]", "v[tv + r]"),
        ("out[tv + v0 + r] = o;", "out[tv + r] = o;"),
        ("const size_t sbase = ((size_t)n * H + h) * plane + (size_t)v0 * K;",
         "const size_t sbase = ((size_t)n * H + h) * plane;")],
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="kda_oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # a planted mistake may overflow
def test_pins_catch_mutant(name, mutant_dir):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    edits = MUTANTS[name]
    for old, new in ([edits] if isinstance(edits, tuple) else edits):
        assert src.count(old) == 1, f"mutation anchor for {name} not found once in the source"
        src = src.replace(old, new, 1)
    msrc = os.path.join(mutant_dir, f"{name}.c")
    with open(msrc, "w") as f:
        f.write(src)
    mlib = os.path.join(mutant_dir, f"lib{name}.so")
    oracle.build(msrc, mlib)
    lib = oracle.load(mlib)
    fwd = _fwd(lib)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(fwd)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


def test_golden_fixture(oracle_lib):
    """The stored oracle fixture (written by tests/golden/make_golden.py) is
    reproduced by the oracle and, independently, by the unrolled form."""
    import json
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small_varlen.json")
    fx = json.load(open(path))
    args = [np.array(fx[n]) for n in ("q", "k", "v", "g_raw", "beta_raw")]
    cu = np.array(fx["cu_seqlens"])
    init = np.array(fx["initial_state"])
    flags = np.array(fx["has_initial_state"], np.uint8)
    out, fin = oracle.forward(*args, cu, init, flags, fx["lower_bound"], fx["eps"], lib=oracle_lib)
    assert np.allclose(out, np.array(fx["out"]), rtol=1e-14, atol=1e-16)
    assert np.allclose(fin, np.array(fx["final_state"]), rtol=1e-14, atol=1e-16)
    bo, bf = pins.brute_force(*args, cu, init, flags, fx["lower_bound"], fx["eps"])
    assert pins.rel(np.array(fx["out"]), bo) < 1e-12
    assert pins.rel(np.array(fx["final_state"]), bf) < 1e-12


def test_scalar_closed_form(oracle_lib):
    """K = V = 1, eps = 0: k^ = q^ = 1, and with raw gate 0 and lower_bound
    -2 ln 2 the decay is exactly 1/2; raw beta 0 gives b = 1/2.  The recurrence
    is then S_t = S_{t-1}/2 * (1 - 1/2) + v_t/2, so from S_0 = 4 with
    v = (2, 4, 8): S = (2, 2.5, 4.625), and o_t = S_t."""
    T = 3
    one = np.ones((T, 1, 1))
    v = np.array([2.0, 4.0, 8.0]).reshape(T, 1, 1)
    out, fin = oracle.forward(one, one, v, np.zeros((T, 1, 1)), np.zeros((T, 1)),
                              np.array([0, T]), np.full((1, 1, 1, 1), 4.0), np.ones(1, np.uint8),
                              -2.0 * np.log(2.0), 0.0, lib=oracle_lib)
    assert np.allclose(out.ravel(), [2.0, 2.5, 4.625], rtol=1e-15, atol=0)
    assert np.allclose(fin.ravel(), [4.625], rtol=1e-15, atol=0)
