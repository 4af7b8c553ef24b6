"""The chunkwise algebra the kernels implement equals the token recurrence
(oracle) in fp64, for several chunk sizes, ragged tails and saturated gates."""
import numpy as np
import pytest

import oracle
from tests import chunked_reference as cref
from tests import kda_pins as pins


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("gate_scale,lb", [(1.0, -5.0), (0.0, 0.0), (8.0, -5.0)])
def test_chunked_equals_token_recurrence(C, gate_scale, lb, oracle_lib):
    rng = np.random.default_rng(C)
    c = pins.rand_case(rng, [1, C - 1, C, C + 1, 0, 3 * C + 5], 2, 16, 8,
                       gate_scale=gate_scale)
    o1, f1 = oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                            c["init"], c["flags"], lb, lib=oracle_lib)
    o2, f2 = cref.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                          c["init"], c["flags"], lb, C=C)
    assert pins.rel(o2, o1) < 1e-10
    assert pins.rel(f2, f1) < 1e-10


@pytest.mark.parametrize("C,seg_chunks,gate_scale", [(16, 1, 1.0), (16, 3, 1.0), (32, 2, 1.0),
                                                     (16, 2, 8.0)])
def test_segmented_walk_equals_token_recurrence(C, seg_chunks, gate_scale, oracle_lib):
    """The segment composition the segmented scan uses (pass A from zero and
    over identity rows with u = 0, the chain of start states, pass B) gives the
    token recurrence's outputs and final states."""
    rng = np.random.default_rng(100 + C + seg_chunks)
    c = pins.rand_case(rng, [5 * C + 3, 0, C, 2 * C + 1, 4], 2, 16, 8, gate_scale=gate_scale)
    o1, f1 = oracle.forward(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"], c["cu"],
                            c["init"], c["flags"], -5.0, lib=oracle_lib)
    o2, f2 = cref.forward_segmented(c["q"], c["k"], c["v"], c["g_raw"], c["beta_raw"],
                                    c["cu"], c["init"], c["flags"], -5.0, C=C,
                                    seg_chunks=seg_chunks)
    assert pins.rel(o2, o1) < 1e-10
    assert pins.rel(f2, f1) < 1e-10
