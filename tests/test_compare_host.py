"""CPU test of the GPU tests' comparison helper: the per-sequence check finds a
wrong result confined to one short sequence of a pack, which the rel-L2 over
the whole pack lets through."""
import numpy as np

from tests.gpu_helpers import per_sequence_rel_l2, rel_l2


def test_per_sequence_check_catches_one_bad_short_sequence():
    rng = np.random.default_rng(0)
    lengths = [6000, 3, 0, 4000]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = int(cu[-1])
    o_ref = rng.standard_normal((T, 2, 128))
    f_ref = rng.standard_normal((len(lengths), 2, 128, 128))
    o_gpu = o_ref * (1 + 1e-3 * rng.standard_normal(o_ref.shape))
    f_gpu = f_ref * (1 + 1e-3 * rng.standard_normal(f_ref.shape))
    # the 3-token sequence is wrong by 20 %
    o_gpu[6000:6003] *= 1.2
    assert rel_l2(o_gpu, o_ref) < 5e-3            # the whole pack passes
    wo, ws = per_sequence_rel_l2(o_gpu, o_ref, f_gpu, f_ref, cu)
    assert wo > 0.15 and ws < 5e-3                  # the sequence check does not
    # a wrong final state of the empty sequence is caught as well
    f_gpu[2] = 0.0
    _, ws = per_sequence_rel_l2(o_gpu, o_ref, f_gpu, f_ref, cu)
    assert ws == 1.0
