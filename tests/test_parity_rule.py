"""The comparison rule of the GPU parity gates, checked on synthetic rows: an
argmax mismatch fails a row whatever the oracle's margin ("Reproducing Kipp",
section "Model-backed CPU and Metal gates": identical argmax and NMSE <=
1e-4); a near tie is only flagged."""
import numpy as np

from helpers import AMBIGUOUS_MARGIN, NMSE_BOUND, check_row


def test_argmax_mismatch_fails_even_on_a_near_tie():
    ref = np.linspace(-1, 1, 1000).astype(np.float32)
    ref[10] = ref[-1] - AMBIGUOUS_MARGIN / 10                 # a near tie with the top logit
    got = ref.copy()
    got[10] = ref[-1] + 1e-4                                  # the GPU tips it the other way
    c = check_row(got, ref)
    assert c.nmse <= NMSE_BOUND and c.ambiguous
    assert c.argmax_gpu != c.argmax_ref and not c.ok


def test_flag_does_not_depend_on_the_gpu_error():
    ref = np.linspace(-1, 1, 1000).astype(np.float32)
    noisy = ref + np.random.default_rng(0).normal(0, 1e-3, ref.shape).astype(np.float32)
    noisy[-1] = ref[-1] + 1.0                                 # keeps the argmax
    a, b = check_row(ref.copy(), ref), check_row(noisy, ref)
    assert a.ambiguous == b.ambiguous                         # fixed margin, not scaled by the error
    assert a.ok and b.argmax_gpu == b.argmax_ref


def test_nmse_over_the_bound_fails():
    ref = np.linspace(-1, 1, 1000).astype(np.float32)
    got = ref * 1.1
    assert not check_row(got, ref).ok
