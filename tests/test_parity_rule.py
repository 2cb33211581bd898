"""The comparison rule of the GPU parity gates, checked on synthetic rows
("Reproducing Kipp", section "Model-backed CPU and Metal gates": identical
argmax and NMSE <= 1e-4).  An argmax mismatch fails unless the oracle's own
top-two margin is below a fixed fraction of its logits' RMS, and even then
the GPU's pick must lie within that margin of the top; the threshold does not
move with the GPU's error."""
import numpy as np

from helpers import AMBIGUOUS_REL, NMSE_BOUND, check_row


def _ref():
    r = np.random.default_rng(1).normal(0, 1, 4096).astype(np.float32)
    r[7] = r.max() + 0.5                                        # a clear top
    return r


def test_a_clear_argmax_must_match():
    ref = _ref()
    ref[8] = ref[7] - 0.1                                       # runner-up, a clear margin below
    got = ref.copy()
    got[8] = ref[7] + 1e-3                                      # the GPU picks the runner-up
    c = check_row(got, ref)
    assert not c.ambiguous and c.nmse <= NMSE_BOUND
    assert not c.ok


def test_a_near_tie_may_flip_to_the_runner_up_only():
    ref = _ref()
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    ref[9] = ref[7] - 0.2 * AMBIGUOUS_REL * rms                # a near tie with index 7
    got = ref.copy()
    got[9] = ref[7] + 1e-6
    c = check_row(got, ref)
    assert c.ambiguous and c.argmax_gpu == 9 and c.ok
    far = ref.copy()
    far[100] = ref[7] + 1e-6                                    # picks an index far below the top
    c2 = check_row(far, ref)
    assert c2.ambiguous and c2.argmax_gpu == 100 and not c2.ok


def test_threshold_does_not_move_with_the_gpu_error():
    ref = _ref()
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    ref[9] = ref[7] - 2 * AMBIGUOUS_REL * rms                  # outside the threshold
    noisy = ref + np.random.default_rng(2).normal(0, 5e-3, ref.shape).astype(np.float32)
    noisy[9] = noisy[7] + 1.0                                   # a noisy GPU tips it over
    c = check_row(noisy, ref)
    assert not c.ambiguous and not c.ok


def test_nmse_over_the_bound_fails():
    ref = _ref()
    assert not check_row(ref * 1.1, ref).ok
