"""Pins for the parity metrics every GPU test reports through.

The metrics are the plainest reading of "relative error" for a tensor: the
normwise-max error (largest absolute difference over the largest reference
magnitude), its per-slice form (each sequence and head judged against its own
scale), and the elementwise error |x - y| / (|y| + 1e-6 max|y|), whose median is
reported beside it.  The values below are worked by hand, so a wrong
denominator, swapped operands or a silent broadcast fails here rather than
making every GPU parity test vacuous.
"""
import numpy as np
import pytest

import oracle


def test_rel_err_hand_values():
    # |[1,2,3] - [1,2,5]| = [0,0,2]; max |ref| = 5  ->  2/5
    assert oracle.rel_err([1.0, 2.0, 3.0], [1.0, 2.0, 5.0]) == pytest.approx(0.4, abs=0)
    # the denominator is the reference's scale, not the candidate's
    assert oracle.rel_err([1.0, 2.0, 5.0], [1.0, 2.0, 3.0]) == pytest.approx(2.0 / 3.0)
    # max of |diff| and max of |ref| are taken separately, over all entries, signs ignored
    assert oracle.rel_err([[-4.0, 0.5], [0.0, 1.0]], [[-3.0, 0.0], [0.0, 8.0]]) == pytest.approx(
        7.0 / 8.0)
    assert oracle.rel_err([2.0, -1.0], [2.0, -1.0]) == 0.0


def test_rel_err_all_zero_reference_is_the_absolute_max():
    assert oracle.rel_err([0.0, -0.25, 0.125], [0.0, 0.0, 0.0]) == 0.25
    assert oracle.rel_err(np.zeros(4), np.zeros(4)) == 0.0
    assert oracle.rel_err(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0


def test_rel_err_rejects_shape_mismatch():
    with pytest.raises(ValueError):
        oracle.rel_err([1.0, 2.0, 3.0], [1.0, 2.0])
    with pytest.raises(ValueError):  # would broadcast silently
        oracle.rel_err(np.ones((3, 4)), np.ones((1, 4)))
    with pytest.raises(ValueError):
        oracle.rel_err(np.ones(4), np.ones((4, 1)))


def test_rel_err_slices_hand_values():
    ref = np.array([[[1.0, 2.0], [100.0, -50.0]],
                    [[0.0, 0.0], [0.5, 0.25]]])
    x = np.array([[[1.0, 2.5], [100.0, -49.0]],
                  [[0.0, 0.125], [0.5, 0.25]]])
    per = oracle.rel_err_slices(x, ref, 2)
    assert per.shape == (2, 2)
    assert per[0, 0] == pytest.approx(0.25)        # 0.5 / 2
    assert per[0, 1] == pytest.approx(0.01)        # 1 / 100
    assert per[1, 0] == pytest.approx(0.125)       # zero reference: absolute max
    assert per[1, 1] == 0.0
    # the whole-tensor metric hides the small slice's 25% error behind the large one
    assert oracle.rel_err(x, ref) == pytest.approx(1.0 / 100.0)
    assert oracle.rel_err_slices(x, ref, 1) == pytest.approx([0.01, 0.25])
    assert oracle.rel_err_slices(x, ref, 0) == pytest.approx(oracle.rel_err(x, ref))
    with pytest.raises(ValueError):
        oracle.rel_err_slices(x, ref[:1], 1)


def test_rel_err_slices_floor_hand_values():
    """The optional floor: denominators of at least floor_frac x the median slice scale."""
    ref = np.array([[4.0, 0.0], [2.0, -8.0], [0.01, 0.0], [1.0, 1.0]])  # slice maxima 4, 8, 0.01, 1
    x = ref + np.array([[0.0, 0.04], [0.0, 0.0], [0.0005, 0.0], [0.0, 0.0]])
    plain = oracle.rel_err_slices(x, ref, 1)
    assert plain == pytest.approx([0.01, 0.0, 0.05, 0.0])
    # median of (4, 8, 0.01, 1) is 2.5; a floor of 0.1 x 2.5 = 0.25 lifts only the third slice
    floored = oracle.rel_err_slices(x, ref, 1, floor_frac=0.1)
    assert floored == pytest.approx([0.01, 0.0, 0.0005 / 0.25, 0.0])


def test_rel_err_segments_hand_values():
    """Packed [tokens][heads][channels]: sequences of 2, 0 and 1 tokens, 2 heads."""
    ref = np.zeros((3, 2, 2))
    ref[0, 0] = [1.0, -2.0]; ref[1, 0] = [0.5, 0.0]      # seq 0, head 0: max |ref| 2
    ref[0, 1] = [10.0, 0.0]; ref[1, 1] = [0.0, 4.0]      # seq 0, head 1: max 10
    ref[2, 0] = [0.0, 0.0]                               # seq 2, head 0: all zero
    ref[2, 1] = [3.0, -1.0]                              # seq 2, head 1: max 3
    x = ref.copy()
    x[1, 0, 1] = 0.1      # seq 0 head 0: 0.1 / 2
    x[0, 1, 1] = -1.0     # seq 0 head 1: 1 / 10
    x[2, 0, 0] = 0.25     # seq 2 head 0: zero reference -> absolute 0.25
    e = oracle.rel_err_segments(x, ref, [0, 2, 2, 3])
    assert e.shape == (3, 2)
    assert e[0] == pytest.approx([0.05, 0.1])
    assert e[1] == pytest.approx([0.0, 0.0])
    assert e[2] == pytest.approx([0.25, 0.0])
    # floor: median of the non-empty slice scales (2, 10, 0, 3) is 2.5 -> denominators >= 0.25
    f = oracle.rel_err_segments(x, ref, [0, 2, 2, 3], floor_frac=0.1)
    assert f[2, 0] == pytest.approx(1.0) and f[0, 0] == pytest.approx(0.05)
    with pytest.raises(ValueError):
        oracle.rel_err_segments(x, ref, [0, 2, 4])
    with pytest.raises(ValueError):
        oracle.rel_err_segments(x, ref[:2], [0, 2])


def test_elementwise_rel_hand_values():
    ref = np.array([4.0, -2.0, 0.0, 1000.0])
    x = np.array([5.0, -2.0, 0.001, 1000.0])
    e = oracle.elementwise_rel(x, ref)
    floor = 1e-6 * 1000.0
    assert e[0] == pytest.approx(1.0 / (4.0 + floor))
    assert e[1] == 0.0
    assert e[2] == pytest.approx(0.001 / floor)   # a zero entry is judged against the floor
    assert e[3] == 0.0
    assert float(np.median(e)) == pytest.approx(0.5 * (1.0 / (4.0 + floor)))
    with pytest.raises(ValueError):
        oracle.elementwise_rel(x, ref[:3])


@pytest.mark.parametrize("mistake", ["den_from_x", "swapped_means", "no_abs"])
def test_metric_pins_catch_planted_mistakes(mistake):
    """Plausible slips in the metric, planted in a copy, each fail a hand value."""
    def bad(x, ref):
        x, ref = np.asarray(x, float), np.asarray(ref, float)
        if mistake == "den_from_x":
            return np.max(np.abs(x - ref)) / np.max(np.abs(x))
        if mistake == "swapped_means":
            return np.max(np.abs(ref)) / max(np.max(np.abs(x - ref)), 1e-300)
        return np.max(x - ref) / np.max(ref)
    cases = [(([1.0, 2.0, 3.0], [1.0, 2.0, 5.0]), 0.4),
             (([[-4.0, 0.5], [0.0, 1.0]], [[-3.0, 0.0], [0.0, 8.0]]), 7.0 / 8.0)]
    assert any(abs(bad(*args) - want) > 1e-9 for args, want in cases)
    assert all(abs(oracle.rel_err(*args) - want) < 1e-12 for args, want in cases)
