"""The parity tests' bf16 tap-rounding tie allowance, checked on the CPU.

A tie is a tap whose exact value lies within the FP32 accumulation error of a
bf16 rounding midpoint: both roundings are correct results.  The helper must
report one bf16 spacing for such a tap and nothing for a tap clear of any
midpoint, and the per-element allowance must add spacing * |operand| over the
element's tied taps only.
"""
import numpy as np

import oracle
from parity import dx_tie_allowance, forward_tie_allowance, tap_tie_flip


def _one_tap_problem(t_value):
    # C = 1, K = 1: one tap per dilation, T = W[o, 0] * y + bias[o] with y = 1
    y = np.ones((1, 1, 1, 1))
    w = np.full((3, 1), t_value)
    b = np.zeros(3)
    return y, w, b


def test_tie_at_a_midpoint_flips_by_one_spacing():
    mid = 1.0 + 2.0 ** -8            # halfway between the bf16 values 1 and 1 + 2^-7
    y, w, b = _one_tap_problem(mid)
    assert tap_tie_flip(oracle, y, w, b, 1, (1, 1, 1), 0, 0, 0, 0) == 2.0 ** -7


def test_tap_clear_of_midpoints_is_not_a_tie():
    y, w, b = _one_tap_problem(1.0 + 2.0 ** -10)
    assert tap_tie_flip(oracle, y, w, b, 1, (1, 1, 1), 0, 0, 0, 0) == 0.0
    y, w, b = _one_tap_problem(3.0)
    assert tap_tie_flip(oracle, y, w, b, 1, (1, 1, 1), 0, 0, 0, 0) == 0.0


def test_allowances_sum_spacing_times_operand_over_tied_taps():
    mid = 1.0 + 2.0 ** -8
    y = np.ones((1, 1, 1, 1))
    w = np.array([[mid], [2.0], [mid]])     # dilations 0 and 2 tied, dilation 1 exact
    b = np.zeros(3)
    x = np.full((1, 1, 1, 1), -3.0)
    h64 = {"x": x, "y": y, "weight": w, "bias": b, "grad_out": np.array([0.5, 1.0, 2.0, 4.0]).reshape(1, 4, 1, 1)}
    # out channels 1, 2, 3 = dilations 0, 1, 2; channel 0 is x itself
    got = forward_tie_allowance(oracle, h64, 1, (1, 1, 1), np.arange(4))
    np.testing.assert_array_equal(got, [0.0, 3.0 * 2.0 ** -7, 0.0, 3.0 * 2.0 ** -7])
    # dx gathers tap * grad of blocks 1..3: the tied taps meet grad 1.0 and 4.0
    got = dx_tie_allowance(oracle, h64, 1, (1, 1, 1), np.arange(1))
    np.testing.assert_array_equal(got, [(1.0 + 4.0) * 2.0 ** -7])
