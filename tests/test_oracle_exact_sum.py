"""Pins the oracle's scale sum to a library routine.

s = (1/B) sum_i g_max(i) ("AdaComp (Adaptive Residual Gradient Compression)", Claims >
Mechanism #r629-local-bin-soft-threshold-and-mean-gmax-quantization). The oracle sums
the fp32 maxima exactly and rounds once to fp64; Python's math.fsum returns exactly
that (the correctly rounded sum of its double inputs, and fp32 values are exact
doubles).
"""
import math

import numpy as np
import pytest

import oracle


def _fsum(x):
    return math.fsum(np.asarray(x, np.float32).astype(np.float64))


@pytest.mark.parametrize("seed", range(6))
def test_random_magnitudes(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 20000))
    e = rng.uniform(-40, 40, n)
    x = (rng.random(n) * 2.0 ** e).astype(np.float32)
    assert oracle.exact_sum_f32(x) == _fsum(x)


def test_wide_dynamic_range_and_subnormals():
    x = np.array([3.0e38, 1.0, 2.0 ** -149, 2.0 ** -126, 1e-45, 7.5, 3.0e38, 1e-30],
                 np.float32)
    assert oracle.exact_sum_f32(x) == _fsum(x)


def test_sum_that_a_left_to_right_double_sum_gets_wrong():
    x = np.array([4.0, 2.0 ** -22] + [2.0 ** -52] * 3, np.float32)
    left = 0.0
    for v in x.astype(np.float64):
        left += v
    assert oracle.exact_sum_f32(x) == _fsum(x) == 4.0 + 2.0 ** -22 + 2.0 ** -50
    assert left != _fsum(x)


def test_many_equal_terms_round_to_even():
    # 2^53 + 1 is a tie between 2^53 and 2^53 + 2: the even one wins
    x = np.concatenate([np.full(2 ** 21, 2.0 ** 32, np.float32), np.ones(1, np.float32)])
    assert oracle.exact_sum_f32(x) == _fsum(x) == 2.0 ** 53


def test_empty_and_zero():
    assert oracle.exact_sum_f32(np.zeros(0, np.float32)) == 0.0
    assert oracle.exact_sum_f32(np.zeros(5, np.float32)) == 0.0
