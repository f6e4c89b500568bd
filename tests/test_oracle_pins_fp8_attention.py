"""Pins of the fp64 oracle's FP8 dot-product attention (CPU only).

Fixed from outside the oracle by cases whose casts are exact (one key gives v; equal scores give
the mean of the values; operands on the E4M3 grid at scale 1), by a scalar-loop restatement on a
tiny case, by the invariance of exact casts under power-of-two scales, by the exact attention in
the limit of operands on the grid, and by the size of the deviation from exact attention.
"""
import math

import numpy as np

from oracle import e4m3 as E4
from oracle import flux as O
from oracle import fp8_attention as A

RNG = np.random.default_rng(41)
GRID = np.array(sorted({E4.e4m3_decode(c) for c in range(256)} - {float("nan")}))
GRID = GRID[np.isfinite(GRID) & (np.abs(GRID) <= 8) & (np.abs(GRID) >= 2.0 ** -3)]


def _grid(shape):
    return RNG.choice(GRID, size=shape)


def test_one_key_gives_its_value_and_equal_scores_give_the_mean():
    v = _grid((1, 1, 16))
    q = RNG.standard_normal((1, 3, 16))
    k = RNG.standard_normal((1, 1, 16))
    # one key: Pt = 1 exactly, so O is the cast of v (exact at scale 1 for grid values)
    np.testing.assert_array_equal(A.fp8_attention(q, k, v, 1.0, 1.0, 1.0), np.broadcast_to(v, (1, 3, 16)))
    # q = 0: every score is 0, Pt = 1 for every key, O = the mean of the (grid) values
    v2 = _grid((1, 4, 16))
    o = A.fp8_attention(np.zeros((1, 2, 16)), RNG.standard_normal((1, 4, 16)), v2, 1.0, 1.0, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v2.mean(axis=1, keepdims=True), (1, 2, 16)), rtol=1e-15)


def test_scalar_loop_restatement_tiny():
    q, k, v = (RNG.standard_normal((5, 8)) for _ in range(3))
    sq, sk, sv = 100.0, 60.0, 200.0
    got = A.fp8_attention(q, k, v, sq, sk, sv)
    for i in range(5):
        scores = []
        for j in range(5):
            acc = 0.0
            for c in range(8):
                acc += float(E4.e4m3_quantize(q[i, c] * sq)) * float(E4.e4m3_quantize(k[j, c] * sk))
            scores.append(acc / (sq * sk) / math.sqrt(8))
        m = max(scores)
        pt = [math.exp(s - m) for s in scores]
        for c in range(8):
            o = sum(float(E4.e4m3_quantize(p * 448.0)) * float(E4.e4m3_quantize(v[j, c] * sv))
                    for j, p in enumerate(pt)) / (448.0 * sv) / sum(pt)
            assert abs(got[i, c] - o) <= 1e-13 * max(1.0, abs(o)), (i, c)


def test_power_of_two_scales_divide_out():
    # casts at scales 2^a and 2^(a+3) agree exactly while no element saturates or goes subnormal
    q, k, v = (RNG.uniform(0.5, 1.0, (2, 6, 16)) * RNG.choice([-1.0, 1.0], (2, 6, 16)) for _ in range(3))
    a = A.fp8_attention(q, k, v, 4.0, 8.0, 16.0)
    b = A.fp8_attention(q, k, v, 32.0, 64.0, 128.0)
    np.testing.assert_array_equal(a, b)


def test_grid_operands_give_exact_scores():
    # q, k on the grid at scale 1: the scores are exact, so the result differs from exact attention
    # only by the casts of Pt and v, at most a few E4M3 half-ulps of the output's scale
    q, k = _grid((2, 12, 32)) / 4, _grid((2, 12, 32)) / 4
    v = RNG.standard_normal((2, 12, 32))
    got = A.fp8_attention(q, k, v, 1.0, 1.0, 448.0 / np.abs(v).max())
    exact = O.attention(q, k, v)
    assert np.abs(got - exact).max() <= 3 * 2.0 ** -4 * np.abs(v).max()


def test_delayed_scales_stay_within_a_few_percent_of_exact_attention():
    # norm-wise: the three-bit mantissas of the operands and of Pt leave a few percent (about 5%
    # at 64 keys of N(0, 1) data); far more would mean a wrong scale, far less no cast at all
    q, k, v = (RNG.standard_normal((2, 3, 64, 128)) for _ in range(3))
    exact = O.attention(q, k, v)
    got = A.fp8_attention_delayed(q, k, v)
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert 0.01 < rel < 0.1, rel
