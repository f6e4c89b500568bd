"""Pins of the fp64 oracle's attention, rectified-flow loss and E4M3 quantiser (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3 as E
from oracle import flux as O

RNG = np.random.default_rng(11)


# ----------------------------------------------------------------------------- attention
def _brute_attention(q, k, v):
    """Triple loop over (query, key, feature): the textbook softmax attention."""
    S, d = q.shape
    T = k.shape[0]
    out = np.zeros((S, v.shape[1]))
    for i in range(S):
        scores = []
        for j in range(T):
            acc = 0.0
            for f in range(d):
                acc += q[i, f] * k[j, f]
            scores.append(acc / math.sqrt(d))
        mx = max(scores)
        w = [math.exp(sc - mx) for sc in scores]
        z = sum(w)
        for j in range(T):
            for f in range(v.shape[1]):
                out[i, f] += w[j] / z * v[j, f]
    return out


def test_attention_brute_force():
    # P4: brute force on S <= 48
    q = RNG.standard_normal((13, 8))
    k = RNG.standard_normal((48, 8))
    v = RNG.standard_normal((48, 5))
    np.testing.assert_allclose(O.attention(q, k, v), _brute_attention(q, k, v), rtol=1e-12, atol=1e-13)


def test_attention_matches_torch_sdpa():
    q = RNG.standard_normal((2, 3, 17, 16))
    k = RNG.standard_normal((2, 3, 29, 16))
    v = RNG.standard_normal((2, 3, 29, 16))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v)).numpy()
    np.testing.assert_allclose(O.attention(q, k, v), ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    v = RNG.standard_normal((9, 6))
    k = RNG.standard_normal((9, 4))
    # one key -> that value exactly
    q = RNG.standard_normal((3, 4))
    np.testing.assert_allclose(O.attention(q, k[:1], v[:1]), np.repeat(v[:1], 3, 0), rtol=1e-15)
    # q = 0 -> uniform weights -> mean of the values
    np.testing.assert_allclose(O.attention(np.zeros((2, 4)), k, v), np.repeat(v.mean(0, keepdims=True), 2, 0),
                               rtol=1e-13)
    # rows of the weight matrix sum to 1: attention of V = ones gives ones
    np.testing.assert_allclose(O.attention(q, k, np.ones((9, 3))), 1.0, rtol=1e-14)
    # large scores do not overflow (max subtraction)
    out = O.attention(1e3 * q, 1e3 * k, v)
    assert np.all(np.isfinite(out))


# ----------------------------------------------------------------------------- flow matching
def test_flow_match_endpoints_and_loss():
    z0 = RNG.standard_normal((3, 4, 5, 6))
    z1 = RNG.standard_normal((3, 4, 5, 6))
    # P9
    np.testing.assert_array_equal(O.flow_match_noise(z0, z1, np.zeros(3)), z0)
    np.testing.assert_array_equal(O.flow_match_noise(z0, z1, np.ones(3)), z1)
    t = np.array([0.25, 0.5, 0.9])
    zt = O.flow_match_noise(z0, z1, t)
    # z_t lies on the straight line: z_t - z0 = t (z1 - z0) per sample
    for b in range(3):
        np.testing.assert_allclose(zt[b] - z0[b], t[b] * (z1[b] - z0[b]), rtol=1e-12, atol=1e-14)
    target = O.flow_match_target(z0, z1)
    assert O.flow_match_loss(target, z0, z1) == 0.0
    # a constant offset c gives loss c^2
    assert O.flow_match_loss(target + 0.3, z0, z1) == pytest.approx(0.09, rel=1e-12)
    # matches torch's mean-reduced MSE
    pred = RNG.standard_normal(z0.shape)
    ref = torch.nn.functional.mse_loss(torch.from_numpy(pred), torch.from_numpy(z1 - z0)).item()
    assert O.flow_match_loss(pred, z0, z1) == pytest.approx(ref, rel=1e-13)


def test_flow_match_loss_of_zero_prediction_is_about_two():
    z0 = RNG.standard_normal((2, 64, 32, 32))
    z1 = RNG.standard_normal((2, 64, 32, 32))
    assert O.flow_match_loss(np.zeros_like(z0), z0, z1) == pytest.approx(2.0, rel=0.02)


# ----------------------------------------------------------------------------- E4M3
def test_e4m3_special_values(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_special_values.json")))
    for c in g["codes"]:
        assert E.e4m3_decode(c["code"]) == c["value"], c
    assert math.isnan(E.e4m3_decode(g["nan_code"]))
    assert math.isnan(E.e4m3_decode(g["nan_code"] | 0x80))


def test_e4m3_exhaustive_round_trip():
    # P10: every finite code round-trips through encode(decode(code)).
    for code in range(256):
        v = E.e4m3_decode(code)
        if math.isnan(v):
            continue
        got = int(E.e4m3_encode(np.array([v]))[0])
        if v == 0.0:
            assert got in (0x00, 0x80)
        else:
            assert got == code, (code, v, got)


def test_e4m3_saturation_and_ties_to_even():
    assert E.e4m3_quantize(np.array([500.0, -1e30, 448.0, 449.0]))[:].tolist() == [448, -448, 448, 448]
    # midpoint of 1.0 (code 0x38, even) and 1.125 (0x39, odd) -> 1.0; midpoint of 1.125 and 1.25 -> 1.25
    assert E.e4m3_quantize(np.array([1.0625, 1.1875])).tolist() == [1.0, 1.25]
    # half the smallest subnormal ties to zero (even); a hair more rounds up
    assert E.e4m3_quantize(np.array([2.0 ** -10, 2.0 ** -10 * 1.0001])).tolist() == [0.0, 2.0 ** -9]
    # amax maps to 448 under the delayed scale
    x = RNG.standard_normal(1000)
    s = E.delayed_scale(np.abs(x).max())
    assert np.abs(E.e4m3_quantize(x * s)).max() == 448.0
    assert E.delayed_scale(None) == 1.0 and E.delayed_scale(0.0) == 1.0


def test_e4m3_matches_torch_float8_cast_on_float32_inputs():
    x = torch.linspace(-460, 460, 200001, dtype=torch.float32)
    ref = x.clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(E.e4m3_quantize(x.double().numpy()), ref)
    small = torch.linspace(-0.03, 0.03, 100001, dtype=torch.float32)
    np.testing.assert_array_equal(E.e4m3_quantize(small.double().numpy()),
                                  small.to(torch.float8_e4m3fn).double().numpy())


def test_fp8_linear_is_exact_on_representable_operands():
    # operands already on the E4M3 grid at scale 1 multiply exactly
    codes = RNG.integers(0x30, 0x48, size=(4, 6))
    x = np.vectorize(E.e4m3_decode)(codes)
    w = np.vectorize(E.e4m3_decode)(RNG.integers(0x30, 0x48, size=(3, 6)))
    np.testing.assert_array_equal(E.fp8_linear(x, w, None, 1.0, 1.0), x @ w.T)


# ----------------------------------------------------------------------------- sampling
def test_cfg_combine_special_cases():
    vc, vu = RNG.standard_normal(50), RNG.standard_normal(50)
    # w = 1 gives the conditional velocity, w = 0 the unconditional one (to rounding)
    np.testing.assert_allclose(O.cfg_combine(vc, vu, 1.0), vc, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(O.cfg_combine(vc, vu, 0.0), vu)
    # affine in w: the midpoint of w = 1 and w = 3 is w = 2
    np.testing.assert_allclose(O.cfg_combine(vc, vu, 2.0),
                               0.5 * (O.cfg_combine(vc, vu, 1.0) + O.cfg_combine(vc, vu, 3.0)), atol=1e-14)


def test_euler_is_exact_on_the_straight_line_flow():
    # z_t = (1 - t) z0 + t z1 has the constant velocity z1 - z0: stepping from z1 (t = 1) to
    # t = 0 in any number of Euler steps lands on z0, and every intermediate is z_t
    z0, z1 = RNG.standard_normal(40), RNG.standard_normal(40)
    v = O.flow_match_target(z0, z1)
    for n in (1, 4, 10):
        z, t = z1.copy(), 1.0
        for _ in range(n):
            z = O.euler_step(z, v, 1.0 / n)
            t -= 1.0 / n
            np.testing.assert_allclose(z, O.flow_match_noise(z0[None], z1[None], np.array([t]))[0],
                                       atol=1e-12)
        np.testing.assert_allclose(z, z0, atol=1e-12)
