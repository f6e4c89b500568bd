"""Pins of the fp64 oracle's E5M2 quantiser and of the FP8 linear backward (CPU only).

E5M2 is pinned against the IEEE half-precision encoding it is the upper byte of (the FP8 formats
paper defines it that way) and against torch's float8_e5m2 cast; the FP8 backward against the
exact backward where the casts are exact, against the format grids where one operand is the
identity, against brute force on a tiny case and against the rounding error bound of the formats.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import backward as BW
from oracle import e4m3 as E4
from oracle import e5m2 as E5
from oracle import fp8_backward as F

RNG = np.random.default_rng(23)
E4M3_GRID = np.array(sorted({E4.e4m3_decode(c) for c in range(256)} - {float("nan")}))
E5M2_VALUES = np.array([E5.e5m2_decode(c) for c in range(256)])


def _on_grid(v, grid):
    """Whether each value is a finite grid value, up to the float64 rounding of one scaling."""
    v = np.asarray(v, np.float64).ravel()
    g = np.sort(grid[np.isfinite(grid)])
    i = np.clip(np.searchsorted(g, v), 1, len(g) - 1)
    near = np.where(np.abs(g[i] - v) < np.abs(g[i - 1] - v), g[i], g[i - 1])
    return np.abs(near - v) <= 1e-12 * np.abs(v)


# ----------------------------------------------------------------------------- E5M2 format
def test_e5m2_decode_is_the_upper_byte_of_ieee_half():
    halves = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    for c in range(256):
        if math.isnan(halves[c]):
            assert math.isnan(E5.e5m2_decode(c)), hex(c)
        else:
            assert E5.e5m2_decode(c) == halves[c], hex(c)
    assert E5.e5m2_decode(0x7B) == 57344.0 == E5.E5M2_MAX
    assert E5.e5m2_decode(0x01) == 2.0 ** -16
    assert E5.e5m2_decode(0x04) == 2.0 ** -14  # smallest normal
    assert E5.e5m2_decode(0x7C) == math.inf and E5.e5m2_decode(0xFC) == -math.inf
    assert sum(math.isnan(E5.e5m2_decode(c)) for c in range(256)) == 6


def test_e5m2_encode_matches_round_to_nearest_even_on_the_half_bit_pattern():
    # every finite half: dropping the low byte of the magnitude with round-to-nearest-even is
    # the E5M2 rounding, saturated at 0x7B
    bits = np.arange(0x10000, dtype=np.uint32)
    mag = bits & 0x7FFF
    finite = mag < 0x7C00
    bits, mag = bits[finite], mag[finite]
    vals = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    r = (mag + 0x7F + ((mag >> 8) & 1)) >> 8
    r = np.minimum(r, 0x7B)
    want = (r | ((bits >> 15) << 7)).astype(np.uint8)
    np.testing.assert_array_equal(E5.e5m2_encode(vals), want)


def test_e5m2_saturation_specials_and_ties():
    q = E5.e5m2_quantize(np.array([1e6, -1e30, np.inf, -np.inf, 57344.0, 61439.0, 61440.0]))
    assert q.tolist() == [57344.0, -57344.0, 57344.0, -57344.0, 57344.0, 57344.0, 57344.0]
    assert math.isnan(E5.e5m2_quantize(np.array([np.nan]))[0])
    assert int(E5.e5m2_encode(np.array([np.nan]))[0]) == 0x7F
    # 1.125 lies halfway between 1.0 (code 0x3C, even) and 1.25 (0x3D): to 1.0;
    # 1.375 halfway between 1.25 (odd) and 1.5 (0x3E, even): to 1.5
    assert E5.e5m2_quantize(np.array([1.125, 1.375, -1.125])).tolist() == [1.0, 1.5, -1.0]
    # half the smallest subnormal rounds to zero (even), just above it to 2^-16
    assert E5.e5m2_quantize(np.array([2.0 ** -17, 2.0 ** -17 * 1.001])).tolist() == [0.0, 2.0 ** -16]
    assert np.signbit(E5.e5m2_quantize(np.array([-1e-30]))[0])


def test_e5m2_matches_torch_float8_e5m2_cast_on_float32_inputs():
    x = torch.randn(20000, dtype=torch.float32) * torch.exp2(torch.randint(-20, 18, (20000,)).float())
    ref = x.clamp(-57344, 57344).to(torch.float8_e5m2).double().numpy()
    np.testing.assert_array_equal(E5.e5m2_quantize(x.double().numpy()), ref)


# ----------------------------------------------------------------------------- FP8 linear backward
def _grid_values(shape, lo, hi):
    return np.vectorize(E4.e4m3_decode)(RNG.integers(lo, hi, size=shape)) * RNG.choice([-1.0, 1.0], size=shape)


@pytest.mark.parametrize("recipe,wgrad", list(itertools.product(F.RECIPES, (True, False))))
def test_fp8_backward_is_the_exact_backward_on_representable_operands(recipe, wgrad):
    # codes 0x30..0x47 are the E4M3 values in [0.5, 3.75]; dy takes those whose lowest mantissa
    # bit is clear, which E5M2 holds too, so that both gradient formats represent it exactly
    common = [c for c in range(0x30, 0x48) if E4.e4m3_decode(c) in set(E5M2_VALUES.tolist())]
    dy = np.vectorize(E4.e4m3_decode)(RNG.choice(common, size=(2, 5, 3))) * RNG.choice([-1, 1], (2, 5, 3))
    x = _grid_values((2, 5, 4), 0x30, 0x48)
    w = _grid_values((3, 4), 0x30, 0x48)
    dx, dw, db = F.fp8_linear_bwd(dy, x, w, 1.0, 1.0, 1.0, recipe, wgrad)
    ex, ew, eb = BW.linear_bwd(dy, x, w)
    np.testing.assert_array_equal(dx, ex)
    np.testing.assert_array_equal(dw, ew)
    np.testing.assert_array_equal(db, eb)


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_fp8_dgrad_with_identity_weight_lands_on_the_gradient_grid(recipe):
    dy = RNG.standard_normal((7, 6))
    s_dy = F.gradient_scale(np.abs(dy).max(), recipe)
    dx, _, _ = F.fp8_linear_bwd(dy, np.zeros((7, 6)), np.eye(6), 1.0, 1.0, s_dy, recipe)
    scaled = dx * s_dy
    grid = E5M2_VALUES if recipe == "hybrid" else E4M3_GRID
    assert _on_grid(scaled, grid).all()
    fmax = 57344.0 if recipe == "hybrid" else 448.0
    assert np.abs(scaled).max() == fmax
    if recipe == "hybrid":
        assert not _on_grid(scaled, E4M3_GRID).all()


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_fp8_wgrad_with_identity_input(recipe):
    dy = RNG.standard_normal((5, 3))
    s_dy = F.gradient_scale(np.abs(dy).max(), recipe)
    w = RNG.standard_normal((3, 5))
    _, dw, _ = F.fp8_linear_bwd(dy, np.eye(5), w, 1.0, 1.0, s_dy, recipe, wgrad=True)
    grid = E5M2_VALUES if recipe == "hybrid" else E4M3_GRID
    assert _on_grid(dw * s_dy, grid).all()
    q = E5.e5m2_quantize if recipe == "hybrid" else E4.e4m3_quantize
    np.testing.assert_array_equal(dw, q(dy.T * s_dy) / s_dy)
    _, dw_hi, _ = F.fp8_linear_bwd(dy, np.eye(5), w, 1.0, 1.0, s_dy, recipe, wgrad=False)
    np.testing.assert_array_equal(dw_hi, dy.T)


def _nearest(v, values):
    """Brute force: the finite value nearest to v, ties to the even code, saturating."""
    best = None
    for c, val in enumerate(values):
        if not math.isfinite(val):
            continue
        d = abs(val - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c, val)
    return best[2]


def test_fp8_backward_brute_force_tiny():
    e4 = [E4.e4m3_decode(c) for c in range(256)]
    e5 = [E5.e5m2_decode(c) for c in range(256)]
    dy = RNG.standard_normal((2, 3))
    x = RNG.standard_normal((2, 4))
    w = RNG.standard_normal((3, 4))
    s_x, s_w, s_dy = 100.0, 70.0, 9000.0
    for recipe, gvals in (("e4m3", e4), ("hybrid", e5)):
        dx, dw, db = F.fp8_linear_bwd(dy, x, w, s_x, s_w, s_dy, recipe)
        for i in range(2):
            for k in range(4):
                acc = 0.0
                for n in range(3):
                    acc += _nearest(dy[i, n] * s_dy, gvals) * _nearest(w[n, k] * s_w, e4)
                assert dx[i, k] == pytest.approx(acc / (s_dy * s_w), rel=1e-14, abs=1e-300)
        for n in range(3):
            for k in range(4):
                acc = 0.0
                for i in range(2):
                    acc += _nearest(dy[i, n] * s_dy, gvals) * _nearest(x[i, k] * s_x, e4)
                assert dw[n, k] == pytest.approx(acc / (s_dy * s_x), rel=1e-14, abs=1e-300)
            assert db[n] == pytest.approx(dy[0, n] + dy[1, n], rel=1e-15)


@pytest.mark.parametrize("recipe", F.RECIPES)
def test_fp8_backward_within_the_formats_rounding_bound(recipe):
    # magnitudes in [amax/16, amax] keep every scaled value normal in both formats, where the
    # relative rounding error is at most 2^-4 (E4M3) or 2^-3 (E5M2)
    def draw(shape):
        return RNG.uniform(1.0 / 16, 1.0, shape) * RNG.choice([-1.0, 1.0], shape)
    dy, x, w = draw((16, 12)), draw((16, 20)), draw((12, 20))
    s = {k: 448.0 / np.abs(v).max() for k, v in (("x", x), ("w", w))}
    s_dy = F.gradient_scale(np.abs(dy).max(), recipe)
    u_g = 2.0 ** -3 if recipe == "hybrid" else 2.0 ** -4
    u_4 = 2.0 ** -4
    dx, dw, _ = F.fp8_linear_bwd(dy, x, w, s["x"], s["w"], s_dy, recipe)
    ex, ew, _ = BW.linear_bwd(dy, x, w)
    rel = u_g + u_4 + u_g * u_4
    assert np.all(np.abs(dx - ex) <= rel * (np.abs(dy) @ np.abs(w)) * (1 + 1e-12))
    assert np.all(np.abs(dw - ew) <= rel * (np.abs(dy).T @ np.abs(x)) * (1 + 1e-12))
    assert np.abs(dx - ex).max() > 0 and np.abs(dw - ew).max() > 0


def test_delayed_scaling_training_records_and_scales_gradients():
    dy = RNG.standard_normal((4, 3)) * 5.0
    x = RNG.standard_normal((4, 6))
    w = RNG.standard_normal((3, 6))
    for recipe, fmax in (("e4m3", 448.0), ("hybrid", 57344.0)):
        ctx = F.DelayedScalingTraining(recipe=recipe)
        ctx.linear("fc", x, w, None)
        ctx.linear_bwd("fc", dy, x, w)
        nxt = ctx.next_scales()
        assert nxt["fc.dy"] == fmax / np.abs(dy).max()
        assert nxt["fc.x"] == 448.0 / np.abs(x).max() and nxt["fc.w"] == 448.0 / np.abs(w).max()
        assert ctx.next_scales(margin=2)["fc.dy"] == fmax / np.abs(dy).max() / 4.0
        # the next call quantises the gradient's largest element to the format's largest value
        q = (E5.e5m2_quantize if recipe == "hybrid" else E4.e4m3_quantize)(dy * nxt["fc.dy"])
        assert np.abs(q).max() == fmax
        ctx2 = F.DelayedScalingTraining(nxt, recipe=recipe)
        dx, dw, _ = ctx2.linear_bwd("fc", dy, x, w)
        want = F.fp8_linear_bwd(dy, x, w, nxt["fc.x"], nxt["fc.w"], nxt["fc.dy"], recipe)
        np.testing.assert_array_equal(dx, want[0])
        np.testing.assert_array_equal(dw, want[1])


def test_zero_gradient_and_unknown_recipe():
    assert F.gradient_scale(0.0, "hybrid") == 1.0 and F.gradient_scale(None) == 1.0
    dx, dw, db = F.fp8_linear_bwd(np.zeros((3, 2)), np.ones((3, 4)), np.ones((2, 4)), 1.0, 1.0, 1.0, "hybrid")
    assert not dx.any() and not dw.any() and not db.any()
    with pytest.raises(ValueError):
        F.DelayedScalingTraining(recipe="e5m2")
