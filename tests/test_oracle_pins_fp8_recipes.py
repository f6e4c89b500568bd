"""Pins of the fp64 oracle's other FP8 scaling recipes: tensorwise, blockwise, MXFP8 (CPU only).

What fixes them from outside the oracle: E8M0 codes against torch's ``float8_e8m0fnu``; the MX
shared exponent at hand-derived amax values; exact casts of values on the block grids;
brute force (the nearest value of the scaled E4M3 grid by search) on small tensors; the E4M3
rounding bound; the tile shapes through which tiles an outlier can reach; independent scalar
loops for the block-summed GEMMs; and the special cases where a recipe reduces to another.
"""
import math

import numpy as np
import pytest
import torch

from oracle import e4m3 as E4
from oracle import fp8_recipes as R

RNG = np.random.default_rng(31)


def _nearest_even(v, grid_codes, grid_vals):
    """Brute force: the grid value nearest to v, ties to the even code, saturating at the ends."""
    d = np.abs(grid_vals - v)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        best = [i for i in best if grid_codes[i] % 2 == 0]
    return grid_vals[best[0]]


_POS_CODES = np.arange(0x7F)
_POS_VALS = np.array([E4.e4m3_decode(c) for c in _POS_CODES])


def _brute_e4m3(v):
    """E4M3 rounding of one value by search over the positive codes, sign applied after."""
    a = min(abs(v), 448.0)
    return math.copysign(_nearest_even(a, _POS_CODES, _POS_VALS), v)


# ----------------------------------------------------------------------------- MX: E8M0 scale
def test_e8m0_codes_match_torch_float8_e8m0fnu_on_powers_of_two():
    for k in range(-127, 128):
        code = int(torch.tensor([2.0 ** k], dtype=torch.float64).to(torch.float32)
                   .to(torch.float8_e8m0fnu).view(torch.uint8)[0])
        assert code == k + 127
        assert R.e8m0_decode(code) == 2.0 ** k
    assert math.isnan(R.e8m0_decode(0xFF))


def test_mx_shared_exponent_hand_derived_values():
    # 448 = 1.75 * 2^8 -> floor(log2) = 8 -> exponent 0 (X = 1); 1 -> -8; 0.75 -> -9;
    # just below 2 -> -8 (a log2 that rounded up would give -7); 2^130 -> 122; tiny and zero -> -127
    amax = [448.0, 1.0, 0.75, np.nextafter(2.0, 0.0), 2.0, 2.0 ** 130, 2.0 ** 140, 2.0 ** -140, 0.0]
    want = [0, -8, -9, -8, -7, 122, 127, -127, -127]
    np.testing.assert_array_equal(R.mx_shared_exponent(amax), want)


def test_mx_block_max_lands_in_the_top_binade():
    # after dividing by X the block maximum lies in [256, 512): the scale puts it at E4M3's top
    # exponent, and everything up to 448 of it is kept
    x = RNG.standard_normal((16, 96)) * np.exp(RNG.uniform(-20, 20, (16, 1)))
    _, e = R.mxfp8_quantize(x)
    for j in range(3):
        m = np.abs(x[:, 32 * j:32 * (j + 1)]).max(axis=1)
        r = np.ldexp(m, -e[:, j])
        assert np.all((r >= 256.0) & (r < 512.0))


# ----------------------------------------------------------------------------- MX: elements
def test_mx_exact_on_powers_of_two_within_the_block_range():
    # a block whose values are +-2^k with k in [m - 17, m] (m the block's top exponent) is exact:
    # V / X = 2^(k - m + 8) with k - m + 8 in [-9, 8], all E4M3 values (2^-9 the smallest subnormal)
    m = 5
    k = RNG.integers(m - 17, m + 1, (4, 32))
    k[:, 0] = m
    x = np.ldexp(1.0, k) * RNG.choice([-1.0, 1.0], (4, 32))
    p, e = R.mxfp8_quantize(x)
    np.testing.assert_array_equal(e, np.full((4, 1), m - 8))
    np.testing.assert_array_equal(R.mxfp8_dequantize(p, e), x)


def test_mx_saturates_quotients_above_448():
    # block max 1.9 * 2^m: V / X = 1.9 * 256 = 486.4 > 448 -> 448, i.e. 1.75 * 2^m
    x = np.zeros((1, 32))
    x[0, 3] = 1.9 * 2.0 ** 3
    x[0, 7] = -1.99 * 2.0 ** 3
    x[0, 9] = 1.5 * 2.0 ** 3
    p, e = R.mxfp8_quantize(x)
    d = R.mxfp8_dequantize(p, e)
    assert e[0, 0] == 3 - 8
    assert d[0, 3] == 1.75 * 8 and d[0, 7] == -1.75 * 8 and d[0, 9] == 1.5 * 8


def test_mx_zero_block_and_ragged_tail():
    x = np.zeros((2, 70))
    x[1, 65] = 3.0                                   # in the 6-wide last block
    p, e = R.mxfp8_quantize(x)
    assert e.shape == (2, 3)
    np.testing.assert_array_equal(e[0], [-127, -127, -127])
    np.testing.assert_array_equal(e[1], [-127, -127, 1 - 8])
    np.testing.assert_array_equal(R.mxfp8_dequantize(p, e), x)


def test_mx_brute_force_tiny():
    x = RNG.standard_normal((3, 40)) * np.array([[1.0], [1e-3], [300.0]])
    x[0, 5] = 0.0
    p, e = R.mxfp8_quantize(x)
    for r in range(3):
        for c in range(40):
            j = c // 32
            amax = np.abs(x[r, 32 * j:min(32 * j + 32, 40)]).max()
            ej = math.floor(math.log2(amax)) - 8 if amax > 0 else -127
            assert e[r, j] == ej
            want = _brute_e4m3(x[r, c] / 2.0 ** ej)
            assert p[r, c] == want, (r, c)


def test_mx_blocks_are_independent():
    x = RNG.standard_normal((4, 96))
    p0, e0 = R.mxfp8_quantize(x)
    y = x.copy()
    y[:, 40] *= 1e4                                  # an outlier in block 1 only
    p1, e1 = R.mxfp8_quantize(y)
    np.testing.assert_array_equal(p0[:, :32], p1[:, :32])
    np.testing.assert_array_equal(p0[:, 64:], p1[:, 64:])
    np.testing.assert_array_equal(e0[:, [0, 2]], e1[:, [0, 2]])
    assert np.all(e1[:, 1] > e0[:, 1])


def test_mx_rounding_bound():
    # elements whose quotient is an E4M3 normal (>= 2^-6) and not saturated are within half an ulp:
    # |Q - V| <= 2^-4 |V|
    x = RNG.standard_normal((64, 256)) * np.exp(RNG.uniform(-8, 8, (64, 256)))
    p, e = R.mxfp8_quantize(x)
    d = R.mxfp8_dequantize(p, e)
    q = np.ldexp(np.abs(x), -np.repeat(e, 32, axis=1))
    ok = (q >= 2.0 ** -6) & (q <= 448.0)
    assert ok.sum() > 0.5 * x.size
    assert np.all(np.abs(d - x)[ok] <= 2.0 ** -4 * np.abs(x)[ok])


def test_mx_linear_scalar_loop_and_exact_case():
    x = RNG.standard_normal((3, 72))
    w = RNG.standard_normal((5, 72)) * 0.02
    b = RNG.standard_normal(5)
    y = R.mxfp8_linear(x, w, b)
    px, ex = R.mxfp8_quantize(x)
    pw, ew = R.mxfp8_quantize(w)
    for i in range(3):
        for n in range(5):
            acc = 0.0
            for c in range(72):
                acc += px[i, c] * 2.0 ** ex[i, c // 32] * pw[n, c] * 2.0 ** ew[n, c // 32]
            assert abs(y[i, n] - (acc + b[n])) <= 1e-12 * (abs(acc) + abs(b[n]))
    # operands on their block grids: the linear is the exact product
    xe = R.mxfp8_dequantize(px, ex)
    we = R.mxfp8_dequantize(pw, ew)
    np.testing.assert_allclose(R.mxfp8_linear(xe, we, None), xe @ we.T, rtol=1e-13, atol=0)


# ----------------------------------------------------------------------------- tensorwise
def test_tensorwise_amax_element_lands_on_448():
    x = RNG.standard_normal((7, 33)) * 3.7
    s = R.tensorwise_scale(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(x[i] * s) == 448.0
    assert E4.e4m3_quantize(x * s).max() <= 448.0
    assert R.tensorwise_scale(np.zeros(4)) == 1.0
    assert R.tensorwise_scale(x, margin=2) == s / 4.0


def test_tensorwise_is_invariant_to_power_of_two_rescaling():
    # the scale follows the tensor, so 2^k x casts to the same codes and the product scales by 2^k;
    # delayed scaling with a fixed scale does not (it saturates or loses the small values)
    x = RNG.standard_normal((4, 64))
    w = RNG.standard_normal((8, 64)) * 0.02
    y = R.tensorwise_linear(x, w, None)
    for k in (-20, -3, 5, 30):
        np.testing.assert_array_equal(R.tensorwise_linear(np.ldexp(x, k), w, None), np.ldexp(y, k))
    s = R.tensorwise_scale(x)
    fixed = E4.fp8_linear(np.ldexp(x, 5), w, None, s, R.tensorwise_scale(w))
    assert not np.array_equal(fixed, np.ldexp(y, 5))


def test_tensorwise_equals_delayed_scaling_at_the_current_amax():
    x = RNG.standard_normal((6, 48))
    w = RNG.standard_normal((10, 48)) * 0.02
    b = RNG.standard_normal(10)
    ds = E4.DelayedScaling()
    ds.linear("l", x, w, b)
    sc = ds.next_scales()
    np.testing.assert_array_equal(R.tensorwise_linear(x, w, b),
                                  E4.fp8_linear(x, w, b, sc["l.x"], sc["l.w"]))


# ----------------------------------------------------------------------------- blockwise
def test_blockwise_tile_shapes_and_each_tile_max_at_448():
    x = RNG.standard_normal((2, 3, 300))
    w = RNG.standard_normal((260, 300))
    qx, sx = R.blockwise_quantize_act(x)
    qw, sw = R.blockwise_quantize_weight(w)
    assert sx.shape == (2, 3, 3) and sw.shape == (3, 3)
    for j, (lo, hi) in enumerate(((0, 128), (128, 256), (256, 300))):
        np.testing.assert_array_equal(np.abs(qx[..., lo:hi]).max(axis=-1), 448.0)
        for i, (rlo, rhi) in enumerate(((0, 128), (128, 256), (256, 260))):
            assert np.abs(qw[rlo:rhi, lo:hi]).max() == 448.0
            assert sw[i, j] == 448.0 / np.abs(w[rlo:rhi, lo:hi]).max()


def test_blockwise_outlier_reaches_only_its_own_tile():
    # an activation outlier changes the casts of its own 1 x 128 tile only (same row, same K
    # slice); a weight outlier changes its own 128 x 128 tile only
    x = RNG.standard_normal((4, 256))
    w = RNG.standard_normal((256, 256))
    qx0, _ = R.blockwise_quantize_act(x)
    qw0, _ = R.blockwise_quantize_weight(w)
    x2 = x.copy()
    x2[1, 10] = 1e5
    qx1, _ = R.blockwise_quantize_act(x2)
    changed = np.argwhere(qx1 != qx0)
    assert len(changed) > 64 and np.all(changed[:, 0] == 1) and np.all(changed[:, 1] < 128)
    w2 = w.copy()
    w2[200, 130] = 1e5
    qw1, _ = R.blockwise_quantize_weight(w2)
    changed = np.argwhere(qw1 != qw0)
    assert len(changed) > 128 * 64 and np.all(changed >= 128)
    # both rows 128..255 and columns 128..255 of the tile are reached, not one row or one column
    assert len(set(changed[:, 0])) > 100 and len(set(changed[:, 1])) > 100


def test_blockwise_linear_scalar_loop_ragged():
    x = RNG.standard_normal((3, 200))
    w = RNG.standard_normal((130, 200)) * 0.02
    b = RNG.standard_normal(130)
    y = R.blockwise_linear(x, w, b)
    qx, sx = R.blockwise_quantize_act(x)
    qw, sw = R.blockwise_quantize_weight(w)
    for i in range(3):
        for n in (0, 1, 127, 128, 129):
            acc = 0.0
            for c in range(200):
                acc += qx[i, c] / sx[i, c // 128] * qw[n, c] / sw[n // 128, c // 128]
            assert abs(y[i, n] - (acc + b[n])) <= 1e-12 * (abs(acc) + abs(b[n])), (i, n)


def test_blockwise_with_one_tile_is_tensorwise():
    # one row of at most 128 elements and a weight of at most 128 x 128: each operand is one tile
    x = RNG.standard_normal((1, 96))
    w = RNG.standard_normal((40, 96)) * 0.02
    b = RNG.standard_normal(40)
    np.testing.assert_array_equal(R.blockwise_linear(x, w, b), R.tensorwise_linear(x, w, b))


def test_tensorwise_and_blockwise_casts_within_the_e4m3_rounding_bound():
    # a cast element is within half an E4M3 ulp of its scaled value: 2^-4 of it for normals, half
    # the subnormal step 2^-10 below them; divided by the scale s of the tensor or tile it is in
    x = RNG.standard_normal((16, 300)) * np.exp(RNG.uniform(-6, 6, (16, 300)))
    s = R.tensorwise_scale(x)
    err = np.abs(E4.e4m3_quantize(x * s) / s - x)
    assert np.all(err <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 / s)
    qx, sx = R.blockwise_quantize_act(x)
    sfull = np.repeat(sx, 128, axis=1)[:, :300]
    err = np.abs(qx / sfull - x)
    assert np.all(err <= 2.0 ** -4 * np.abs(x) + 2.0 ** -10 / sfull)
    # the per-tile scales lose less to the subnormal floor than the per-tensor scale: over the
    # whole tensor, the blockwise error is no larger
    assert np.abs(qx / sfull - x).sum() <= np.abs(E4.e4m3_quantize(x * s) / s - x).sum()


@pytest.mark.parametrize("f", [R.tensorwise_linear, R.blockwise_linear, R.mxfp8_linear])
def test_recipes_zero_operand(f):
    x = np.zeros((2, 64))
    w = RNG.standard_normal((3, 64))
    b = RNG.standard_normal(3)
    np.testing.assert_array_equal(f(x, w, b), np.broadcast_to(b, (2, 3)))


def test_tensorwise_recipe_object_in_a_block_is_the_tensorwise_linear():
    """The block oracle's tensorwise object: each linear equals tensorwise_linear of its
    (optionally bf16-stored) input, records 448 / amax per tensor, and a whole double block run
    with it differs from the delayed recipe at the scales those amax give only through the
    delayed recipe's use of the previous call's scales (equal here: same inputs twice)."""
    from oracle import flux as O
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 7, 64)) * 3.0
    w = rng.standard_normal((96, 64)) * 0.05
    b = rng.standard_normal(96) * 0.01
    tw = R.TensorwiseScaling()
    assert np.array_equal(tw.linear("fc1", x, w, b), R.tensorwise_linear(x, w, b))
    assert tw.scales["fc1.x"] == 448.0 / np.abs(x).max() and tw.scales["fc1.w"] == 448.0 / np.abs(w).max()
    tb = R.TensorwiseScaling(act_cast=O.round_bf16)
    assert np.array_equal(tb.linear("fc1", x, w, b), R.tensorwise_linear(O.round_bf16(x), w, b))
    # a whole block: tensorwise == delayed scaling handed the tensorwise scales of the same inputs
    from diffusion_transformer_flux_gb300 import synth
    inp = synth.block_inputs(1, 16, 5, 256, "f32", 3, (4, 4))
    wi = synth.stream_weights(rng, 256, 2, 128, 512, "f32", 0.05)
    wt = synth.stream_weights(rng, 256, 2, 128, 512, "f32", 0.05)
    c, s = O.rope_cos_sin(inp.ids)
    t1 = R.TensorwiseScaling()
    y_tw = O.double_block(inp.x_img, inp.x_txt, inp.vec, c, s, wi, wt, 2, fp8=t1)
    y_dl = O.double_block(inp.x_img, inp.x_txt, inp.vec, c, s, wi, wt, 2,
                          fp8=E4.DelayedScaling(dict(t1.scales)))
    for a, bb in zip(y_tw, y_dl):
        assert np.array_equal(a, bb)


def test_blockwise_scaling_object_is_the_recipe_on_the_stored_input():
    # the block oracle's fp8 object: blockwise_linear of the act_cast input, and exact wherever
    # every tile is already on the E4M3 grid with its maximum at 448 (every scale 1, no rounding)
    from oracle import flux as O
    x = RNG.standard_normal((2, 5, 256))
    w = RNG.standard_normal((256, 256)) * 0.02
    b = RNG.standard_normal(256)
    bw = R.BlockwiseScaling(act_cast=O.round_bf16)
    np.testing.assert_array_equal(bw.linear("qkv", x, w, b), R.blockwise_linear(O.round_bf16(x), w, b))
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 448.0])
    xg = RNG.choice(grid, size=(3, 256)) * RNG.choice([-1.0, 1.0], size=(3, 256))
    xg[:, 0] = 448.0
    xg[:, 128] = 448.0
    wg = RNG.choice(grid, size=(128, 256))
    wg[0, 0] = 448.0
    wg[0, 128] = 448.0
    np.testing.assert_array_equal(R.BlockwiseScaling().linear("o", xg, wg, None), xg @ wg.T)


def test_mx_scaling_object_is_the_recipe_on_the_stored_input():
    # the block oracle's fp8 object: mxfp8_linear of the act_cast input, and exact wherever every
    # 32-element block already holds E4M3 values whose maximum lies in [256, 448] (shared
    # exponent 0: nothing is rescaled or rounded)
    from oracle import flux as O
    x = RNG.standard_normal((2, 5, 128))
    w = RNG.standard_normal((64, 128)) * 0.02
    b = RNG.standard_normal(64)
    mx = R.MxScaling(act_cast=O.round_bf16)
    np.testing.assert_array_equal(mx.linear("qkv", x, w, b), R.mxfp8_linear(O.round_bf16(x), w, b))
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 448.0])
    xg = RNG.choice(grid, size=(3, 128)) * RNG.choice([-1.0, 1.0], size=(3, 128))
    xg[:, ::32] = 448.0
    wg = RNG.choice(grid, size=(64, 128))
    wg[:, ::32] = 256.0
    np.testing.assert_array_equal(R.MxScaling().linear("o", xg, wg, None), xg @ wg.T)
