"""Pins of the oracle's bf16-autocast precision mode (CPU only).

``round_bf16`` is checked against torch's bfloat16 conversion (a library routine) and the
format's special cases; the ``mm_cast`` mode is checked to leave grid-aligned operands exact,
to reduce to closed forms where the rounded probabilities are exact, and to stay within
bf16-level distance of the exact fp64 block.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

RNG = np.random.default_rng(21)


def test_round_bf16_matches_torch_on_float32_inputs():
    x = np.concatenate([RNG.standard_normal(200000) * 10.0 ** RNG.integers(-30, 30, 200000),
                        np.linspace(-3, 3, 100001)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_special_cases():
    # representable values are fixed points
    grid = np.array([1.0, -2.0, 1.0 + 2 ** -7, 3.0 * 2.0 ** -100, 0.0, 2.0 ** 127])
    np.testing.assert_array_equal(O.round_bf16(grid), grid)
    # midpoints round to the even significand: 1 + 2^-8 -> 1 (even), 1 + 3 * 2^-8 -> 1 + 2^-6
    np.testing.assert_array_equal(O.round_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8])),
                                  [1.0, 1 + 2 ** -6])
    # directly from float64: no double rounding through float32
    x = 1 + 2 ** -8 + 2 ** -40  # just above a midpoint; float32 would round it onto the midpoint
    assert O.round_bf16(np.array([x]))[0] == 1 + 2 ** -7
    # sign symmetry and the relative error bound 2^-8
    y = RNG.standard_normal(10000) * 1e3
    np.testing.assert_array_equal(O.round_bf16(-y), -O.round_bf16(y))
    assert np.all(np.abs(O.round_bf16(y) - y) <= 2.0 ** -8 * np.abs(y))


def test_cast_mode_is_exact_on_grid_operands():
    x = synth.bf16_round(RNG.standard_normal((5, 32)).astype(np.float32))
    w = synth.bf16_round(RNG.standard_normal((7, 32)).astype(np.float32))
    np.testing.assert_array_equal(O.linear(x, w, None, O.round_bf16), O.linear(x, w))


def test_cast_mode_attention_closed_forms():
    v = RNG.standard_normal((7, 16))
    k = RNG.standard_normal((7, 4))
    # q = 0: uniform weights (kept exact) -> mean of the rounded values, for any key count
    out = O.attention(np.zeros((2, 4)), k, v, O.round_bf16)
    np.testing.assert_allclose(out, np.repeat(O.round_bf16(v).mean(0, keepdims=True), 2, 0), rtol=1e-14)
    # a single key: weight 1 -> the rounded value exactly
    out = O.attention(RNG.standard_normal((3, 4)), k[:1], v[:1], O.round_bf16)
    np.testing.assert_array_equal(out, np.repeat(O.round_bf16(v[:1]), 3, 0))
    # the cast mode is the exact attention of the rounded inputs
    q = RNG.standard_normal((5, 4))
    np.testing.assert_allclose(O.attention(q, k, v, O.round_bf16),
                               O.attention(O.round_bf16(q), O.round_bf16(k), O.round_bf16(v)), rtol=1e-15)


def test_cast_mode_block_stays_close_to_exact_block():
    rng = np.random.default_rng(2)
    D, H, F = 256, 2, 512
    w = synth.stream_weights(rng, D, H, 128, F, "bf16", 0.05)
    x = synth.bf16_round(rng.standard_normal((1, 40, D)).astype(np.float32))
    vec = synth.bf16_round(rng.standard_normal((1, D)).astype(np.float32))
    ids = synth.position_ids(1, 5, 8, 0)
    c, s = O.rope_cos_sin(ids)
    y = O.single_block(x, vec, c, s, w, H)
    yc = O.single_block(x, vec, c, s, w, H, mm_cast=O.round_bf16)
    rel = np.abs(yc - y).max() / np.sqrt(np.mean(y ** 2))
    assert 1e-4 < rel < 3e-2  # bf16-level, not identical, not gross
    # zero gates: still the identity under the cast
    w0 = dict(w)
    w0["w_mod"] = w["w_mod"].copy()
    w0["b_mod"] = w["b_mod"].copy()
    for ch in (2, 5):
        w0["w_mod"][ch * D:(ch + 1) * D] = 0
        w0["b_mod"][ch * D:(ch + 1) * D] = 0
    np.testing.assert_array_equal(O.single_block(x, vec, c, s, w0, H, mm_cast=O.round_bf16), x)
