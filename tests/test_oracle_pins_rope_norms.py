"""Pins of the fp64 oracle's RoPE, norms, activations and modulation (CPU only).

Each check ties the oracle to something other than itself: values derived by
hand from the pages' formulas (tests/golden/), textbook constants, library
routines (torch fp64 on CPU, scipy), or invariants that a dropped term, wrong
sign, wrong index or transposed operand would break.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import flux as O

RNG = np.random.default_rng(7)


# ----------------------------------------------------------------------------- RoPE
def test_rope_golden_angles(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "rope_frequencies.json")))
    for case in g["cases"]:
        ang = O.rope_angles(np.array(case["ids"], float), tuple(g["axes_dim"]), g["theta"])
        assert ang.shape == (64,)
        assert ang[case["index"]] == pytest.approx(case["angle"], rel=1e-12, abs=1e-15), case


def test_rope_identity_at_origin():
    # P1: id (0,0,0) gives cos 1, sin 0 for every pair, so the rotation is the identity.
    c, s = O.rope_cos_sin(np.zeros((5, 3)))
    assert np.all(c == 1.0) and np.all(s == 0.0)
    x = RNG.standard_normal((5, 128))
    for inter in (True, False):
        np.testing.assert_array_equal(O.apply_rope(x, c, s, inter), x)


def test_rope_preserves_pair_and_vector_norms():
    # P2
    ids = RNG.integers(0, 200, size=(7, 3)).astype(float)
    c, s = O.rope_cos_sin(ids)
    x = RNG.standard_normal((7, 128))
    for inter in (True, False):
        y = O.apply_rope(x, c, s, inter)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
        if inter:
            px, py = x[:, 0::2] ** 2 + x[:, 1::2] ** 2, y[:, 0::2] ** 2 + y[:, 1::2] ** 2
        else:
            px, py = x[:, :64] ** 2 + x[:, 64:] ** 2, y[:, :64] ** 2 + y[:, 64:] ** 2
        np.testing.assert_allclose(py, px, rtol=1e-12)


def test_rope_pair_is_a_rotation_by_the_angle():
    # A pair (1, 0) rotated by angle a lands on (cos a, sin a): fixes the sign convention.
    ids = np.array([[0.0, 3.0, 11.0]])
    ang = O.rope_angles(ids)
    c, s = np.cos(ang), np.sin(ang)
    x = np.zeros((1, 128))
    x[0, 2 * 20] = 1.0  # interleaved pair 20, first element
    y = O.apply_rope(x, c, s, True)
    assert y[0, 40] == pytest.approx(math.cos(ang[0, 20]), abs=1e-15)
    assert y[0, 41] == pytest.approx(math.sin(ang[0, 20]), abs=1e-15)
    assert np.count_nonzero(y) == 2
    x = np.zeros((1, 128))
    x[0, 20] = 1.0  # half-split pair 20
    y = O.apply_rope(x, c, s, False)
    assert y[0, 20] == pytest.approx(math.cos(ang[0, 20]), abs=1e-15)
    assert y[0, 84] == pytest.approx(math.sin(ang[0, 20]), abs=1e-15)


def test_rope_interleaved_and_half_split_agree_up_to_permutation():
    ids = RNG.integers(0, 50, size=(4, 3)).astype(float)
    c, s = O.rope_cos_sin(ids)
    x = RNG.standard_normal((4, 128))
    perm = np.concatenate([np.arange(0, 128, 2), np.arange(1, 128, 2)])  # interleaved -> half-split
    y_int = O.apply_rope(x, c, s, True)
    y_half = O.apply_rope(x[:, perm], c, s, False)
    np.testing.assert_allclose(y_half, y_int[:, perm], rtol=0, atol=1e-14)


def test_rope_relative_position_invariance_of_scores():
    # P3 at the score level: <R(m) q, R(n) k> depends only on m - n, per axis.
    q = RNG.standard_normal(128)
    k = RNG.standard_normal(128)
    for axis in range(3):
        base = np.array([[2.0, 5.0, 9.0], [4.0, 1.0, 3.0]])
        shift = np.zeros(3)
        shift[axis] = 37.0
        vals = []
        for ids in (base, base + shift):
            c, s = O.rope_cos_sin(ids)
            rq = O.apply_rope(q[None], c[:1], s[:1])[0]
            rk = O.apply_rope(k[None], c[1:], s[1:])[0]
            vals.append(rq @ rk)
        assert vals[0] == pytest.approx(vals[1], rel=1e-10, abs=1e-10)


# ----------------------------------------------------------------------------- norms / activations
def test_layernorm_matches_torch_and_moments():
    x = RNG.standard_normal((3, 5, 64)) * 3 + 1.5
    y = O.layernorm(x, 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (64,), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # P6: zero mean, variance var/(var+eps)
    var = x.var(axis=-1)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-13)
    np.testing.assert_allclose(y.var(-1), var / (var + 1e-6), rtol=1e-12)


def test_rmsnorm_matches_torch():
    x = RNG.standard_normal((4, 128))
    g = 1 + 0.1 * RNG.standard_normal(128)
    y = O.rmsnorm(x, g, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    # unit gain -> RMS close to 1
    y1 = O.rmsnorm(x, np.ones(128))
    np.testing.assert_allclose(np.sqrt((y1 ** 2).mean(-1)), 1, rtol=1e-5)


def test_gelu_textbook_values_and_torch(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "normal_cdf_values.json")))
    for c in g["cases"]:
        assert O.gelu(np.array(c["x"])) == pytest.approx(c["x"] * c["phi"], rel=1e-13)
    x = np.linspace(-8, 8, 1001)
    np.testing.assert_allclose(O.gelu(x), torch.nn.functional.gelu(torch.from_numpy(x)).numpy(),
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(
        O.gelu(x, tanh=True),
        torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy(), rtol=1e-13, atol=1e-15)
    assert O.gelu(np.array(0.0)) == 0.0
    # the two GELU forms differ by well under the block tolerance
    assert np.abs(O.gelu(x) - O.gelu(x, True)).max() < 1e-3


def test_silu_matches_torch():
    x = np.linspace(-20, 20, 801)
    np.testing.assert_allclose(O.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-13, atol=1e-16)
    assert O.silu(np.array(0.0)) == 0.0
    assert O.silu(np.array(1.0)) == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)


def test_linear_orientation_matches_torch():
    x = RNG.standard_normal((2, 3, 6))
    w = RNG.standard_normal((5, 6))
    b = RNG.standard_normal(5)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(O.linear(x, w, b), ref, rtol=1e-13)


# ----------------------------------------------------------------------------- modulation
def test_modulation_chunk_order():
    # The API page lists the six AdaLN outputs as
    # shift, scale, gate, shift_mlp, scale_mlp, gate_mlp: chunk j <- bias block j.
    D = 8
    w = np.zeros((6 * D, D))
    b = np.repeat(np.arange(1.0, 7.0), D)
    vec = RNG.standard_normal((2, D))
    chunks = O.modulation(vec, w, b)
    assert len(chunks) == 6
    for j, c in enumerate(chunks):
        np.testing.assert_array_equal(c, np.full((2, D), j + 1.0))


def test_modulation_applies_silu_before_linear():
    D = 4
    vec = np.array([[1.0, -2.0, 0.5, 3.0]])
    w = np.zeros((6 * D, D))
    w[0, 1] = 1.0  # shift[0] reads vec[1] through SiLU
    shift = O.modulation(vec, w, np.zeros(6 * D))[0]
    assert shift[0, 0] == pytest.approx(-2.0 / (1 + math.exp(2.0)), rel=1e-14)


def test_modulate_uses_one_plus_scale():
    # scale = -1 and shift = c turn the modulated LayerNorm into the constant c
    x = RNG.standard_normal((2, 5, 16))
    c = RNG.standard_normal((2, 16))
    y = O.modulate(x, c, -np.ones((2, 16)))
    np.testing.assert_allclose(y, np.broadcast_to(c[:, None, :], y.shape), atol=1e-15)
    # scale = 0 and shift = 0 give the plain LayerNorm
    np.testing.assert_allclose(O.modulate(x, 0 * c, 0 * c), O.layernorm(x), atol=0)
