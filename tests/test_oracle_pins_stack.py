"""Pins of the oracle's conditioning path and whole-model forward (CPU only).

Architecture page, §Model components › 1. Input embeddings › Conditioning and §Data flow ›
Complete forward pass; API page, §Components API › Embeddings (TimeStepEmbedder, MLPEmbedder).
Each pin fixes a fact independently of the oracle's code:
* the sinusoidal features at points where they are textbook values of cos and sin (math
  module), the frequency ladder 10000^(-i/128) read off the small-angle limit, unit pairs;
* the embedder's layer order and its SiLU, against a closed form built from math.exp;
* the guidance term is affine in g;
* the stack's wiring: with every gate zero the blocks pass the residual stream through, so
  the prediction is the head applied to the embedded latents; with only the attention gates
  zero no image row can see the text, so the prediction ignores the text (this fails if the
  head reads the wrong rows or the concatenation order is wrong).
"""
import json
import math
import os

import numpy as np

from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

RNG = np.random.default_rng(31)
AX = (4, 6, 6)  # RoPE axes of the 16-wide heads below


def test_timestep_features_textbook_values():
    # dim 4: frequencies 10000^0 = 1 and 10000^(-1/2) = 0.01; t = 0.001 is tau = 1
    f = O.timestep_features(np.array([0.001]), dim=4)[0]
    exp = [math.cos(1.0), math.cos(0.01), math.sin(1.0), math.sin(0.01)]
    np.testing.assert_allclose(f, exp, rtol=0, atol=1e-15)
    f = O.timestep_features(np.array([0.0005]), dim=4)[0]
    exp = [math.cos(0.5), math.cos(0.005), math.sin(0.5), math.sin(0.005)]
    np.testing.assert_allclose(f, exp, rtol=0, atol=1e-15)


def test_timestep_features_at_zero_and_unit_pairs():
    f = O.timestep_features(np.array([0.0, 0.37, 1.0]))
    assert f.shape == (3, 256)
    np.testing.assert_array_equal(f[0], np.r_[np.ones(128), np.zeros(128)])
    np.testing.assert_allclose(f[:, :128] ** 2 + f[:, 128:] ** 2, 1.0, atol=1e-14)


def test_timestep_frequency_ladder():
    # sin(tau f_i) / tau -> f_i as tau -> 0: the frequencies are 10000^(-i/128)
    tau = 1e-7
    f = O.timestep_features(np.array([tau / 1000.0]))[0]
    got = f[128:] / tau
    exp = np.array([math.pow(10000.0, -i / 128.0) for i in range(128)])
    np.testing.assert_allclose(got, exp, rtol=1e-9)
    assert abs(got[64] - 0.01) < 1e-11


def test_mlp_embedder_closed_form():
    # w1 = 2I, b1 = 1, w2 = 3I, b2 = -1: out = 3 SiLU(2x + 1) - 1
    x = RNG.standard_normal((3, 4))
    eye = np.eye(4)
    got = O.mlp_embedder(x, 2 * eye, np.ones(4), 3 * eye, -np.ones(4))
    silu = np.vectorize(lambda v: v / (1.0 + math.exp(-v)))
    np.testing.assert_allclose(got, 3 * silu(2 * x + 1) - 1, rtol=1e-14, atol=1e-14)


def test_guidance_term_is_affine_in_g():
    w, b = RNG.standard_normal(6), RNG.standard_normal(6)
    np.testing.assert_array_equal(O.guidance_embed(np.array([0.0]), w, b)[0], b)
    g = np.array([1.0, 2.5])
    e = O.guidance_embed(g, w, b)
    np.testing.assert_allclose(e[1] - e[0], 1.5 * w, atol=1e-14)


def test_conditioning_vec_is_the_sum_of_its_terms():
    D = 8
    w = {"time_in": synth.mlp_embedder_weights(RNG, 256, D, "f32", 0.3),
         "vector_in": synth.mlp_embedder_weights(RNG, 12, D, "f32", 0.3),
         "guidance_in": (RNG.standard_normal(D), RNG.standard_normal(D))}
    t, y, g = np.array([0.2, 0.9]), RNG.standard_normal((2, 12)), np.array([3.5, 1.0])
    v = O.conditioning_vec(t, y, w, g)
    parts = (O.mlp_embedder(O.timestep_features(t), *w["time_in"])
             + O.mlp_embedder(y, *w["vector_in"]) + O.guidance_embed(g, *w["guidance_in"]))
    np.testing.assert_allclose(v, parts, atol=1e-14)
    # without the guidance term the vector differs by exactly that term
    np.testing.assert_allclose(v - O.conditioning_vec(t, y, w), O.guidance_embed(g, *w["guidance_in"]),
                               atol=1e-14)


def _stack(n_double=2, n_single=2, D=32, H=2, F=64, lat=4, S_t=5, B=2, txt_dim=16, vec_dim=12, seed=0,
           single_parallel=False):
    rng = np.random.default_rng(seed)
    w = synth.flux_weights(rng, D, H, F, n_double, n_single, txt_dim, vec_dim, dtype="f32", std=0.2,
                           single_parallel=single_parallel)
    z = rng.standard_normal((B, 64, lat, lat))
    txt = rng.standard_normal((B, S_t, txt_dim))
    t = rng.uniform(size=B)
    y = rng.standard_normal((B, vec_dim))
    ids = synth.position_ids(B, lat, lat, S_t)
    return w, z, txt, t, y, ids, H


def _zero_gates(ws, which=(2, 5)):
    D = ws["w_mod"].shape[1]
    ws = dict(ws)
    ws["w_mod"], ws["b_mod"] = ws["w_mod"].copy(), ws["b_mod"].copy()
    for c in which:
        ws["w_mod"][c * D:(c + 1) * D] = 0
        ws["b_mod"][c * D:(c + 1) * D] = 0
    return ws


def test_stack_with_zero_gates_is_the_head_of_the_embedded_latents():
    w, z, txt, t, y, ids, H = _stack()
    w["double"] = [(_zero_gates(a), _zero_gates(b)) for a, b in w["double"]]
    w["single"] = [_zero_gates(s) for s in w["single"]]
    pred = O.flux_forward(z, txt, t, y, ids, w, H, axes_dim=AX)
    vec = O.conditioning_vec(t, y, w)
    f = w["final"]
    exp = O.final_layer(O.img_in(z, *w["img_in"]), vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], 4, 4)
    np.testing.assert_allclose(pred, exp, atol=1e-13)
    # and the blocks do change it once the gates are back
    w2, *_ = _stack()
    assert np.abs(O.flux_forward(z, txt, t, y, ids, w2, H, axes_dim=AX) - exp).max() > 1e-3


def test_stack_without_attention_gates_ignores_the_text():
    w, z, txt, t, y, ids, H = _stack(seed=4)
    w["double"] = [(_zero_gates(a, (2,)), _zero_gates(b, (2,))) for a, b in w["double"]]
    w["single"] = [_zero_gates(s, (2,)) for s in w["single"]]
    pred = O.flux_forward(z, txt, t, y, ids, w, H, axes_dim=AX)
    other = np.random.default_rng(9).standard_normal(txt.shape)
    np.testing.assert_allclose(O.flux_forward(z, other, t, y, ids, w, H, axes_dim=AX), pred, atol=1e-13)
    # with the attention gates on, the text reaches the image rows
    w2, *_ = _stack(seed=4)
    a = O.flux_forward(z, txt, t, y, ids, w2, H, axes_dim=AX)
    assert np.abs(O.flux_forward(z, other, t, y, ids, w2, H, axes_dim=AX) - a).max() > 1e-4


def test_stack_with_no_blocks_and_identity_blocks_agree():
    w, z, txt, t, y, ids, H = _stack(n_double=1, n_single=1, seed=6)
    base = O.flux_forward(z, txt, t, y, ids, w, H, axes_dim=AX)
    # appending blocks whose gates are all zero changes nothing
    w2 = dict(w)
    w2["double"] = w["double"] + [tuple(_zero_gates(s) for s in w["double"][0])]
    w2["single"] = w["single"] + [_zero_gates(w["single"][0])]
    np.testing.assert_allclose(O.flux_forward(z, txt, t, y, ids, w2, H, axes_dim=AX), base, atol=1e-13)


def _tree_params(w):
    """Number of parameters in a weight tree (dicts, lists and tuples of arrays)."""
    if isinstance(w, dict):
        return sum(_tree_params(v) for v in w.values())
    if isinstance(w, (list, tuple)):
        return sum(_tree_params(v) for v in w)
    return int(np.size(w))


def _count(D, F, d, n_double, n_single, parallel, txt_dim=4096, vec_dim=768, time_dim=256, channels=64):
    """Parameters of the whole model from its weight shapes (the trees flux_weights draws)."""
    stream = 6 * D * D + 6 * D + 3 * D * D + 3 * D + 2 * d + D * D + D + F * D + F + D * F + D
    single = stream - 3 * D * D - 3 * D if parallel else stream   # three modulation chunks, not six
    emb = (channels * D + D) + (txt_dim * D + D) + (time_dim * D + D + D * D + D) \
        + (vec_dim * D + D + D * D + D) + (2 * D * D + 2 * D + channels * D + channels)
    return n_double * 2 * stream + n_single * single + emb


def test_parameter_counts_against_the_model_variants_table():
    # The API reference's parameter-count table prints ~535 million for 1 double + 1 single block
    # and ~12 billion for 19 + 38 (hidden 3072, MLP 12288).  The shape formula is first checked
    # against real weight trees at a small size, then evaluated at those sizes: the blocks as
    # built land within 0.5% and 1% of the printed counts with the parallel-branch single block, while
    # the sequential single block drawn in the single-block section gives 563.6 million and 12.97
    # billion (5% and 8% high).  The printed counts thus favour the parallel form.
    rng = np.random.default_rng(3)
    D, H, F = 64, 2, 256
    w = synth.flux_weights(rng, D, H, F, 2, 3, txt_dim=48, vec_dim=24, time_dim=16, channels=8, dtype="f32")
    assert _tree_params(w) == _count(D, F, D // H, 2, 3, False, 48, 24, 16, 8)
    w = synth.flux_weights(rng, D, H, F, 2, 3, txt_dim=48, vec_dim=24, time_dim=16, channels=8, dtype="f32",
                           single_parallel=True)
    assert _tree_params(w) == _count(D, F, D // H, 2, 3, True, 48, 24, 16, 8)
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "parameter_counts.json")))
    D, F = gold["hidden"], gold["mlp_hidden"]
    d = D // gold["heads"]
    (small, large) = gold["variants"]
    par535 = _count(D, F, d, small["joint_layers"], small["single_layers"], True)
    par12 = _count(D, F, d, large["joint_layers"], large["single_layers"], True)
    seq535 = _count(D, F, d, small["joint_layers"], small["single_layers"], False)
    seq12 = _count(D, F, d, large["joint_layers"], large["single_layers"], False)
    # parallel: 535.3 M and 11.89 B; sequential: 563.6 M and 12.97 B
    assert abs(par535 / small["total_params"] - 1) < 0.005 and abs(par12 / large["total_params"] - 1) < 0.015
    assert seq535 / small["total_params"] > 1.04 and seq12 / large["total_params"] > 1.07


def test_parallel_stack_with_zero_gates_and_its_wiring():
    # single blocks of the parallel form: zero gates everywhere give the head of the embedded
    # latents; with the gates on, one double and one parallel single block equal that chain
    # written out (the single block over [img; txt], the head on the image rows)
    w, z, txt, t, y, ids, H = _stack(seed=11, single_parallel=True)
    w0 = dict(w)
    w0["double"] = [(_zero_gates(a), _zero_gates(b)) for a, b in w["double"]]
    w0["single"] = [_zero_gates(s, (2,)) for s in w["single"]]
    vec = O.conditioning_vec(t, y, w)
    f = w["final"]
    exp = O.final_layer(O.img_in(z, *w["img_in"]), vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], 4, 4)
    np.testing.assert_allclose(O.flux_forward(z, txt, t, y, ids, w0, H, axes_dim=AX, single_parallel=True), exp,
                               atol=1e-13)
    w1 = dict(w, double=w["double"][:1], single=w["single"][:1])
    cos, sin = O.rope_cos_sin(ids, AX)
    xi, xt = O.double_block(O.img_in(z, *w["img_in"]), O.txt_in(txt, *w["txt_in"]), vec, cos, sin,
                            *w["double"][0], H)
    c = O.single_block_parallel(np.concatenate([xi, xt], axis=1), vec, cos, sin, w["single"][0], H)
    chain = O.final_layer(c[:, :16], vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], 4, 4)
    got = O.flux_forward(z, txt, t, y, ids, w1, H, axes_dim=AX, single_parallel=True)
    np.testing.assert_allclose(got, chain, atol=1e-12)
    assert np.abs(got - exp).max() > 1e-3
