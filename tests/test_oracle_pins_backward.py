"""Pins of the block-backward oracle by finite differences of the forward (CPU only).

For L = <dy, block(inputs, weights)> with a random dy, the gradient of L with respect to any
tensor T is what the backward returns for T.  Each check compares <grad_T, V> for a random
direction V with the central difference (L(T + eps V) - L(T - eps V)) / (2 eps) of the forward
oracle in float64: an error in any step of the backward (a dropped term, a transposed operand,
a wrong sign) shows as a mismatch far above the O(eps^2) difference error.  Covered: the double
block (both streams, the joint attention, both RoPE pairings, the tanh GELU) and the single
block, for the block inputs, the conditioning vector and every weight.
"""
import math

import numpy as np
import pytest

from diffusion_transformer_flux_gb300 import synth
from oracle import backward as BW
from oracle import flux as O

AX = (2, 2, 4)  # RoPE axes of the 8-wide heads below
EPS = 1e-6


def _case(seed, single, B=2, S_i=5, S_t=3, D=16, H=2, F=32):
    rng = np.random.default_rng(seed)
    # float64 copies: a perturbation of EPS must not be rounded away by a float32 tensor
    w_img = {k: v.astype(np.float64) for k, v in synth.stream_weights(rng, D, H, D // H, F, "f32", 0.3,
                                                                      gain_jitter=0.2).items()}
    w_txt = {k: v.astype(np.float64) for k, v in synth.stream_weights(rng, D, H, D // H, F, "f32", 0.3,
                                                                      gain_jitter=0.2).items()}
    x_img = rng.standard_normal((B, S_i, D))
    x_txt = rng.standard_normal((B, S_t, D))
    vec = rng.standard_normal((B, D))
    ids = synth.position_ids(B, 1, S_i, S_t)
    ids[..., 0] = rng.integers(0, 3, size=ids.shape[:-1])  # non-zero ids on every axis
    cos, sin = O.rope_cos_sin(ids, AX)
    if single:
        x = np.concatenate([x_img, x_txt], axis=1)
        return dict(x=x), dict(w=w_img), vec, cos, sin, H, rng
    return dict(x_img=x_img, x_txt=x_txt), dict(w_img=w_img, w_txt=w_txt), vec, cos, sin, H, rng


def _directional(loss, grad, T, rng, n=3):
    """Compare <grad, V> with the central difference of loss along V for n random V."""
    for _ in range(n):
        V = rng.standard_normal(np.shape(T))
        base = np.array(T, dtype=np.float64, copy=True)

        def at(s):
            T[...] = base + s * EPS * V
            return loss()
        fd = (at(1.0) - at(-1.0)) / (2 * EPS)
        T[...] = base
        an = float(np.sum(grad * V))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (fd, an)


@pytest.mark.parametrize("interleaved,tanh", [(True, False), (False, True)])
def test_double_block_gradients_match_finite_differences(interleaved, tanh):
    xs, ws, vec, cos, sin, H, rng = _case(11, False)
    dy_i = rng.standard_normal(xs["x_img"].shape)
    dy_t = rng.standard_normal(xs["x_txt"].shape)

    def loss():
        yi, yt = O.double_block(xs["x_img"], xs["x_txt"], vec, cos, sin, ws["w_img"], ws["w_txt"], H,
                                interleaved, tanh)
        return float(np.sum(yi * dy_i) + np.sum(yt * dy_t))

    dxi, dxt, dvec, gi, gt = BW.double_block_backward(xs["x_img"], xs["x_txt"], vec, cos, sin, ws["w_img"],
                                                      ws["w_txt"], H, dy_i, dy_t, interleaved, tanh)
    _directional(loss, dxi, xs["x_img"], rng)
    _directional(loss, dxt, xs["x_txt"], rng)
    _directional(loss, dvec, vec, rng)
    for w, g in ((ws["w_img"], gi), (ws["w_txt"], gt)):
        assert set(g) == set(w)
        for name in w:
            _directional(loss, g[name], w[name], rng, n=2)


def test_single_block_gradients_match_finite_differences():
    xs, ws, vec, cos, sin, H, rng = _case(12, True)
    dy = rng.standard_normal(xs["x"].shape)

    def loss():
        return float(np.sum(O.single_block(xs["x"], vec, cos, sin, ws["w"], H) * dy))

    dx, dvec, g = BW.single_block_backward(xs["x"], vec, cos, sin, ws["w"], H, dy)
    _directional(loss, dx, xs["x"], rng)
    _directional(loss, dvec, vec, rng)
    for name in ws["w"]:
        _directional(loss, g[name], ws["w"][name], rng, n=2)


def test_backward_forward_intermediates_match_the_forward_oracle():
    # the backward's own recomputation of the forward agrees with oracle.flux (so the pins above
    # test the gradient of the block the forward oracle defines)
    xs, ws, vec, cos, sin, H, rng = _case(13, True)
    m = BW._modulation(vec, ws["w"])
    c = BW._stream_pre(xs["x"], m, ws["w"], H, BW.LN_EPS, BW.RMS_EPS)
    q = BW.rope_rotate(c["qn"], cos[:, None], sin[:, None])
    k = BW.rope_rotate(c["kn"], cos[:, None], sin[:, None])
    o, _ = BW.attention_fwd(q, k, c["v"])
    y, _ = BW._stream_post(xs["x"], BW._merge(o), m, ws["w"], False, BW.LN_EPS)
    np.testing.assert_allclose(y, O.single_block(xs["x"], vec, cos, sin, ws["w"], H), atol=1e-12)


def _f64_tree(w):
    if isinstance(w, dict):
        return {k: _f64_tree(v) for k, v in w.items()}
    if isinstance(w, (list, tuple)):
        return type(w)(_f64_tree(v) for v in w)
    return np.array(w, dtype=np.float64)


def test_loss_gradient_matches_finite_differences():
    rng = np.random.default_rng(20)
    z0, z1, pred = (rng.standard_normal((2, 3, 4, 5)) for _ in range(3))
    grad = BW.flow_match_loss_grad(pred, z0, z1)
    _directional(lambda: O.flow_match_loss(pred, z0, z1), grad, pred, rng)


def test_whole_model_gradients_match_finite_differences():
    # 1 double + 1 single block, 8-wide heads, guidance on: every input and every weight group
    rng = np.random.default_rng(21)
    D, H, F, lat_h, lat_w, S_t, txt_dim, vec_dim, B = 16, 2, 32, 2, 3, 3, 8, 8, 2
    w = _f64_tree(synth.flux_weights(rng, D, H, F, 1, 1, txt_dim=txt_dim, vec_dim=vec_dim, guidance=True,
                                     dtype="f32", std=0.3))
    z = rng.standard_normal((B, 64, lat_h, lat_w))
    txt = rng.standard_normal((B, S_t, txt_dim))
    t = rng.uniform(0.1, 0.9, B)
    y = rng.standard_normal((B, vec_dim))
    g = np.array([1.5, 3.0])
    ids = synth.position_ids(B, lat_h, lat_w, S_t)
    cos, sin = O.rope_cos_sin(ids, AX)
    dpred = rng.standard_normal(z.shape)

    def loss():
        return float(np.sum(O.flux_forward(z, txt, t, y, ids, w, H, g=g, axes_dim=AX) * dpred))

    ins, gw = BW.model_backward(z, txt, t, y, cos, sin, w, H, dpred, g=g)
    for name, T in (("z_t", z), ("txt", txt), ("y", y), ("g", g)):
        _directional(loss, ins[name], T, rng, n=2)
    # t: through the sinusoid (angles up to 1000 rad: a smaller step keeps the difference exact)
    base = t.copy()
    for _ in range(2):
        V = rng.standard_normal(t.shape)
        e = 1e-8
        t[...] = base + e * V
        a = loss()
        t[...] = base - e * V
        b = loss()
        t[...] = base
        fd, an = (a - b) / (2 * e), float(np.sum(ins["t"] * V))
        assert abs(fd - an) <= 1e-4 * max(1.0, abs(fd)), (fd, an)
    for key in ("img_in", "txt_in", "time_in", "vector_in", "guidance_in"):
        for T, G in zip(w[key], gw[key]):
            _directional(loss, G, T, rng, n=1)
    for name in w["final"]:
        _directional(loss, gw["final"][name], w["final"][name], rng, n=1)
    for name in ("w_mod", "w_qkv", "g_k", "w_1", "b_2"):
        _directional(loss, gw["double"][0][0][name], w["double"][0][0][name], rng, n=1)
        _directional(loss, gw["double"][0][1][name], w["double"][0][1][name], rng, n=1)
        _directional(loss, gw["single"][0][name], w["single"][0][name], rng, n=1)


def test_parallel_single_block_gradients_match_finite_differences():
    xs, ws, vec, cos, sin, H, rng = _case(14, True)
    w = ws["w"]
    D = w["w_o"].shape[0]
    w["w_mod"], w["b_mod"] = w["w_mod"][:3 * D].copy(), w["b_mod"][:3 * D].copy()
    dy = rng.standard_normal(xs["x"].shape)

    def loss():
        return float(np.sum(O.single_block_parallel(xs["x"], vec, cos, sin, w, H) * dy))

    dx, dvec, g = BW.single_block_parallel_backward(xs["x"], vec, cos, sin, w, H, dy)
    _directional(loss, dx, xs["x"], rng)
    _directional(loss, dvec, vec, rng)
    assert set(g) == set(w)
    for name in w:
        _directional(loss, g[name], w[name], rng, n=2)


def test_attention_backward_in_the_saved_log_sum_exp_form():
    # The form a flash-style backward computes in: P recomputed from the scores and the row
    # log-sum-exp L saved by the forward, P = exp(S / sqrt(d) - L); and the row term of the
    # softmax gradient taken as D = rowsum(dO * O) instead of rowsum(P * dP).  Both are
    # identities (O = P V, so rowsum(P * (dO V^T)) = rowsum(dO * (P V))); they are checked here
    # against brute force over the keys, and the oracle's gradients against the form they give.
    rng = np.random.default_rng(7)
    B, H, S, d = 1, 2, 37, 16
    q, k, v = (rng.standard_normal((B, H, S, d)) * 2.0 for _ in range(3))
    do = rng.standard_normal((B, H, S, d))
    s = q @ np.swapaxes(k, -1, -2) / math.sqrt(d)
    lse = np.empty((B, H, S))
    for h in range(H):
        for i in range(S):
            m = max(s[0, h, i])
            lse[0, h, i] = m + math.log(sum(math.exp(x - m) for x in s[0, h, i]))
    p = np.exp(s - lse[..., None])
    o, p_oracle = BW.attention_fwd(q, k, v)
    np.testing.assert_allclose(p, p_oracle, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=1e-13)
    dp = do @ np.swapaxes(v, -1, -2)
    D = (do * o).sum(axis=-1)
    np.testing.assert_allclose(D, (p * dp).sum(axis=-1), rtol=1e-10, atol=1e-12)
    ds = p * (dp - D[..., None])
    dq, dk, dv = BW.attention_bwd(do, q, k, v, p_oracle)
    np.testing.assert_allclose(dq, ds @ k / math.sqrt(d), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, np.swapaxes(ds, -1, -2) @ q / math.sqrt(d), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, np.swapaxes(p, -1, -2) @ do, rtol=1e-10, atol=1e-12)


def test_whole_model_with_parallel_single_blocks_matches_finite_differences():
    # the parallel-branch single blocks in the whole model: inputs, the conditioning path and the
    # single block's weights (three modulation chunks)
    rng = np.random.default_rng(22)
    D, H, F, lat_h, lat_w, S_t, txt_dim, vec_dim, B = 16, 2, 32, 2, 3, 3, 8, 8, 2
    w = _f64_tree(synth.flux_weights(rng, D, H, F, 1, 2, txt_dim=txt_dim, vec_dim=vec_dim, dtype="f32",
                                     std=0.3, single_parallel=True))
    z = rng.standard_normal((B, 64, lat_h, lat_w))
    txt = rng.standard_normal((B, S_t, txt_dim))
    t = rng.uniform(0.1, 0.9, B)
    y = rng.standard_normal((B, vec_dim))
    ids = synth.position_ids(B, lat_h, lat_w, S_t)
    cos, sin = O.rope_cos_sin(ids, AX)
    dpred = rng.standard_normal(z.shape)

    def loss():
        return float(np.sum(O.flux_forward(z, txt, t, y, ids, w, H, axes_dim=AX, single_parallel=True) * dpred))

    ins, gw = BW.model_backward(z, txt, t, y, cos, sin, w, H, dpred, single_parallel=True)
    for name, T in (("z_t", z), ("txt", txt), ("y", y)):
        _directional(loss, ins[name], T, rng, n=2)
    for key in ("time_in", "vector_in"):
        for T, G in zip(w[key], gw[key]):
            _directional(loss, G, T, rng, n=1)
    for i in range(2):
        for name in ("w_mod", "b_mod", "w_qkv", "g_q", "w_o", "w_1", "b_1", "w_2", "b_o"):
            _directional(loss, gw["single"][i][name], w["single"][i][name], rng, n=1)
