"""Pins of the fp64 oracle's whole blocks, output head and embeddings (CPU only).

* A scalar-loop restatement of the double block on tiny shapes (brute force).
* Closed forms: zero gates give the identity; scale = -1, shift = 0 makes the
  attention branch a constant (the attention of identical values), which the
  block must reproduce through its output projection.
* Invariants: stream symmetry (double block with equal weights == single
  block), permutation equivariance, RoPE shift invariance, row sampling.
"""
import math

import numpy as np
import pytest

from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

TINY = dict(B=2, S_i=5, S_t=3, D=16, H=2, F=24)
AX = (2, 2, 4)  # sum = head_dim 8


def _weights(rng, D, H, F, std=0.3):
    w = synth.stream_weights(rng, D, H, D // H, F, dtype="f32", std=std, gain_jitter=0.1)
    return {k: v.astype(np.float64) for k, v in w.items()}


def _setup(seed=0, std=0.3, **kw):
    p = dict(TINY, **kw)
    rng = np.random.default_rng(seed)
    B, S_i, S_t, D, H, F = p["B"], p["S_i"], p["S_t"], p["D"], p["H"], p["F"]
    wi, wt = _weights(rng, D, H, F, std), _weights(rng, D, H, F, std)
    x_img = rng.standard_normal((B, S_i, D))
    x_txt = rng.standard_normal((B, S_t, D))
    vec = rng.standard_normal((B, D))
    ids = np.concatenate([rng.integers(0, 9, size=(B, S_i, 3)), np.zeros((B, S_t, 3))], 1).astype(float)
    cos, sin = O.rope_cos_sin(ids, AX)
    return p, wi, wt, x_img, x_txt, vec, ids, cos, sin


# ----------------------------------------------------------------------------- brute force
def _bf_block(x_img, x_txt, vec, ids, wi, wt, H, axes, theta=1e4):
    """Scalar loops, written from the pages' step list, sharing nothing with the oracle."""
    B, S_i, D = x_img.shape
    S_t = x_txt.shape[1]
    d = D // H

    def lin(row, W, b):
        return [sum(W[o][i] * row[i] for i in range(len(row))) + b[o] for o in range(len(b))]

    def ln(row):
        mu = sum(row) / len(row)
        var = sum((r - mu) ** 2 for r in row) / len(row)
        return [(r - mu) / math.sqrt(var + 1e-6) for r in row]

    def gelu(z):
        return 0.5 * z * (1 + math.erf(z / math.sqrt(2)))

    def angle(pid, j):
        # pair j of the concatenated per-axis pairs
        off = 0
        for a, da in enumerate(axes):
            if j < off + da // 2:
                i = j - off
                return pid[a] / theta ** (2 * i / da)
            off += da // 2
        raise AssertionError

    out_img = np.zeros_like(x_img)
    out_txt = np.zeros_like(x_txt)
    for b in range(B):
        sv = [v / (1 + math.exp(-v)) for v in vec[b]]
        mod = {}
        for name, w in (("img", wi), ("txt", wt)):
            m = lin(sv, w["w_mod"], w["b_mod"])
            mod[name] = [m[c * D:(c + 1) * D] for c in range(6)]
        toks = [("img", x_img[b, s]) for s in range(S_i)] + [("txt", x_txt[b, s]) for s in range(S_t)]
        W = {"img": wi, "txt": wt}
        Q, K, V = [], [], []
        for n, (st, x) in enumerate(toks):
            sh, sc = mod[st][0], mod[st][1]
            h = [v * (1 + sc[i]) + sh[i] for i, v in enumerate(ln(list(x)))]
            qkv = lin(h, W[st]["w_qkv"], W[st]["b_qkv"])
            qh, kh, vh = [], [], []
            for hh in range(H):
                for which, dst, g in ((0, qh, W[st]["g_q"]), (1, kh, W[st]["g_k"])):
                    seg = qkv[which * D + hh * d: which * D + (hh + 1) * d]
                    r = math.sqrt(sum(z * z for z in seg) / d + 1e-6)
                    seg = [z / r * g[j] for j, z in enumerate(seg)]
                    rot = list(seg)
                    for j in range(d // 2):
                        a = angle(ids[b, n], j)
                        x0, x1 = seg[2 * j], seg[2 * j + 1]
                        rot[2 * j] = x0 * math.cos(a) - x1 * math.sin(a)
                        rot[2 * j + 1] = x0 * math.sin(a) + x1 * math.cos(a)
                    dst.append(rot)
                vh.append(qkv[2 * D + hh * d: 2 * D + (hh + 1) * d])
            Q.append(qh), K.append(kh), V.append(vh)
        S = len(toks)
        for n, (st, x) in enumerate(toks):
            att = []
            for hh in range(H):
                sc_ = [sum(Q[n][hh][j] * K[m][hh][j] for j in range(d)) / math.sqrt(d) for m in range(S)]
                mx = max(sc_)
                e = [math.exp(z - mx) for z in sc_]
                z = sum(e)
                att += [sum(e[m] / z * V[m][hh][j] for m in range(S)) for j in range(d)]
            w = W[st]
            md = mod[st]
            proj = lin(att, w["w_o"], w["b_o"])
            x1 = [x[i] + md[2][i] * proj[i] for i in range(D)]
            h2 = [v * (1 + md[4][i]) + md[3][i] for i, v in enumerate(ln(x1))]
            u = [gelu(z) for z in lin(h2, w["w_1"], w["b_1"])]
            y = lin(u, w["w_2"], w["b_2"])
            x2 = [x1[i] + md[5][i] * y[i] for i in range(D)]
            if st == "img":
                out_img[b, n] = x2
            else:
                out_txt[b, n - S_i] = x2
    return out_img, out_txt


def test_double_block_matches_scalar_brute_force():
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup()
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wt, p["H"])
    bi, bt = _bf_block(x_img, x_txt, vec, ids, wi, wt, p["H"], AX)
    np.testing.assert_allclose(yi, bi, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(yt, bt, rtol=1e-11, atol=1e-11)


# ----------------------------------------------------------------------------- closed forms
def _zero_gate(w, D):
    w = dict(w)
    w["w_mod"] = w["w_mod"].copy()
    w["b_mod"] = w["b_mod"].copy()
    for c in (2, 5):
        w["w_mod"][c * D:(c + 1) * D] = 0
        w["b_mod"][c * D:(c + 1) * D] = 0
    return w


def test_zero_gates_make_blocks_the_identity():
    # P5
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(1)
    D = p["D"]
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, _zero_gate(wi, D), _zero_gate(wt, D), p["H"])
    np.testing.assert_array_equal(yi, x_img)
    np.testing.assert_array_equal(yt, x_txt)
    x = np.concatenate([x_img, x_txt], 1)
    np.testing.assert_array_equal(O.single_block(x, vec, cos, sin, _zero_gate(wi, D), p["H"]), x)
    # all-zero modulation (weights and bias) is the identity too
    w0 = dict(wi, w_mod=0 * wi["w_mod"], b_mod=0 * wi["b_mod"])
    np.testing.assert_array_equal(O.single_block(x, vec, cos, sin, w0, p["H"]), x)


def _const_mod(w, D, chunks):
    """Modulation that ignores vec: chunk c = constant vector chunks[c]."""
    w = dict(w)
    w["w_mod"] = np.zeros_like(w["w_mod"])
    w["b_mod"] = np.concatenate([np.broadcast_to(np.asarray(c, float), (D,)) for c in chunks])
    return w


def test_attention_branch_closed_form_when_scale_is_minus_one():
    # shift1 = 0, scale1 = -1: every token's modulated input is 0, so qkv = b_qkv;
    # with one value bias b_v for both streams every value is b_v and the
    # attention output is b_v whatever the weights;
    # with gate1 = 1 and gate2 = 0 the block returns x + (b_v W_o^T + b_o).
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(2)
    D = p["D"]
    wi = _const_mod(wi, D, [0, -1, 1, 0, 0, 0])
    wt = _const_mod(wt, D, [0, -1, 1, 0, 0, 0])
    # joint attention mixes both streams' values: give them the same value bias
    wt["b_qkv"] = np.concatenate([wt["b_qkv"][:2 * D], wi["b_qkv"][2 * D:]])
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wt, p["H"])
    for y, x, w in ((yi, x_img, wi), (yt, x_txt, wt)):
        b_v = w["b_qkv"][2 * D:]
        branch = np.array([sum(w["w_o"][o, i] * b_v[i] for i in range(D)) + w["b_o"][o] for o in range(D)])
        np.testing.assert_allclose(y, x + branch, rtol=1e-12, atol=1e-12)


def test_mlp_branch_closed_form_when_scale_is_minus_one():
    # gate1 = 0; shift2 = c, scale2 = -1: the MLP input is c for every token.
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(3)
    D = p["D"]
    c = np.linspace(-1, 1, D)
    w = _const_mod(wi, D, [0, 0, 0, c, -1, 1])
    x = np.concatenate([x_img, x_txt], 1)
    y = O.single_block(x, vec, cos, sin, w, p["H"])
    pre = w["w_1"] @ c + w["b_1"]
    u = np.array([z * 0.5 * (1 + math.erf(z / math.sqrt(2))) for z in pre])
    branch = w["w_2"] @ u + w["b_2"]
    np.testing.assert_allclose(y, x + branch, rtol=1e-12, atol=1e-12)


def test_final_layer_closed_form_and_unpatchify_layout():
    rng = np.random.default_rng(4)
    B, H, W, C, D = 2, 3, 4, 5, 8
    x = rng.standard_normal((B, H * W, D))
    vec = rng.standard_normal((B, D))
    w_out = rng.standard_normal((C, D))
    b_out = rng.standard_normal(C)
    c = rng.standard_normal(D)
    w_ada = np.zeros((2 * D, D))
    b_ada = np.concatenate([c, -np.ones(D)])  # shift = c, scale = -1
    y = O.final_layer(x, vec, w_ada, b_ada, w_out, b_out, H, W)
    assert y.shape == (B, C, H, W)
    np.testing.assert_allclose(y, np.broadcast_to((w_out @ c + b_out)[None, :, None, None], y.shape), rtol=1e-12)
    # token r*W + col lands at [:, :, r, col]
    w_ada = rng.standard_normal((2 * D, D))
    b_ada = rng.standard_normal(2 * D)
    y = O.final_layer(x, vec, w_ada, b_ada, w_out, b_out, H, W)
    sh, sc = O.modulation(vec, w_ada, b_ada, 2)
    tok = O.linear(O.modulate(x, sh, sc), w_out, b_out)
    for r in range(H):
        for col in range(W):
            np.testing.assert_array_equal(y[:, :, r, col], tok[:, r * W + col, :])
    z = rng.standard_normal((B, C, H, W))
    t = O.patchify(z)
    for r in range(H):
        for col in range(W):
            np.testing.assert_array_equal(t[:, r * W + col, :], z[:, :, r, col])
    np.testing.assert_array_equal(O.unpatchify(t, H, W), z)


# ----------------------------------------------------------------------------- invariants
def test_stream_symmetry_double_equals_single():
    # P7: equal weights in both streams -> the double block is the single block on [img; txt].
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(5)
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wi, p["H"])
    y = O.single_block(np.concatenate([x_img, x_txt], 1), vec, cos, sin, wi, p["H"])
    np.testing.assert_allclose(np.concatenate([yi, yt], 1), y, rtol=1e-12, atol=1e-12)


def test_permutation_equivariance():
    # P8: permuting tokens together with their ids permutes the outputs.
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(6)
    x = np.concatenate([x_img, x_txt], 1)
    y = O.single_block(x, vec, cos, sin, wi, p["H"])
    perm = np.random.default_rng(0).permutation(x.shape[1])
    yp = O.single_block(x[:, perm], vec, cos[:, perm], sin[:, perm], wi, p["H"])
    np.testing.assert_allclose(yp, y[:, perm], rtol=1e-12, atol=1e-12)
    # double block: permute within each stream
    pi = np.random.default_rng(1).permutation(p["S_i"])
    pt = np.random.default_rng(2).permutation(p["S_t"])
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wt, p["H"])
    jp = np.concatenate([pi, p["S_i"] + pt])
    yip, ytp = O.double_block(x_img[:, pi], x_txt[:, pt], vec, cos[:, jp], sin[:, jp], wi, wt, p["H"])
    np.testing.assert_allclose(yip, yi[:, pi], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ytp, yt[:, pt], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("axis", [1, 2])
def test_rope_shift_invariance_of_the_block(axis):
    # P3: the same offset added to every token's axis id leaves the block unchanged.
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(7)
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wt, p["H"])
    ids2 = ids.copy()
    ids2[..., axis] += 13.0
    c2, s2 = O.rope_cos_sin(ids2, AX)
    yi2, yt2 = O.double_block(x_img, x_txt, vec, c2, s2, wi, wt, p["H"])
    np.testing.assert_allclose(yi2, yi, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(yt2, yt, rtol=1e-10, atol=1e-10)


def test_half_split_rope_path_also_shift_invariant():
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(8)
    x = np.concatenate([x_img, x_txt], 1)
    y = O.single_block(x, vec, cos, sin, wi, p["H"], interleaved=False)
    ids2 = ids + np.array([0.0, 4.0, 0.0])
    c2, s2 = O.rope_cos_sin(ids2, AX)
    np.testing.assert_allclose(O.single_block(x, vec, c2, s2, wi, p["H"], interleaved=False), y,
                               rtol=1e-10, atol=1e-10)


def test_row_sampled_blocks_equal_full_blocks():
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(9, S_i=11, S_t=6)
    yi, yt = O.double_block(x_img, x_txt, vec, cos, sin, wi, wt, p["H"])
    ri, rt = np.array([0, 3, 10]), np.array([1, 5])
    si, st = O.double_block_rows(x_img, x_txt, vec, cos, sin, wi, wt, p["H"], ri, rt)
    np.testing.assert_allclose(si, yi[:, ri], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st, yt[:, rt], rtol=1e-12, atol=1e-12)
    x = np.concatenate([x_img, x_txt], 1)
    y = O.single_block(x, vec, cos, sin, wi, p["H"])
    rows = np.array([2, 12, 16])
    np.testing.assert_allclose(O.single_block_rows(x, vec, cos, sin, wi, p["H"], rows), y[:, rows],
                               rtol=1e-12, atol=1e-12)


def test_text_tokens_at_origin_are_not_rotated():
    # P1 at block level: with all ids 0 the block equals one computed with RoPE disabled
    # (cos = 1, sin = 0 everywhere), independent of the pairing convention.
    p, wi, wt, x_img, x_txt, vec, ids, cos, sin = _setup(10)
    c0, s0 = O.rope_cos_sin(np.zeros_like(ids), AX)
    a = O.double_block(x_img, x_txt, vec, c0, s0, wi, wt, p["H"], interleaved=True)
    b = O.double_block(x_img, x_txt, vec, c0, s0, wi, wt, p["H"], interleaved=False)
    for u, v in zip(a, b):
        np.testing.assert_allclose(u, v, rtol=1e-13, atol=1e-13)
