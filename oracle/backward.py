"""fp64 CPU oracle of the Flux block backward: gradients of the double- and single-block
forward of ``oracle.flux`` with respect to its inputs, its conditioning vector and every weight.

TEST INFRASTRUCTURE ONLY, like ``oracle.flux``: nothing in the library imports it and it shares
no code with the CUDA path.  The pages train these blocks ("Flux architecture deep dive",
§Training data flow; "Flux model API reference", §Training workflow example) but print no
backward.  Each function here is the chain rule applied to the forward step it names, written
out op by op in reverse order, in float64.  The forward intermediates the backward needs are
recomputed here from their definitions, not taken from ``oracle.flux``.  The gradients are
pinned in the tests by finite differences of the (separately pinned) forward.
"""
from __future__ import annotations

import math

import numpy as np

LN_EPS = 1e-6
RMS_EPS = 1e-6


def _f(x):
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------- per-op backward
def linear_fwd(x, w, b):
    """y = x W^T + b, W [out, in]."""
    return _f(x) @ _f(w).T + _f(b)


def linear_bwd(dy, x, w):
    """(dx, dW, db) of y = x W^T + b: dx = dy W, dW = sum over rows of dy^T x, db = sum dy."""
    dy, x, w = _f(dy), _f(x), _f(w)
    dx = dy @ w
    dw = dy.reshape(-1, dy.shape[-1]).T @ x.reshape(-1, x.shape[-1])
    db = dy.reshape(-1, dy.shape[-1]).sum(axis=0)
    return dx, dw, db


def layernorm_fwd(x, eps=LN_EPS):
    """xhat = (x - mean) r with r = 1/sqrt(biased var + eps); returns (xhat, r)."""
    x = _f(x)
    mu = x.mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(((x - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    return (x - mu) * r, r


def layernorm_bwd(dxhat, xhat, r):
    """dx of xhat = (x - mean(x)) r(x): r (dxhat - mean(dxhat) - xhat mean(dxhat xhat))."""
    dxhat = _f(dxhat)
    return r * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))


def modulate_bwd(dh, xhat, r, scale):
    """Gradients of h = xhat (1 + scale[b]) + shift[b] (xhat the LayerNorm of x):
    (dx, dshift [B, D], dscale [B, D])."""
    dh = _f(dh)
    dshift = dh.sum(axis=1)
    dscale = (dh * xhat).sum(axis=1)
    dx = layernorm_bwd(dh * (1.0 + _f(scale)[:, None, :]), xhat, r)
    return dx, dshift, dscale


def gated_residual_bwd(dy, gate, z):
    """Gradients of y = x + gate[b] z: (dx, dz, dgate [B, D])."""
    dy = _f(dy)
    return dy, dy * _f(gate)[:, None, :], (dy * _f(z)).sum(axis=1)


def rmsnorm_fwd(x, g, eps=RMS_EPS):
    """y = x r g with r = 1/sqrt(mean(x^2) + eps) over the last axis; returns (y, xn, r), xn = x r."""
    x = _f(x)
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    xn = x * r
    return xn * _f(g), xn, r


def rmsnorm_bwd(dy, xn, r, g):
    """(dx, dg) of y = x r(x) g: dg = sum dy xn; dx = r (dy g - xn mean(dy g xn))."""
    dy = _f(dy)
    dyg = dy * _f(g)
    dx = r * (dyg - xn * (dyg * xn).mean(axis=-1, keepdims=True))
    dg = (dy * xn).reshape(-1, xn.shape[-1]).sum(axis=0)
    return dx, dg


def rope_rotate(x, cos, sin, interleaved=True):
    """Each pair (a, b) of x's last axis -> (a cos - b sin, a sin + b cos)."""
    x = _f(x)
    d = x.shape[-1]
    a, b = (x[..., 0::2], x[..., 1::2]) if interleaved else (x[..., : d // 2], x[..., d // 2:])
    out = np.empty_like(x)
    ra, rb = a * cos - b * sin, a * sin + b * cos
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


def rope_bwd(dy, cos, sin, interleaved=True):
    """The rotation is orthogonal: its gradient is the rotation by the opposite angle."""
    return rope_rotate(dy, cos, -_f(sin), interleaved)


def attention_fwd(q, k, v):
    """O = P V with P = softmax(q k^T / sqrt(d)); returns (O, P)."""
    q, k, v = _f(q), _f(k), _f(v)
    s = q @ np.swapaxes(k, -1, -2) / math.sqrt(q.shape[-1])
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v, p


def attention_bwd(do, q, k, v, p):
    """(dq, dk, dv): dV = P^T dO; dP = dO V^T; dS = P (dP - rowsum(P dP)); dQ = dS K / sqrt(d);
    dK = dS^T Q / sqrt(d)."""
    do, q, k, v = _f(do), _f(q), _f(k), _f(v)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    sc = 1.0 / math.sqrt(q.shape[-1])
    return ds @ k * sc, np.swapaxes(ds, -1, -2) @ q * sc, dv


def gelu_fwd(u, tanh=False):
    u = _f(u)
    if tanh:
        c = math.sqrt(2.0 / math.pi)
        return 0.5 * u * (1.0 + np.tanh(c * (u + 0.044715 * u ** 3)))
    return 0.5 * u * (1.0 + np.vectorize(math.erf, otypes=[np.float64])(u / math.sqrt(2.0)))


def gelu_grad(u, tanh=False):
    """d/du of GELU: Phi(u) + u phi(u) (erf form), or the derivative of the tanh form."""
    u = _f(u)
    if tanh:
        c = math.sqrt(2.0 / math.pi)
        t = np.tanh(c * (u + 0.044715 * u ** 3))
        return 0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * c * (1.0 + 3 * 0.044715 * u * u)
    cdf = 0.5 * (1.0 + np.vectorize(math.erf, otypes=[np.float64])(u / math.sqrt(2.0)))
    return cdf + u * np.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)


def silu_fwd(v):
    v = _f(v)
    return v / (1.0 + np.exp(-v))


def silu_grad(v):
    """d/dv of v sigma(v): sigma(v) (1 + v (1 - sigma(v)))."""
    sg = 1.0 / (1.0 + np.exp(-_f(v)))
    return sg * (1.0 + _f(v) * (1.0 - sg))


def _heads(x, h):
    B, S, HD = x.shape
    return x.reshape(B, S, h, HD // h).transpose(0, 2, 1, 3)


def _merge(x):
    B, H, S, d = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B, S, H * d)


# ----------------------------------------------------------------------------- one stream
def _stream_pre(x, m, w, heads, ln_eps, rms_eps):
    """Attention-branch prologue of one stream: LN1-modulate, QKV linear, per-head RMSNorm."""
    D = np.shape(x)[-1]
    xhat1, r1 = layernorm_fwd(x, ln_eps)
    h1 = xhat1 * (1.0 + m[1][:, None, :]) + m[0][:, None, :]
    qkv = linear_fwd(h1, w["w_qkv"], w["b_qkv"])
    q, k, v = (_heads(qkv[..., i * D:(i + 1) * D], heads) for i in range(3))
    qn, qxn, qr = rmsnorm_fwd(q, w["g_q"], rms_eps)
    kn, kxn, kr = rmsnorm_fwd(k, w["g_k"], rms_eps)
    return dict(xhat1=xhat1, r1=r1, h1=h1, qn=qn, qxn=qxn, qr=qr, kn=kn, kxn=kxn, kr=kr, v=v)


def _stream_post(x, o, m, w, gelu_tanh, ln_eps):
    """Everything after the attention for one stream, with its intermediates."""
    a = linear_fwd(o, w["w_o"], w["b_o"])
    x1 = _f(x) + m[2][:, None, :] * a
    xhat2, r2 = layernorm_fwd(x1, ln_eps)
    h2 = xhat2 * (1.0 + m[4][:, None, :]) + m[3][:, None, :]
    u_pre = linear_fwd(h2, w["w_1"], w["b_1"])
    u = gelu_fwd(u_pre, gelu_tanh)
    z = linear_fwd(u, w["w_2"], w["b_2"])
    y = x1 + m[5][:, None, :] * z
    return y, dict(o=o, a=a, x1=x1, xhat2=xhat2, r2=r2, h2=h2, u_pre=u_pre, u=u, z=z)


def _stream_post_bwd(dy, m, w, c, gelu_tanh):
    """Backward of _stream_post: (dx, do, dm [6 chunks], weight grads)."""
    g = {}
    dx1, dz, dg2 = gated_residual_bwd(dy, m[5], c["z"])
    du, g["w_2"], g["b_2"] = linear_bwd(dz, c["u"], w["w_2"])
    du_pre = du * gelu_grad(c["u_pre"], gelu_tanh)
    dh2, g["w_1"], g["b_1"] = linear_bwd(du_pre, c["h2"], w["w_1"])
    dx1_ln, dsh2, dsc2 = modulate_bwd(dh2, c["xhat2"], c["r2"], m[4])
    dx1 = dx1 + dx1_ln
    dx, da, dg1 = gated_residual_bwd(dx1, m[2], c["a"])
    do, g["w_o"], g["b_o"] = linear_bwd(da, c["o"], w["w_o"])
    return dx, do, [None, None, dg1, dsh2, dsc2, dg2], g


def _stream_pre_bwd(dq, dk, dv, m, w, c, heads):
    """Backward of _stream_pre given the gradients of the normalized q, k and of v ([B,H,S,d]):
    (dx, dshift1, dscale1, weight grads)."""
    g = {}
    dq_raw, g["g_q"] = rmsnorm_bwd(dq, c["qxn"], c["qr"], w["g_q"])
    dk_raw, g["g_k"] = rmsnorm_bwd(dk, c["kxn"], c["kr"], w["g_k"])
    dqkv = np.concatenate([_merge(dq_raw), _merge(dk_raw), _merge(_f(dv))], axis=-1)
    dh1, g["w_qkv"], g["b_qkv"] = linear_bwd(dqkv, c["h1"], w["w_qkv"])
    dx, dsh1, dsc1 = modulate_bwd(dh1, c["xhat1"], c["r1"], m[1])
    return dx, dsh1, dsc1, g


def _modulation(vec, w, n_chunks=6):
    sv = silu_fwd(vec)
    return np.split(linear_fwd(sv, w["w_mod"], w["b_mod"]), n_chunks, axis=-1)


def _modulation_bwd(dm_chunks, vec, w):
    """(dvec, dW_mod, db_mod) of m = SiLU(vec) W_mod^T + b_mod."""
    dm = np.concatenate(dm_chunks, axis=-1)
    sv = silu_fwd(vec)
    dsv, dw, db = linear_bwd(dm, sv, w["w_mod"])
    return dsv * silu_grad(vec), dw, db


# ----------------------------------------------------------------------------- blocks
def double_block_backward(x_img, x_txt, vec, cos, sin, w_img, w_txt, heads, dy_img, dy_txt,
                          interleaved=True, gelu_tanh=False, ln_eps=LN_EPS, rms_eps=RMS_EPS):
    """Gradients of the double block (architecture page, §Model components › 3. MMDiT layer).

    Returns (dx_img, dx_txt, dvec, grads_img, grads_txt); each grads dict has the stream weight
    names (w_mod, b_mod, w_qkv, b_qkv, g_q, g_k, w_o, b_o, w_1, b_1, w_2, b_2).
    """
    S_i = np.shape(x_img)[1]
    mi, mt = _modulation(vec, w_img), _modulation(vec, w_txt)
    ci = _stream_pre(x_img, mi, w_img, heads, ln_eps, rms_eps)
    ct = _stream_pre(x_txt, mt, w_txt, heads, ln_eps, rms_eps)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    q = rope_rotate(np.concatenate([ci["qn"], ct["qn"]], axis=2), cs, sn, interleaved)
    k = rope_rotate(np.concatenate([ci["kn"], ct["kn"]], axis=2), cs, sn, interleaved)
    v = np.concatenate([ci["v"], ct["v"]], axis=2)
    o, p = attention_fwd(q, k, v)
    o = _merge(o)
    _, pi = _stream_post(x_img, o[:, :S_i], mi, w_img, gelu_tanh, ln_eps)
    _, pt = _stream_post(x_txt, o[:, S_i:], mt, w_txt, gelu_tanh, ln_eps)
    # reverse
    dxi, doi, dmi, gi = _stream_post_bwd(dy_img, mi, w_img, pi, gelu_tanh)
    dxt, dot, dmt, gt = _stream_post_bwd(dy_txt, mt, w_txt, pt, gelu_tanh)
    do = _heads(np.concatenate([doi, dot], axis=1), heads)
    dq, dk, dv = attention_bwd(do, q, k, v, p)
    dq, dk = rope_bwd(dq, cs, sn, interleaved), rope_bwd(dk, cs, sn, interleaved)
    dxi2, dmi[0], dmi[1], gi2 = _stream_pre_bwd(dq[:, :, :S_i], dk[:, :, :S_i], dv[:, :, :S_i], mi,
                                                w_img, ci, heads)
    dxt2, dmt[0], dmt[1], gt2 = _stream_pre_bwd(dq[:, :, S_i:], dk[:, :, S_i:], dv[:, :, S_i:], mt,
                                                w_txt, ct, heads)
    gi.update(gi2)
    gt.update(gt2)
    dvi, gi["w_mod"], gi["b_mod"] = _modulation_bwd(dmi, vec, w_img)
    dvt, gt["w_mod"], gt["b_mod"] = _modulation_bwd(dmt, vec, w_txt)
    return dxi + dxi2, dxt + dxt2, dvi + dvt, gi, gt


def single_block_backward(x, vec, cos, sin, w, heads, dy, interleaved=True, gelu_tanh=False,
                          ln_eps=LN_EPS, rms_eps=RMS_EPS):
    """Gradients of the single block over [img; txt] (architecture page, §Model components ›
    4. Flux single block): (dx, dvec, grads)."""
    m = _modulation(vec, w)
    c = _stream_pre(x, m, w, heads, ln_eps, rms_eps)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    q = rope_rotate(c["qn"], cs, sn, interleaved)
    k = rope_rotate(c["kn"], cs, sn, interleaved)
    o, p = attention_fwd(q, k, c["v"])
    _, pc = _stream_post(x, _merge(o), m, w, gelu_tanh, ln_eps)
    dx, do, dm, g = _stream_post_bwd(dy, m, w, pc, gelu_tanh)
    dq, dk, dv = attention_bwd(_heads(do, heads), q, k, c["v"], p)
    dq, dk = rope_bwd(dq, cs, sn, interleaved), rope_bwd(dk, cs, sn, interleaved)
    dx2, dm[0], dm[1], g2 = _stream_pre_bwd(dq, dk, dv, m, w, c, heads)
    g.update(g2)
    dvec, g["w_mod"], g["b_mod"] = _modulation_bwd(dm, vec, w)
    return dx + dx2, dvec, g


# ----------------------------------------------------------------------------- whole model
def flow_match_loss_grad(pred, z0, z1):
    """d/dpred of mean((pred - (z1 - z0))^2) over all elements: 2 (pred - target) / N."""
    pred = _f(pred)
    return 2.0 * (pred - (_f(z1) - _f(z0))) / pred.size


def _patchify(z):
    B, C, H, W = np.shape(z)
    return _f(z).reshape(B, C, H * W).transpose(0, 2, 1)


def _unpatchify(tok, H, W):
    B, S, C = np.shape(tok)
    return _f(tok).transpose(0, 2, 1).reshape(B, C, H, W)


def _sinusoid(t, dim, time_factor, max_period):
    """[cos(tau f), sin(tau f)], tau = time_factor t, f_i = max_period^(-i/half); also tau f."""
    half = dim // 2
    f = max_period ** (-np.arange(half, dtype=np.float64) / half)
    ang = time_factor * _f(t).reshape(-1, 1) * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1), ang, f


def _embedder_fwd(x, w1, b1, w2, b2):
    h = linear_fwd(x, w1, b1)
    a = silu_fwd(h)
    return linear_fwd(a, w2, b2), (x, h, a)


def _embedder_bwd(dout, cache, w1, w2):
    """Backward of Linear2(SiLU(Linear1(x))): (dx, (dw1, db1, dw2, db2))."""
    x, h, a = cache
    da, dw2, db2 = linear_bwd(dout, a, w2)
    dx, dw1, db1 = linear_bwd(da * silu_grad(h), x, w1)
    return dx, (dw1, db1, dw2, db2)


def _double_fwd(x_img, x_txt, vec, cos, sin, wi, wt, heads, interleaved, gelu_tanh):
    """The double block's outputs, recomputed from the pieces above."""
    S_i = np.shape(x_img)[1]
    mi, mt = _modulation(vec, wi), _modulation(vec, wt)
    ci = _stream_pre(x_img, mi, wi, heads, LN_EPS, RMS_EPS)
    ct = _stream_pre(x_txt, mt, wt, heads, LN_EPS, RMS_EPS)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    q = rope_rotate(np.concatenate([ci["qn"], ct["qn"]], axis=2), cs, sn, interleaved)
    k = rope_rotate(np.concatenate([ci["kn"], ct["kn"]], axis=2), cs, sn, interleaved)
    o, _ = attention_fwd(q, k, np.concatenate([ci["v"], ct["v"]], axis=2))
    o = _merge(o)
    yi, _ = _stream_post(x_img, o[:, :S_i], mi, wi, gelu_tanh, LN_EPS)
    yt, _ = _stream_post(x_txt, o[:, S_i:], mt, wt, gelu_tanh, LN_EPS)
    return yi, yt


def _single_fwd(x, vec, cos, sin, w, heads, interleaved, gelu_tanh):
    m = _modulation(vec, w)
    c = _stream_pre(x, m, w, heads, LN_EPS, RMS_EPS)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    o, _ = attention_fwd(rope_rotate(c["qn"], cs, sn, interleaved), rope_rotate(c["kn"], cs, sn, interleaved),
                         c["v"])
    y, _ = _stream_post(x, _merge(o), m, w, gelu_tanh, LN_EPS)
    return y


def _single_parallel_fwd(x, vec, cos, sin, w, heads, interleaved, gelu_tanh):
    m = _modulation(vec, w, 3)
    c = _stream_pre(x, m, w, heads, LN_EPS, RMS_EPS)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    o, _ = attention_fwd(rope_rotate(c["qn"], cs, sn, interleaved), rope_rotate(c["kn"], cs, sn, interleaved),
                         c["v"])
    u = gelu_fwd(linear_fwd(c["h1"], w["w_1"], w["b_1"]), gelu_tanh)
    branch = linear_fwd(_merge(o), w["w_o"], w["b_o"]) + linear_fwd(u, w["w_2"], w["b_2"])
    return _f(x) + m[2][:, None, :] * branch


def model_backward(z_t, txt, t, y, cos, sin, w, heads, dpred, g=None, interleaved=True, gelu_tanh=False,
                   time_dim=256, time_factor=1000.0, max_period=10000.0, single_parallel=False):
    """Gradients of the whole forward of ``oracle.flux.flux_forward`` (conditioning, img_in,
    txt_in, the double blocks, the single blocks over [img; txt], the output head) for the
    cotangent ``dpred`` of the prediction.  ``cos``/``sin`` are the RoPE tables of the joint
    ids.  Returns (inputs, weights): inputs holds dz_t, dtxt, dt, dy (and dg with guidance);
    weights mirrors ``w`` (tuples and stream dicts of the same names).  ``single_parallel``: the
    single blocks are the parallel-branch form, as in ``flux_forward``."""
    single_fwd = _single_parallel_fwd if single_parallel else _single_fwd
    single_bwd = single_block_parallel_backward if single_parallel else single_block_backward
    B, C, H, W = np.shape(z_t)
    S_i = H * W
    # forward, keeping what the backward reads
    feat, ang, freqs = _sinusoid(t, time_dim, time_factor, max_period)
    vt, c_t = _embedder_fwd(feat, *w["time_in"])
    vy, c_y = _embedder_fwd(y, *w["vector_in"])
    vec = vt + vy
    if g is not None:
        wg, bg = (_f(a) for a in w["guidance_in"])
        vec = vec + _f(g).reshape(-1, 1) * wg[None, :] + bg[None, :]
    patches = _patchify(z_t)
    x_img = linear_fwd(patches, *w["img_in"])
    x_txt = linear_fwd(txt, *w["txt_in"])
    ins_d = []
    for wi, wt in w["double"]:
        ins_d.append((x_img, x_txt))
        x_img, x_txt = _double_fwd(x_img, x_txt, vec, cos, sin, wi, wt, heads, interleaved, gelu_tanh)
    c = np.concatenate([x_img, x_txt], axis=1)
    ins_s = []
    for ws in w["single"]:
        ins_s.append(c)
        c = single_fwd(c, vec, cos, sin, ws, heads, interleaved, gelu_tanh)
    f = w["final"]
    sv = silu_fwd(vec)
    shift, scale = np.split(linear_fwd(sv, f["w_ada"], f["b_ada"]), 2, axis=-1)
    xhat, r = layernorm_fwd(c[:, :S_i], LN_EPS)
    h = xhat * (1.0 + scale[:, None, :]) + shift[:, None, :]
    # backward: head
    gw = {"final": {}}
    dh, gw["final"]["w_out"], gw["final"]["b_out"] = linear_bwd(_patchify(dpred), h, f["w_out"])
    dx_img, dshift, dscale = modulate_bwd(dh, xhat, r, scale)
    dsv, gw["final"]["w_ada"], gw["final"]["b_ada"] = linear_bwd(np.concatenate([dshift, dscale], axis=-1), sv,
                                                                 f["w_ada"])
    dvec = dsv * silu_grad(vec)
    # the single blocks, last first, then the split of [img; txt]
    dc = np.zeros_like(c)
    dc[:, :S_i] = dx_img
    gw["single"] = [None] * len(w["single"])
    for i in reversed(range(len(w["single"]))):
        dc, dv, gw["single"][i] = single_bwd(ins_s[i], vec, cos, sin, w["single"][i], heads, dc,
                                             interleaved, gelu_tanh)
        dvec = dvec + dv
    d_img, d_txt = dc[:, :S_i], dc[:, S_i:]
    gw["double"] = [None] * len(w["double"])
    for i in reversed(range(len(w["double"]))):
        wi, wt = w["double"][i]
        d_img, d_txt, dv, gi, gt = double_block_backward(ins_d[i][0], ins_d[i][1], vec, cos, sin, wi, wt, heads,
                                                         d_img, d_txt, interleaved, gelu_tanh)
        gw["double"][i] = (gi, gt)
        dvec = dvec + dv
    # embeddings
    dpatch, dw_in, db_in = linear_bwd(d_img, patches, w["img_in"][0])
    gw["img_in"] = (dw_in, db_in)
    dtxt, dw_t, db_t = linear_bwd(d_txt, txt, w["txt_in"][0])
    gw["txt_in"] = (dw_t, db_t)
    # conditioning: both embedders, the guidance term, and t through the sinusoid
    dfeat, gw["time_in"] = _embedder_bwd(dvec, c_t, w["time_in"][0], w["time_in"][2])
    dy_in, gw["vector_in"] = _embedder_bwd(dvec, c_y, w["vector_in"][0], w["vector_in"][2])
    half = time_dim // 2
    dang = -dfeat[:, :half] * np.sin(ang) + dfeat[:, half:] * np.cos(ang)
    dt = (dang * freqs[None, :]).sum(axis=1) * time_factor
    ins = {"z_t": _unpatchify(dpatch, H, W), "txt": dtxt, "t": dt, "y": dy_in}
    if g is not None:
        gw["guidance_in"] = ((dvec * _f(g).reshape(-1, 1)).sum(axis=0), dvec.sum(axis=0))
        ins["g"] = (dvec * wg[None, :]).sum(axis=1)
    return ins, gw


def single_block_parallel_backward(x, vec, cos, sin, w, heads, dy, interleaved=True, gelu_tanh=False,
                                   ln_eps=LN_EPS, rms_eps=RMS_EPS):
    """Gradients of the parallel-branch single block of ``oracle.flux.single_block_parallel``
    (one LayerNorm-modulate h feeding QKV and fc1; y = x + gate ([o | u] [W_o | W_2]^T + b_o + b_2);
    three modulation chunks): (dx, dvec, grads).  The two branches' gradients meet at h."""
    m = _modulation(vec, w, 3)
    c = _stream_pre(x, m, w, heads, ln_eps, rms_eps)
    cs, sn = _f(cos)[:, None], _f(sin)[:, None]
    q = rope_rotate(c["qn"], cs, sn, interleaved)
    k = rope_rotate(c["kn"], cs, sn, interleaved)
    o, p = attention_fwd(q, k, c["v"])
    o = _merge(o)
    u_pre = linear_fwd(c["h1"], w["w_1"], w["b_1"])
    u = gelu_fwd(u_pre, gelu_tanh)
    branch = linear_fwd(o, w["w_o"], w["b_o"]) + linear_fwd(u, w["w_2"], w["b_2"])
    g = {}
    dx, dbranch, dgate = gated_residual_bwd(dy, m[2], branch)
    do, g["w_o"], g["b_o"] = linear_bwd(dbranch, o, w["w_o"])
    du, g["w_2"], g["b_2"] = linear_bwd(dbranch, u, w["w_2"])
    dh_mlp, g["w_1"], g["b_1"] = linear_bwd(du * gelu_grad(u_pre, gelu_tanh), c["h1"], w["w_1"])
    dq, dk, dv = attention_bwd(_heads(do, heads), q, k, c["v"], p)
    dq, dk = rope_bwd(dq, cs, sn, interleaved), rope_bwd(dk, cs, sn, interleaved)
    dq_raw, g["g_q"] = rmsnorm_bwd(dq, c["qxn"], c["qr"], w["g_q"])
    dk_raw, g["g_k"] = rmsnorm_bwd(dk, c["kxn"], c["kr"], w["g_k"])
    dqkv = np.concatenate([_merge(dq_raw), _merge(dk_raw), _merge(dv)], axis=-1)
    dh_att, g["w_qkv"], g["b_qkv"] = linear_bwd(dqkv, c["h1"], w["w_qkv"])
    dx_ln, dshift, dscale = modulate_bwd(dh_att + dh_mlp, c["xhat1"], c["r1"], m[1])
    dvec, g["w_mod"], g["b_mod"] = _modulation_bwd([dshift, dscale, dgate], vec, w)
    return dx + dx_ln, dvec, g
