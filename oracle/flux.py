"""fp64 CPU oracle of the Flux MMDiT block forward and the rectified-flow loss.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA path.  Every function is the plain definition, written in numpy
float64, in the order the pages give the steps.

Page titles used in citations:
  * "Flux model API reference" (the API page),
  * "Flux architecture deep dive" (the architecture page),
  * "FP8 training for Flux models" (the FP8 page).

Readings taken where the pages are silent or disagree (each is listed in the
design notes of the repository as well):
  * RoPE pairs are interleaved ``(x[2j], x[2j+1])`` by default (API page,
    §Configuration table, ``rotary_interleaved=True``); the half-split pairing
    ``(x[j], x[j+d/2])`` printed in the architecture page (§3D RoPE
    mathematics) is available behind ``interleaved=False``.
  * Frequency index ``i`` runs over ``0 <= i < d_axis/2`` (the printed range
    ``i = 0..d_axis/2`` has one index too many for a ``d_axis``-wide axis).
  * QK-RMSNorm is applied per head over ``head_dim`` on q and k, after the QKV
    bias and before RoPE, with a learned gain and eps 1e-6.
  * LayerNorm has no affine parameters (the modulation supplies scale/shift),
    biased variance, eps 1e-6 (API page, §Configuration, layernorm_epsilon).
  * Every linear has a bias.  The attention output projection is included.
  * GELU is the exact erf form; the tanh form is behind ``gelu_tanh=True``.  Both forms are
    pinned to textbook values; which of them the pages mean is a reading that no outside
    value settles (parity unpinned for that choice only).
  * Attention scale is 1/sqrt(head_dim), no mask.
  * The single block runs attention then MLP in sequence with six modulation
    chunks, over the whole concatenated sequence, and returns every row.  The
    parallel-branch form (``single_block_parallel``) is the one the API page's
    parameter-count table fits; ``flux_forward(..., single_parallel=True)`` uses it.
  * The output head takes (shift, scale) from a SiLU + linear of ``vec``.
  * Loss is the mean over all elements.
  * Conditioning: the timestep enters as tau = 1000 t (the TimeStepEmbedder's input range),
    encoded as [cos(tau f_i), sin(tau f_i)] with f_i = 10000^(-i/128), i < 128; both
    embedders are Linear, SiLU, Linear; the optional guidance term is a Linear of the scalar.
  * Precision: by default every step runs in float64.  ``mm_cast=round_bf16`` evaluates the
    method at the precision the pages fix for training, bf16 autocast (architecture page,
    §Performance optimizations › 5. Mixed precision; API page, §Optimization tips): the
    operands of every linear layer and the attention's inputs q, k, v are rounded to bf16;
    everything else (including the softmax weights inside the fused attention) stays float64.
  * FP8 (``fp8=oracle.e4m3.DelayedScaling(...)``, FP8 page §Configuration): the four linears
    of each stream (QKV, attention output projection, fc1, fc2) cast input and weight to E4M3
    with per-tensor scales; the modulation, embeddings, head and attention do not.  The
    projection reads the attention output in the activation type (``mm_cast``); the LayerNorm
    and GELU results are cast directly from the arithmetic that makes them (a fused cast).
"""
from __future__ import annotations

import math

import numpy as np

LN_EPS = 1e-6
RMS_EPS = 1e-6
AXES_DIM = (16, 56, 56)
THETA = 10000.0

F64 = np.float64


def _f64(x):
    return np.asarray(x, dtype=F64)


def round_bf16(x):
    """Nearest bfloat16 value (8 significant bits, exponent range of float32, ties to even).

    bfloat16 keeps the sign and 8-bit exponent of IEEE binary32 and 7 stored fraction bits, so
    a normal value with leading bit 2^e is rounded to a multiple of 2^(e-7); below the float32
    normal range the quantum stays 2^-133.  Computed directly from float64 (no double rounding).
    """
    x = _f64(x)
    mag = np.abs(x)
    _, E = np.frexp(np.where(mag > 0, mag, 1.0))  # mag = m * 2^E, m in [0.5, 1)
    lead = np.maximum(E - 1, -126)
    quantum = np.ldexp(1.0, lead - 7)
    return np.where(mag > 0, np.rint(x / quantum) * quantum, x)


def _cast(x, mm_cast):
    return _f64(x) if mm_cast is None else mm_cast(_f64(x))


# ----------------------------------------------------------------------------- 3D RoPE
def rope_angles(ids, axes_dim=AXES_DIM, theta=THETA):
    """Per-token rotation angles, ``[..., sum(axes_dim)/2]``.

    Architecture page, §Model components › 2. Position embeddings (3D RoPE)
    and §Mathematical formulation › 3D RoPE mathematics: for axis ``a`` of
    width ``d_a`` the frequencies are ``theta^(-2i/d_a)`` for ``i < d_a/2``
    and the angle is ``pid[a] * theta^(-2i/d_a)``; the three axes' angles are
    concatenated in axis order.
    """
    ids = _f64(ids)
    parts = []
    for a, d_a in enumerate(axes_dim):
        i = np.arange(d_a // 2, dtype=F64)
        inv_freq = float(theta) ** (-2.0 * i / d_a)
        parts.append(ids[..., a:a + 1] * inv_freq)
    return np.concatenate(parts, axis=-1)


def rope_cos_sin(ids, axes_dim=AXES_DIM, theta=THETA):
    ang = rope_angles(ids, axes_dim, theta)
    return np.cos(ang), np.sin(ang)


def apply_rope(x, cos, sin, interleaved=True):
    """Rotate pairs of ``x[..., d]`` by the angles whose cos/sin are ``[..., d/2]``.

    Interleaved pairs ``(x[2j], x[2j+1])`` (API page, §Configuration,
    ``rotary_interleaved``); half-split pairs ``(x[j], x[j+d/2])``
    (architecture page, §3D RoPE mathematics, "RoPE Rotation").  Each pair
    (a, b) becomes (a cos - b sin, a sin + b cos).
    """
    x = _f64(x)
    d = x.shape[-1]
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : d // 2], x[..., d // 2:]
    ra = a * cos - b * sin
    rb = a * sin + b * cos
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


# ----------------------------------------------------------------------------- norms, activations
def layernorm(x, eps=LN_EPS):
    """LayerNorm over the last axis, biased variance, no affine."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def rmsnorm(x, g, eps=RMS_EPS):
    """API page, §Normalization › RMSNorm: x / sqrt(mean(x^2) + eps) * g."""
    x = _f64(x)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * _f64(g)


def silu(x):
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


_erf = np.vectorize(math.erf, otypes=[F64])


def gelu(x, tanh=False):
    """GELU: x * Phi(x) with the exact normal CDF; or the tanh approximation."""
    x = _f64(x)
    if tanh:
        return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def linear(x, w, b=None, mm_cast=None):
    """y = x W^T + b with W stored [out, in]; ``mm_cast`` rounds the two matmul operands."""
    y = _cast(x, mm_cast) @ _cast(w, mm_cast).T
    return y if b is None else y + _f64(b)


def block_linear(name, x, w, b, mm_cast=None, fp8=None):
    """One of a block's four linears (QKV, attention output projection, fc1, fc2).

    With ``fp8`` (an ``oracle.e4m3.DelayedScaling``) the input and weight are
    cast to E4M3 with their per-tensor scales, as the FP8 page configures the
    linears (§Configuration › FP8 model configuration); the modulation,
    embedding and head linears and the attention are never FP8.  Otherwise
    this is ``linear``.
    """
    if fp8 is None:
        return linear(x, w, b, mm_cast)
    return fp8.linear(name, x, w, b)


# ----------------------------------------------------------------------------- AdaLN
def modulation(vec, w_mod, b_mod, n_chunks=6, mm_cast=None):
    """AdaLN.forward: Linear(SiLU(vec)) split into chunks along the feature axis.

    API page, §Normalization › AdaLN (six chunks named shift, scale, gate,
    shift_mlp, scale_mlp, gate_mlp, in that order); architecture page,
    §Implementation details › Adaptive layer normalization.
    """
    m = linear(silu(vec), w_mod, b_mod, mm_cast)  # [B, n*D]
    return np.split(m, n_chunks, axis=-1)


def modulate(x, shift, scale, eps=LN_EPS):
    """AdaLN.modulate: LayerNorm(x) * (1 + scale) + shift, shift/scale per batch row."""
    return layernorm(x, eps) * (1.0 + _f64(scale)[:, None, :]) + _f64(shift)[:, None, :]


def gated_residual(x, gate, y):
    """AdaLN.scale_add: x + gate * y, gate per batch row."""
    return _f64(x) + _f64(gate)[:, None, :] * _f64(y)


# ----------------------------------------------------------------------------- attention
def attention(q, k, v, mm_cast=None):
    """softmax(q k^T / sqrt(d)) v over the key axis, no mask.  q,k,v: [..., S, d].

    Architecture page, §Implementation details › Attention implementation
    (no mask) and › Joint Attention Trick (one call over the joint sequence).
    ``mm_cast`` rounds the attention's inputs q, k, v.  The softmax weights are kept
    exact: the pages run attention as one fused kernel (architecture page, §Performance
    optimizations › 2. Flash attention), whose inputs are the autocast operands; its
    internal probabilities are not.
    """
    q, k, v = _cast(q, mm_cast), _cast(k, mm_cast), _cast(v, mm_cast)
    d = q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(d)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v


# ----------------------------------------------------------------------------- block pieces
def _heads(x, heads):
    """[B, S, H*d] -> [B, H, S, d] (column h*d + j is head h, element j)."""
    B, S, HD = x.shape
    return x.reshape(B, S, heads, HD // heads).transpose(0, 2, 1, 3)


def _merge(x):
    """[B, H, S, d] -> [B, S, H*d]."""
    B, H, S, d = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B, S, H * d)


def qkv_heads(x, shift, scale, w, heads, ln_eps=LN_EPS, rms_eps=RMS_EPS, mm_cast=None,
              fp8=None, name=""):
    """Attention-branch pre-norm and projection of one stream, before RoPE.

    Architecture page, §3. MMDiT layer (double block), steps 1-2:
    AdaLN-modulated LayerNorm, then the QKV linear (with bias); then per-head
    RMSNorm of q and k.  Returns q, k, v as [B, H, S, d].
    """
    h = modulate(x, shift, scale, ln_eps)
    qkv = block_linear(name + ".qkv", h, w["w_qkv"], w["b_qkv"], mm_cast, fp8)
    q, k, v = np.split(qkv, 3, axis=-1)
    q = rmsnorm(_heads(q, heads), w["g_q"], rms_eps)
    k = rmsnorm(_heads(k, heads), w["g_k"], rms_eps)
    return q, k, _heads(v, heads)


def mlp_branch(x, shift, scale, w, gelu_tanh=False, ln_eps=LN_EPS, mm_cast=None, fp8=None,
               name=""):
    """Architecture page, §3. MMDiT layer, step 4: AdaLN -> Linear -> GELU -> Linear."""
    h = modulate(x, shift, scale, ln_eps)
    u = gelu(block_linear(name + ".fc1", h, w["w_1"], w["b_1"], mm_cast, fp8), gelu_tanh)
    return block_linear(name + ".fc2", u, w["w_2"], w["b_2"], mm_cast, fp8)


def out_proj(o, w, name="", mm_cast=None, fp8=None):
    """Attention output projection of one stream.  The attention returns its output in the
    activation type (``mm_cast``), and that tensor is what the projection (or its E4M3 cast)
    reads."""
    return block_linear(name + ".o", _cast(o, mm_cast), w["w_o"], w["b_o"], mm_cast, fp8)


def double_block(x_img, x_txt, vec, cos, sin, w_img, w_txt, heads,
                 interleaved=True, gelu_tanh=False, ln_eps=LN_EPS, rms_eps=RMS_EPS, mm_cast=None,
                 fp8=None):
    """Double-stream (joint) block forward.

    Architecture page, §Model components › 3. MMDiT layer (double block);
    API page, §Layer specifications › MMDiTLayer.  ``cos``/``sin`` are
    ``[B, S_img + S_txt, d/2]`` in the joint order [image; text].  ``fp8``
    (``oracle.e4m3.DelayedScaling``) makes the four linears of each stream
    E4M3, with tensors named ``img.*`` and ``txt.*``.
    Returns (y_img, y_txt).
    """
    c = mm_cast
    S_i = np.shape(x_img)[1]
    mi = modulation(vec, w_img["w_mod"], w_img["b_mod"], mm_cast=c)
    mt = modulation(vec, w_txt["w_mod"], w_txt["b_mod"], mm_cast=c)
    qi, ki, vi = qkv_heads(x_img, mi[0], mi[1], w_img, heads, ln_eps, rms_eps, c, fp8, "img")
    qt, kt, vt = qkv_heads(x_txt, mt[0], mt[1], w_txt, heads, ln_eps, rms_eps, c, fp8, "txt")
    q = np.concatenate([qi, qt], axis=2)
    k = np.concatenate([ki, kt], axis=2)
    v = np.concatenate([vi, vt], axis=2)
    cs, sn = _f64(cos)[:, None], _f64(sin)[:, None]
    q = apply_rope(q, cs, sn, interleaved)
    k = apply_rope(k, cs, sn, interleaved)
    o = _merge(attention(q, k, v, c))
    o_img, o_txt = o[:, :S_i], o[:, S_i:]
    x_img = gated_residual(x_img, mi[2], out_proj(o_img, w_img, "img", c, fp8))
    x_txt = gated_residual(x_txt, mt[2], out_proj(o_txt, w_txt, "txt", c, fp8))
    x_img = gated_residual(x_img, mi[5],
                           mlp_branch(x_img, mi[3], mi[4], w_img, gelu_tanh, ln_eps, c, fp8, "img"))
    x_txt = gated_residual(x_txt, mt[5],
                           mlp_branch(x_txt, mt[3], mt[4], w_txt, gelu_tanh, ln_eps, c, fp8, "txt"))
    return x_img, x_txt


def single_block(x, vec, cos, sin, w, heads, interleaved=True, gelu_tanh=False,
                 ln_eps=LN_EPS, rms_eps=RMS_EPS, mm_cast=None, fp8=None):
    """Single-stream block forward over the concatenated sequence ``x = [img; txt]``.

    Architecture page, §Model components › 4. Flux single block: AdaLN,
    QKV, attention, gated residual, AdaLN, MLP, gated residual, all with one
    weight set.  Returns all rows (the caller keeps the image rows after the
    last single block).  ``fp8`` names its tensors ``single.*``.
    """
    c = mm_cast
    m = modulation(vec, w["w_mod"], w["b_mod"], mm_cast=c)
    q, k, v = qkv_heads(x, m[0], m[1], w, heads, ln_eps, rms_eps, c, fp8, "single")
    cs, sn = _f64(cos)[:, None], _f64(sin)[:, None]
    q = apply_rope(q, cs, sn, interleaved)
    k = apply_rope(k, cs, sn, interleaved)
    o = _merge(attention(q, k, v, c))
    x = gated_residual(x, m[2], out_proj(o, w, "single", c, fp8))
    return gated_residual(x, m[5], mlp_branch(x, m[3], m[4], w, gelu_tanh, ln_eps, c, fp8, "single"))


# ----------------------------------------------------------------------------- row-sampled blocks
def _rows_after_attention(x_rows, o_rows, m, w, gelu_tanh, ln_eps, mm_cast, fp8=None, name=""):
    x1 = gated_residual(x_rows, m[2], out_proj(o_rows, w, name, mm_cast, fp8))
    return gated_residual(x1, m[5], mlp_branch(x1, m[3], m[4], w, gelu_tanh, ln_eps, mm_cast, fp8, name))


def _attend_rows(q_rows, k, v, c_rows, s_rows, c_all, s_all, interleaved, mm_cast):
    q = apply_rope(q_rows, c_rows[:, None], s_rows[:, None], interleaved)
    kk = apply_rope(k, c_all[:, None], s_all[:, None], interleaved)
    return _merge(attention(q, kk, v, mm_cast))


def double_block_rows(x_img, x_txt, vec, cos, sin, w_img, w_txt, heads, rows_img, rows_txt,
                      interleaved=True, gelu_tanh=False, ln_eps=LN_EPS, rms_eps=RMS_EPS,
                      mm_cast=None, fp8=None):
    """The double block's output at selected rows only (same batch rows for every sample).

    Keys and values need every token; queries, attention, the output
    projection and the MLP are row-wise, so computing them for a subset of
    rows gives those rows of ``double_block`` exactly.  With ``fp8`` the
    scales must be given: the amax this records for the tensors after the
    attention covers the selected rows only.
    """
    c = mm_cast
    S_i = np.shape(x_img)[1]
    mi = modulation(vec, w_img["w_mod"], w_img["b_mod"], mm_cast=c)
    mt = modulation(vec, w_txt["w_mod"], w_txt["b_mod"], mm_cast=c)
    # keys/values for every token (queries are recomputed only for the chosen rows)
    _, ki, vi = qkv_heads(x_img, mi[0], mi[1], w_img, heads, ln_eps, rms_eps, c, fp8, "img")
    _, kt, vt = qkv_heads(x_txt, mt[0], mt[1], w_txt, heads, ln_eps, rms_eps, c, fp8, "txt")
    k = np.concatenate([ki, kt], axis=2)
    v = np.concatenate([vi, vt], axis=2)
    cos, sin = _f64(cos), _f64(sin)
    rows_img = np.asarray(rows_img)
    rows_txt = np.asarray(rows_txt)
    qi, _, _ = qkv_heads(_f64(x_img)[:, rows_img], mi[0], mi[1], w_img, heads, ln_eps, rms_eps, c,
                         fp8, "img")
    qt, _, _ = qkv_heads(_f64(x_txt)[:, rows_txt], mt[0], mt[1], w_txt, heads, ln_eps, rms_eps, c,
                         fp8, "txt")
    jr_i, jr_t = rows_img, S_i + rows_txt
    oi = _attend_rows(qi, k, v, cos[:, jr_i], sin[:, jr_i], cos, sin, interleaved, c)
    ot = _attend_rows(qt, k, v, cos[:, jr_t], sin[:, jr_t], cos, sin, interleaved, c)
    yi = _rows_after_attention(_f64(x_img)[:, rows_img], oi, mi, w_img, gelu_tanh, ln_eps, c, fp8,
                               "img")
    yt = _rows_after_attention(_f64(x_txt)[:, rows_txt], ot, mt, w_txt, gelu_tanh, ln_eps, c, fp8,
                               "txt")
    return yi, yt


def single_block_rows(x, vec, cos, sin, w, heads, rows, interleaved=True, gelu_tanh=False,
                      ln_eps=LN_EPS, rms_eps=RMS_EPS, mm_cast=None, fp8=None):
    """The single block's output at selected rows only (see ``double_block_rows``)."""
    c = mm_cast
    m = modulation(vec, w["w_mod"], w["b_mod"], mm_cast=c)
    _, k, v = qkv_heads(x, m[0], m[1], w, heads, ln_eps, rms_eps, c, fp8, "single")
    rows = np.asarray(rows)
    q, _, _ = qkv_heads(_f64(x)[:, rows], m[0], m[1], w, heads, ln_eps, rms_eps, c, fp8, "single")
    cos, sin = _f64(cos), _f64(sin)
    o = _attend_rows(q, k, v, cos[:, rows], sin[:, rows], cos, sin, interleaved, c)
    return _rows_after_attention(_f64(x)[:, rows], o, m, w, gelu_tanh, ln_eps, c, fp8, "single")


# ----------------------------------------------------------------------------- parallel single block
def _parallel_branches(x_rows, o_rows, shift, scale, gate, w, gelu_tanh, ln_eps, mm_cast):
    """x + gate ([o | m] [W_o | W_2]^T + b_o + b_2), m = GELU(h W_1^T + b_1), h the one
    LayerNorm-modulate both branches share: the fused output linear on the concatenation."""
    h = modulate(x_rows, shift, scale, ln_eps)
    m = gelu(linear(h, w["w_1"], w["b_1"], mm_cast), gelu_tanh)
    om = np.concatenate([_cast(o_rows, mm_cast), m], axis=-1)
    w_cat = np.concatenate([_f64(w["w_o"]), _f64(w["w_2"])], axis=1)
    return gated_residual(x_rows, gate, linear(om, w_cat, _f64(w["b_o"]) + _f64(w["b_2"]), mm_cast))


def single_block_parallel(x, vec, cos, sin, w, heads, interleaved=True, gelu_tanh=False,
                          ln_eps=LN_EPS, rms_eps=RMS_EPS, mm_cast=None, rows=None):
    """Single-stream block with parallel branches (the whole-model row's shape option: the
    attention and the MLP fed from one LayerNorm, the QKV and fc1 linears reading the same
    modulated input, and one gated residual through the output linear of the concatenation).

    Modulation: three chunks (shift, scale, gate) of SiLU(vec) W_mod^T + b_mod, W_mod [3D, D].
    The output linear is [W_o | W_2] [D, D + F] with bias b_o + b_2 (the stream's output
    projection and fc2 weights side by side).  ``rows``: compute only those rows of the output
    (keys and values still come from every token; everything after the attention is row-wise).
    """
    c = mm_cast
    shift, scale, gate = modulation(vec, w["w_mod"], w["b_mod"], 3, mm_cast=c)
    q, k, v = qkv_heads(x, shift, scale, w, heads, ln_eps, rms_eps, c)
    cos, sin = _f64(cos), _f64(sin)
    if rows is None:
        rows = np.arange(np.shape(x)[1])
    else:
        rows = np.asarray(rows)
        q, _, _ = qkv_heads(_f64(x)[:, rows], shift, scale, w, heads, ln_eps, rms_eps, c)
    o = _attend_rows(q, k, v, cos[:, rows], sin[:, rows], cos, sin, interleaved, c)
    return _parallel_branches(_f64(x)[:, rows], o, shift, scale, gate, w, gelu_tanh, ln_eps, c)


# ----------------------------------------------------------------------------- embeddings and head
def patchify(z):
    """[B, C, H, W] -> [B, H*W, C] with patch size 1 (architecture page, §Memory layout)."""
    z = _f64(z)
    B, C, H, W = z.shape
    return z.reshape(B, C, H * W).transpose(0, 2, 1)


def unpatchify(tokens, H, W):
    """[B, H*W, C] -> [B, C, H, W]."""
    t = _f64(tokens)
    B, S, C = t.shape
    return t.transpose(0, 2, 1).reshape(B, C, H, W)


def img_in(z, w, b, mm_cast=None):
    """Image path: patchify, then Linear C -> D (architecture page, §1. Input embeddings)."""
    return linear(patchify(z), w, b, mm_cast)


def txt_in(txt, w, b, mm_cast=None):
    """Text path: Linear ctx_dim -> D (architecture page, §1. Input embeddings)."""
    return linear(txt, w, b, mm_cast)


def final_layer(x_img, vec, w_ada, b_ada, w_out, b_out, H, W, ln_eps=LN_EPS, mm_cast=None):
    """Output head: AdaLNContinuous(vec), Linear D -> C, reshape to [B, C, H, W].

    Architecture page, §Model components › 5. Output processing; API page,
    §Normalization › AdaLNContinuous.  (shift, scale) = SiLU(vec) W^T + b.
    """
    shift, scale = modulation(vec, w_ada, b_ada, 2, mm_cast)
    y = linear(modulate(x_img, shift, scale, ln_eps), w_out, b_out, mm_cast)
    return unpatchify(y, H, W)


# ----------------------------------------------------------------------------- conditioning
TIME_DIM = 256
TIME_FACTOR = 1000.0
TIME_MAX_PERIOD = 10000.0


def timestep_features(t, dim=TIME_DIM, time_factor=TIME_FACTOR, max_period=TIME_MAX_PERIOD):
    """Sinusoidal encoding of the timestep: t in [0, 1] -> [B, 256] (architecture page,
    §Model components › 1. Input embeddings › Conditioning; API page, §Components API ›
    Embeddings › TimeStepEmbedder, whose inputs lie in [0, 1000]).

    Reading (the pages print no formula): tau = 1000 t; frequencies f_i = max_period^(-i/half)
    for i < half = dim/2; features [cos(tau f_0 .. f_half-1), sin(tau f_0 .. f_half-1)].
    """
    tau = time_factor * _f64(t).reshape(-1, 1)
    half = dim // 2
    freqs = max_period ** (-np.arange(half, dtype=F64) / half)
    ang = tau * freqs[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def mlp_embedder(x, w1, b1, w2, b2, mm_cast=None):
    """Two-layer MLP: Linear(in -> D), SiLU, Linear(D -> D) (API page, §Components API ›
    Embeddings › MLPEmbedder; the TimeStepEmbedder's MLP after the sinusoidal encoding).
    Reading: SiLU between the two layers (the activation of the conditioning path)."""
    return linear(silu(linear(x, w1, b1, mm_cast)), w2, b2, mm_cast)


def guidance_embed(g, w, b):
    """Guidance scale g -> Linear -> [B, D] (architecture page, §Conditioning, the optional
    guidance term).  Reading: a Linear of the scalar, g w + b with w, b of length D."""
    return _f64(g).reshape(-1, 1) * _f64(w)[None, :] + _f64(b)[None, :]


def conditioning_vec(t, y, w, g=None, mm_cast=None):
    """vec = timestep_emb + clip_pooled_emb [+ guidance_emb] (architecture page,
    §Conditioning, Combined Conditioning Vector).  ``w["time_in"]`` and ``w["vector_in"]``
    hold (w1, b1, w2, b2); ``w["guidance_in"]`` holds (w, b)."""
    vec = mlp_embedder(timestep_features(t), *w["time_in"], mm_cast=mm_cast)
    vec = vec + mlp_embedder(y, *w["vector_in"], mm_cast=mm_cast)
    if g is not None:
        vec = vec + guidance_embed(g, *w["guidance_in"])
    return vec


def flux_forward(z_t, txt, t, y, ids, w, heads, g=None, interleaved=True, gelu_tanh=False,
                 mm_cast=None, store=None, axes_dim=AXES_DIM, single_parallel=False):
    """The whole model (architecture page, §Data flow › Complete forward pass; §Model variants:
    19 double and 38 single blocks for Flux 12B, 1 and 1 for Flux 535M).

    conditioning vector; img_in(z_t), txt_in(txt); the double blocks in order; the single
    blocks over the concatenation [img; txt]; the output head on the image rows of the last
    block.  ``store`` (e.g. ``round_bf16``) is applied to every tensor the model hands from one
    step to the next (vec, the embedded tokens, each block's outputs), the values an
    implementation that stores them in the activation type holds.  ``single_parallel``: the single
    blocks are the parallel-branch form (``single_block_parallel``), the form whose parameter
    count matches the API reference's parameter-count table.
    """
    keep = store if store is not None else _f64
    single = single_block_parallel if single_parallel else single_block
    B, C, H, W = np.shape(z_t)
    vec = keep(conditioning_vec(t, y, w, g, mm_cast))
    x_img = keep(img_in(z_t, w["img_in"][0], w["img_in"][1], mm_cast))
    x_txt = keep(txt_in(txt, w["txt_in"][0], w["txt_in"][1], mm_cast))
    cos, sin = rope_cos_sin(ids, axes_dim)
    for wi, wt in w["double"]:
        x_img, x_txt = double_block(x_img, x_txt, vec, cos, sin, wi, wt, heads, interleaved,
                                    gelu_tanh, mm_cast=mm_cast)
        x_img, x_txt = keep(x_img), keep(x_txt)
    c = np.concatenate([x_img, x_txt], axis=1)
    for ws in w["single"]:
        c = keep(single(c, vec, cos, sin, ws, heads, interleaved, gelu_tanh, mm_cast=mm_cast))
    f = w["final"]
    return final_layer(c[:, : H * W], vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], H, W,
                       mm_cast=mm_cast)


# ----------------------------------------------------------------------------- rectified flow
def flow_match_noise(z0, z1, t):
    """z_t = (1 - t) z0 + t z1, t per sample (architecture page, §Flow matching objective;
    API page, §Noise application › apply_flow_matching_noise)."""
    z0, z1 = _f64(z0), _f64(z1)
    tt = _f64(t).reshape((-1,) + (1,) * (z0.ndim - 1))
    return (1.0 - tt) * z0 + tt * z1


def flow_match_target(z0, z1):
    """Velocity target v* = z1 - z0 (architecture page, §Flow matching objective)."""
    return _f64(z1) - _f64(z0)


def flow_match_loss(pred, z0, z1):
    """MSE(pred, z1 - z0), mean over all elements (API page, §Loss computation ›
    compute_flow_matching_loss)."""
    diff = _f64(pred) - flow_match_target(z0, z1)
    return float(np.mean(diff * diff))


# ----------------------------------------------------------------------------- sampling
def cfg_combine(v_cond, v_uncond, w):
    """Classifier-free guidance: v_uncond + w (v_cond - v_uncond) (architecture page,
    §Mathematical formulation › Classifier-free guidance)."""
    v_cond, v_uncond = _f64(v_cond), _f64(v_uncond)
    return v_uncond + float(w) * (v_cond - v_uncond)


def euler_step(z, v, dt):
    """One Euler step of the flow ODE towards t = 0: z_{t - dt} = z_t - dt v_t (architecture
    page, §Sampling (inference) › Euler integration)."""
    return _f64(z) - float(dt) * _f64(v)
