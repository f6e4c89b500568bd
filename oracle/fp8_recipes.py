"""The other FP8 scaling recipes of the block linears, fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/flux.py``).

The "FP8 training for Flux models" page (§Configuration › FP8 model configuration) offers, beside
its default ``fp8_recipe: "delayed"`` (``oracle.e4m3``), the recipes ``"tensorwise"``,
``"blockwise"`` and ``"mxfp8"`` (and §Training configuration › Aggressive picks
``"tensorwise"``), and prints the names only.  The readings taken, every cast being E4M3 with
round-to-nearest-even and saturation (``oracle.e4m3``):

* **tensorwise** -- per-tensor *current* scaling: a tensor's scale comes from its own absolute
  maximum in the same call, ``s = 448 / amax / 2^margin`` (1 for an all-zero tensor), with no
  history; the GEMM runs on the casts and is divided by both scales, as in delayed scaling.
* **blockwise** -- current scaling per tile, one fp32 scale ``448 / amax(tile)`` each:
  activations in 1 x 128 tiles (one scale per row and per 128 consecutive elements of the
  contraction dimension K), weights [N, K] in 128 x 128 tiles; the last tile of a dimension
  that is not a multiple of 128 holds the remainder.  The GEMM sums, over the 128-wide slices
  of K, the slice products of the casts divided by the scales of the two tiles they came from.
* **mxfp8** -- the OCP Microscaling (MX) formats specification v1.0 with E4M3 elements
  (MXFP8 E4M3): 32 consecutive elements along K share one E8M0 scale
  ``X = 2^(floor(log2 amax) - 8)`` (8 is the exponent of E4M3's largest normal,
  448 = 1.75 * 2^8), its exponent clamped to the E8M0 range [-127, 127]; each element is stored
  as ``P = Q(V / X)`` and stands for ``X * P``.  Quotients up to 2^9 can exceed 448 and saturate
  to it (the reading taken for the conversion's overflow).  A block of zeros takes the smallest
  scale, 2^-127.  The GEMM is the product of the two operands' represented values, which in
  float64 is the sum over blocks of ``X_a X_w * sum(P_a P_w)``.

Each K-slice product is exact in float64 here; the device accumulates in fp32.
"""
from __future__ import annotations

import math

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_quantize

E4M3_EMAX = 8          # exponent of the largest E4M3 normal: 448 = 1.75 * 2^8
MX_BLOCK = 32          # elements per MX scaling block
E8M0_MIN_EXP, E8M0_MAX_EXP = -127, 127
BLOCKWISE_TILE = 128


def _amax(a) -> float:
    a = np.asarray(a, np.float64)
    return float(np.max(np.abs(a))) if a.size else 0.0


def _scale_of(amax: float, margin: int = 0) -> float:
    """448 / amax / 2^margin, 1 for a zero amax."""
    return E4M3_MAX / amax / (2.0 ** margin) if amax > 0 else 1.0


# --------------------------------------------------------------------------------- tensorwise
def tensorwise_scale(x, margin: int = 0) -> float:
    """Current per-tensor scale: 448 / amax(x) / 2^margin (1 for an all-zero tensor)."""
    return _scale_of(_amax(x), margin)


def tensorwise_linear(x, w, b, margin: int = 0):
    """y = Q(x s_x) Q(W s_w)^T / (s_x s_w) + b with both scales from the tensors themselves."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    sx, sw = tensorwise_scale(x, margin), tensorwise_scale(w, margin)
    y = e4m3_quantize(x * sx) @ e4m3_quantize(w * sw).T / (sx * sw)
    return y if b is None else y + np.asarray(b, np.float64)


class TensorwiseScaling:
    """The tensorwise recipe as the block oracle's ``fp8`` object (``oracle.flux.block_linear``
    calls ``linear``): every linear's input and weight are cast with scales from their own
    absolute maxima in the same call (``tensorwise_linear``).  ``act_cast``, if given, is applied
    to a linear's input first -- the value it holds as a stored activation tensor (e.g.
    ``oracle.flux.round_bf16``: the LayerNorm and GELU outputs are bf16 tensors that the recipe
    then scales and casts).  ``scales`` and ``amax`` record, per tensor name (``"<linear>.x"``,
    ``"<linear>.w"``), the scale used and the absolute maximum it came from."""

    def __init__(self, margin: int = 0, act_cast=None):
        self.margin = margin
        self.act_cast = act_cast
        self.scales = {}
        self.amax = {}

    def linear(self, name, x, w, b):
        x = np.asarray(x, np.float64)
        if self.act_cast is not None:
            x = np.asarray(self.act_cast(x), np.float64)
        w = np.asarray(w, np.float64)
        for key, t in ((name + ".x", x), (name + ".w", w)):
            self.amax[key] = _amax(t)
            self.scales[key] = _scale_of(self.amax[key], self.margin)
        return tensorwise_linear(x, w, b, self.margin)


# --------------------------------------------------------------------------------- blockwise
def _slices(n: int, tile: int):
    return [slice(j, min(j + tile, n)) for j in range(0, n, tile)]


def blockwise_quantize_act(x, tile: int = BLOCKWISE_TILE):
    """Casts of x [..., K] in 1 x tile tiles: (Q(x s) per tile, scales [..., ceil(K / tile)])."""
    x = np.asarray(x, np.float64)
    ks = _slices(x.shape[-1], tile)
    q = np.empty_like(x)
    s = np.empty(x.shape[:-1] + (len(ks),))
    for j, sl in enumerate(ks):
        part = x[..., sl]
        amax = np.max(np.abs(part), axis=-1)
        sj = np.where(amax > 0, E4M3_MAX / np.where(amax > 0, amax, 1.0), 1.0)
        s[..., j] = sj
        q[..., sl] = e4m3_quantize(part * sj[..., None])
    return q, s


def blockwise_quantize_weight(w, tile: int = BLOCKWISE_TILE):
    """Casts of W [N, K] in tile x tile tiles: (Q(W s) per tile, scales [ceil(N/tile), ceil(K/tile)])."""
    w = np.asarray(w, np.float64)
    ns, ks = _slices(w.shape[0], tile), _slices(w.shape[1], tile)
    q = np.empty_like(w)
    s = np.empty((len(ns), len(ks)))
    for i, si in enumerate(ns):
        for j, sj in enumerate(ks):
            s[i, j] = _scale_of(_amax(w[si, sj]))
            q[si, sj] = e4m3_quantize(w[si, sj] * s[i, j])
    return q, s


class BlockwiseScaling:
    """The blockwise recipe as the block oracle's ``fp8`` object (``oracle.flux.block_linear`` calls
    ``linear``): every linear is ``blockwise_linear`` of its input and weight, with no state.
    ``act_cast``, if given, is applied to a linear's input first (the value it holds as a stored
    activation tensor, as for ``TensorwiseScaling``)."""

    def __init__(self, act_cast=None, tile: int = None):
        self.act_cast = act_cast
        self.tile = BLOCKWISE_TILE if tile is None else tile

    def linear(self, name, x, w, b):
        x = np.asarray(x, np.float64)
        if self.act_cast is not None:
            x = np.asarray(self.act_cast(x), np.float64)
        return blockwise_linear(x, w, b, self.tile)


def blockwise_linear(x, w, b, tile: int = BLOCKWISE_TILE):
    """y = sum over K slices j of Q_j(x) Q_j(W)^T / (s_x[row, j] s_w[tile row, j]) + b."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    qx, sx = blockwise_quantize_act(x, tile)
    qw, sw = blockwise_quantize_weight(w, tile)
    w_tile_row = np.arange(w.shape[0]) // tile          # the weight tile row of each output
    y = np.zeros(x.shape[:-1] + (w.shape[0],))
    for j, sl in enumerate(_slices(x.shape[-1], tile)):
        part = qx[..., sl] @ qw[:, sl].T
        y += part / (sx[..., j][..., None] * sw[w_tile_row, j])
    return y if b is None else y + np.asarray(b, np.float64)


# --------------------------------------------------------------------------------- MXFP8
def e8m0_decode(code: int) -> float:
    """Value of an E8M0 scale code: 2^(code - 127); 0xFF is NaN."""
    code = int(code) & 0xFF
    return float("nan") if code == 0xFF else math.ldexp(1.0, code - 127)


def mx_shared_exponent(amax):
    """floor(log2 amax) - 8, clamped to [-127, 127]; -127 for amax 0."""
    amax = np.asarray(amax, np.float64)
    pos = amax > 0
    # amax = m 2^k with m in [0.5, 1): floor(log2 amax) = k - 1, exactly (no log rounding)
    _, k = np.frexp(np.where(pos, amax, 1.0))
    e = np.where(pos, k.astype(np.int64) - 1 - E4M3_EMAX, E8M0_MIN_EXP)
    return np.clip(e, E8M0_MIN_EXP, E8M0_MAX_EXP).astype(np.int64)


def mxfp8_quantize(x, block: int = MX_BLOCK):
    """MXFP8 E4M3 casts of x [..., K] in blocks of ``block`` along K.

    Returns (P, e): the E4M3 element values P [..., K] (float64) and the shared exponents
    e [..., ceil(K / block)] (the E8M0 codes are e + 127).  The represented value is P * 2^e.
    """
    x = np.asarray(x, np.float64)
    ks = _slices(x.shape[-1], block)
    p = np.empty_like(x)
    e = np.empty(x.shape[:-1] + (len(ks),), np.int64)
    for j, sl in enumerate(ks):
        part = x[..., sl]
        ej = mx_shared_exponent(np.max(np.abs(part), axis=-1))
        e[..., j] = ej
        p[..., sl] = e4m3_quantize(np.ldexp(part, -ej[..., None]))
    return p, e


def mxfp8_dequantize(p, e, block: int = MX_BLOCK):
    """The values P * 2^e that an MXFP8 tensor stands for."""
    p = np.asarray(p, np.float64)
    out = np.empty_like(p)
    for j, sl in enumerate(_slices(p.shape[-1], block)):
        out[..., sl] = np.ldexp(p[..., sl], np.asarray(e)[..., j][..., None])
    return out


def mxfp8_linear(x, w, b, block: int = MX_BLOCK):
    """y = X_x W_x^T + b with X_x, W_x the values the two MXFP8 tensors stand for (P * 2^e), that
    is the sum over K blocks j of 2^(e_x[row, j] + e_w[n, j]) * P_x,j P_w,j^T; every product is
    exact in float64, so one product of the represented values gives the same sums."""
    px, ex = mxfp8_quantize(x, block)
    pw, ew = mxfp8_quantize(w, block)
    y = mxfp8_dequantize(px, ex, block) @ mxfp8_dequantize(pw, ew, block).T
    return y if b is None else y + np.asarray(b, np.float64)


class MxScaling:
    """The MXFP8 recipe as the block oracle's ``fp8`` object (``oracle.flux.block_linear`` calls
    ``linear``): every linear is ``mxfp8_linear`` of its input and weight, with no state.
    ``act_cast``, if given, is applied to a linear's input first (the value it holds as a stored
    activation tensor, as for ``TensorwiseScaling``)."""

    def __init__(self, act_cast=None, block: int = None):
        self.act_cast = act_cast
        self.block = MX_BLOCK if block is None else block

    def linear(self, name, x, w, b):
        x = np.asarray(x, np.float64)
        if self.act_cast is not None:
            x = np.asarray(self.act_cast(x), np.float64)
        return mxfp8_linear(x, w, b, self.block)
