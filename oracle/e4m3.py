"""FP8 E4M3 quantisation and delayed per-tensor scaling, fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/flux.py``).

E4M3 as defined in "FP8 Formats for Deep Learning" (Micikevicius et al.,
2022), the format the "FP8 training for Flux models" page selects
(§Configuration › FP8 model configuration, ``fp8: "e4m3"``): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits, no infinities, the single
NaN pattern S.1111.111, largest finite magnitude 1.75 * 2^8 = 448, smallest
subnormal 2^-9.  Conversion rounds to nearest, ties to even, and saturates
to +-448.

Delayed scaling (same page, same section: margin 0, amax history 1024,
``most_recent``): the scale applied to a tensor is ``448 / amax / 2^margin``
where ``amax`` is the most recent recorded absolute maximum; with an empty
history the scale is 1.  The scaled tensor is quantised, the GEMM runs on the
quantised operands and its result is divided by the product of the scales.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of an 8-bit E4M3 code from the format definition (NaN for S.1111.111)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def _finite_table():
    """Non-negative finite codes 0x00..0x7E with their values (ascending)."""
    codes = np.arange(0x7F)
    vals = np.array([e4m3_decode(c) for c in codes], dtype=np.float64)
    return codes, vals


_CODES, _VALS = _finite_table()


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code (ties to the even code), saturating; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    a = np.where(np.isnan(a), 0.0, a)
    # the two table neighbours of |x|: largest value <= |x| and the next one up
    hi = np.searchsorted(_VALS, a, side="right")
    lo = hi - 1
    hi_c = np.minimum(hi, len(_VALS) - 1)
    dlo = a - _VALS[lo]
    dhi = _VALS[hi_c] - a
    lo_odd = (_CODES[lo] & 1) == 1
    take_hi = (hi < len(_VALS)) & ((dhi < dlo) | ((dhi == dlo) & lo_odd))
    code = np.where(take_hi, _CODES[hi_c], _CODES[lo]).astype(np.uint8)
    neg = np.signbit(x)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_quantize(x) -> np.ndarray:
    """x rounded to the nearest E4M3 value (float64 result)."""
    codes = e4m3_encode(x)
    dec = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return dec[codes]


def delayed_scale(amax_history_recent: float | None, margin: int = 0) -> float:
    """Scale from the most recent amax: 448 / amax / 2^margin; 1 with no history or amax 0."""
    if amax_history_recent is None or not amax_history_recent > 0:
        return 1.0
    return E4M3_MAX / float(amax_history_recent) / (2.0 ** margin)


def fp8_linear(x, w, b, scale_x: float, scale_w: float):
    """y = (Q(x*s_x) Q(w*s_w)^T) / (s_x s_w) + b with Q the E4M3 rounding."""
    qx = e4m3_quantize(np.asarray(x, np.float64) * scale_x)
    qw = e4m3_quantize(np.asarray(w, np.float64) * scale_w)
    y = qx @ qw.T / (scale_x * scale_w)
    return y if b is None else y + np.asarray(b, np.float64)


class DelayedScaling:
    """E4M3 casts of the block linears with per-tensor delayed scaling.

    "FP8 training for Flux models", §Configuration › FP8 model configuration
    (``fp8: "e4m3"``, ``amax_history_len: 1024``, ``amax_compute_algo:
    most_recent``, ``margin: 0``): every linear's input and weight are cast
    to E4M3 with the scale the tensor was given, the product is divided by
    both scales, and the tensor's absolute maximum is recorded so that the
    next call's scale is ``448 / amax`` (``delayed_scale``).

    ``scales`` maps a tensor name (``"<linear>.x"`` for the input,
    ``"<linear>.w"`` for the weight) to the scale it is cast with; names not
    given use 1, the scale of an empty history.  ``amax`` collects, per name,
    the largest |value| the tensor held in this evaluation.
    """

    def __init__(self, scales=None):
        self.scales = dict(scales or {})
        self.amax = {}

    def _record(self, name, a):
        m = float(np.max(np.abs(a))) if np.size(a) else 0.0
        self.amax[name] = max(self.amax.get(name, 0.0), m)

    def linear(self, name, x, w, b):
        """y = x W^T + b on E4M3 operands: x and w are cast as given (no other rounding)."""
        x = np.asarray(x, np.float64)
        w = np.asarray(w, np.float64)
        self._record(name + ".x", x)
        self._record(name + ".w", w)
        sx = float(self.scales.get(name + ".x", 1.0))
        sw = float(self.scales.get(name + ".w", 1.0))
        return fp8_linear(x, w, b, sx, sw)

    def next_scales(self, margin: int = 0):
        """The scales of the next call under ``most_recent``: 448 / amax / 2^margin."""
        return {k: delayed_scale(a, margin) for k, a in self.amax.items()}


def history_scale(amaxes, algo: str = "most_recent", margin: int = 0) -> float:
    """The delayed scale from a tensor's recorded amax values, oldest first.

    "FP8 training for Flux models", §Configuration (``fp8_amax_compute_algo: most_recent`` or
    ``max``, ``fp8_margin``) and §Troubleshooting (``max`` as the conservative choice): the amax
    the scale is taken from is the most recent recorded value, or the largest in the history
    window; the scale is then ``448 / amax / 2^margin`` (1 while no positive amax is recorded).
    """
    vals = [float(a) for a in amaxes]
    if not vals:
        return 1.0
    if algo == "most_recent":
        a = vals[-1]
    elif algo == "max":
        a = max(vals)
    else:
        raise ValueError(algo)
    return delayed_scale(a, margin)
