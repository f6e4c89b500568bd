"""FP8 E5M2 quantisation, fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/flux.py``).

E5M2 as defined in "FP8 Formats for Deep Learning" (Micikevicius et al.,
2022), the gradient format of the ``"hybrid"`` setting that the "FP8 training
for Flux models" page offers beside E4M3 (§Configuration › FP8 model
configuration: E4M3 activations and weights, E5M2 gradients).  The format
follows the IEEE 754 conventions: 1 sign bit, 5 exponent bits with bias 15,
2 mantissa bits; exponent field 31 holds the infinities (mantissa 0) and the
NaNs (mantissa 1..3); the largest finite magnitude is 1.75 * 2^15 = 57344 and
the smallest subnormal 2^-16.

Conversion rounds to nearest, ties to the even code, and saturates to +-57344
(the reading taken for overflow, the same as for E4M3: a delayed scale taken
from an older amax can push a value past the largest finite one, and the
saturating conversion keeps it finite).  NaN converts to the code 0x7F.
"""
from __future__ import annotations

import numpy as np

E5M2_MAX = 57344.0


def e5m2_decode(code: int) -> float:
    """Value of an 8-bit E5M2 code from the format definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 2) & 0x1F
    man = code & 0x3
    if exp == 0x1F:
        return sign * float("inf") if man == 0 else float("nan")
    if exp == 0:
        return sign * (man / 4.0) * 2.0 ** (1 - 15)
    return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 15)


# non-negative finite codes 0x00..0x7B and their values, ascending
_CODES = np.arange(0x7C)
_VALS = np.array([e5m2_decode(c) for c in _CODES], dtype=np.float64)
_DECODE = np.array([e5m2_decode(c) for c in range(256)], dtype=np.float64)


def e5m2_encode(x) -> np.ndarray:
    """Nearest E5M2 code (ties to the even code), saturating to +-57344; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.where(np.isnan(x), 0.0, np.minimum(np.abs(x), E5M2_MAX))
    # the table neighbours of |x|: the largest value <= |x| and the one above it
    hi = np.searchsorted(_VALS, a, side="right")
    lo = hi - 1
    hi_c = np.minimum(hi, len(_VALS) - 1)
    dlo = a - _VALS[lo]
    dhi = _VALS[hi_c] - a
    lo_odd = (_CODES[lo] & 1) == 1
    take_hi = (hi < len(_VALS)) & ((dhi < dlo) | ((dhi == dlo) & lo_odd))
    code = np.where(take_hi, _CODES[hi_c], _CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def e5m2_quantize(x) -> np.ndarray:
    """x rounded to the nearest E5M2 value, saturating (float64 result)."""
    return _DECODE[e5m2_encode(x)]
