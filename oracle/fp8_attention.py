"""FP8 dot-product attention (the opt-in ``fp8_dot_product_attention``), fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/flux.py``).

The "FP8 training for Flux models" page (§Configuration › FP8 model configuration) keeps attention
out of FP8 by default (``fp8_dot_product_attention: false``) and names the switch without its
arithmetic.  The reading taken for the switch turned on: both products of the attention run on
E4M3 operands (``oracle.e4m3``: round to nearest even, saturating), the softmax stays in high
precision between them, and the probabilities enter the second product in the form a fused
attention kernel holds them, unnormalised:

  S   = Q4(q s_q) Q4(k s_k)^T / (s_q s_k sqrt(d))
  Pt  = exp(S - rowmax(S))            (each row's largest entry is exactly 1)
  O   = Q4(Pt s_p) Q4(v s_v) / (s_p s_v) / rowsum(Pt)

with s_q, s_k, s_v the tensors' scales (delayed scaling gives 448 / amax) and s_p = 448, the
scale of a tensor whose amax is 1.  The row sum is taken over the unquantised Pt.  This is a
diagnostic oracle with its own tolerance; the pass/fail oracle of the blocks keeps attention
exact (``oracle.flux.attention``).
"""
from __future__ import annotations

import math

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_quantize


def fp8_attention(q, k, v, s_q: float, s_k: float, s_v: float, s_p: float = E4M3_MAX):
    """Attention over the key axis of q, k, v [..., S, d] with E4M3 operands, as read above."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    d = q.shape[-1]
    s = (e4m3_quantize(q * s_q) @ np.swapaxes(e4m3_quantize(k * s_k), -1, -2)) / (s_q * s_k * math.sqrt(d))
    pt = np.exp(s - s.max(axis=-1, keepdims=True))
    o = e4m3_quantize(pt * s_p) @ e4m3_quantize(v * s_v) / (s_p * s_v)
    return o / pt.sum(axis=-1, keepdims=True)


def fp8_attention_delayed(q, k, v):
    """fp8_attention with each operand's scale at 448 / its amax (1 for an all-zero tensor)."""
    def scale(x):
        a = float(np.max(np.abs(x))) if np.size(x) else 0.0
        return E4M3_MAX / a if a > 0 else 1.0
    return fp8_attention(q, k, v, scale(q), scale(k), scale(v))
