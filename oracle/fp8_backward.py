"""Backward of the FP8 block linears with delayed scaling, fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/flux.py``).

The "FP8 training for Flux models" page (§Configuration › FP8 model configuration) names the
settings and not the arithmetic: ``fp8: "e4m3"`` casts every FP8 operand to E4M3; ``"hybrid"``
keeps E4M3 for activations and weights and casts the gradients to E5M2; ``fp8_wgrad: true``
computes the weight gradient from FP8 operands as well.  The readings taken, for the linear
y = x W^T + b whose forward ran on Q4(x s_x) and Q4(W s_w) (``oracle.e4m3.fp8_linear``):

* the incoming gradient dy gets a delayed scale of its own, s_dy = fmax / amax / 2^margin with
  fmax the largest finite value of the gradient format (448 for E4M3, 57344 for E5M2), and is
  cast to that format: G = Qg(dy s_dy);
* dgrad: dx = G Q4(W s_w) / (s_dy s_w), on the weight cast of the forward;
* wgrad with ``fp8_wgrad``: dW = G^T Q4(x s_x) / (s_dy s_x), on the input cast of the forward,
  summed over every row of the batch; without it dW = dy^T x on the unquantised tensors;
* db is the column sum of the unquantised dy (a bias gradient is a reduction, not a GEMM).

The products are exact in float64 here, as the GEMMs accumulate in fp32 or wider on the device.
"""
from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, DelayedScaling, e4m3_quantize
from .e5m2 import E5M2_MAX, e5m2_quantize

RECIPES = ("e4m3", "hybrid")


def gradient_format(recipe: str):
    """(quantiser, largest finite value) of the gradient format of a recipe."""
    if recipe == "e4m3":
        return e4m3_quantize, E4M3_MAX
    if recipe == "hybrid":
        return e5m2_quantize, E5M2_MAX
    raise ValueError(recipe)


def gradient_scale(amax: float | None, recipe: str = "e4m3", margin: int = 0) -> float:
    """Delayed scale of a gradient: fmax / amax / 2^margin; 1 while no positive amax is recorded."""
    if amax is None or not amax > 0:
        return 1.0
    return gradient_format(recipe)[1] / float(amax) / (2.0 ** margin)


def fp8_linear_bwd(dy, x, w, s_x: float, s_w: float, s_dy: float, recipe: str = "e4m3",
                   wgrad: bool = True):
    """(dx, dW, db) of y = x W^T + b run on E4M3 operands, with the gradient cast per ``recipe``.

    dy [..., N], x [..., K], W [N, K]; dW sums over every leading index of dy and x.
    """
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    qg = gradient_format(recipe)[0]
    g = qg(dy * s_dy)
    dx = g @ e4m3_quantize(w * s_w) / (s_dy * s_w)
    g2 = g.reshape(-1, g.shape[-1])
    x2 = x.reshape(-1, x.shape[-1])
    if wgrad:
        dw = g2.T @ e4m3_quantize(x2 * s_x) / (s_dy * s_x)
    else:
        dw = dy.reshape(-1, dy.shape[-1]).T @ x2
    db = dy.reshape(-1, dy.shape[-1]).sum(axis=0)
    return dx, dw, db


class DelayedScalingTraining(DelayedScaling):
    """Forward and backward of the FP8 linears under one recipe, with delayed scales.

    Extends the forward context of ``oracle.e4m3.DelayedScaling`` with the gradient tensors:
    ``"<linear>.dy"`` names the gradient arriving at a linear's output.  Its scale comes from
    ``scales`` like the others (1 when not given) and its amax is recorded per call, so that
    ``next_scales`` gives every tensor its ``most_recent`` scale against its own format's maximum.
    """

    def __init__(self, scales=None, recipe: str = "e4m3", wgrad: bool = True):
        super().__init__(scales)
        gradient_format(recipe)
        self.recipe = recipe
        self.wgrad = wgrad

    def linear_bwd(self, name, dy, x, w):
        """(dx, dW, db) of the linear ``name`` whose forward ran on (x, w)."""
        self._record(name + ".dy", np.asarray(dy, np.float64))
        s = lambda k: float(self.scales.get(name + k, 1.0))  # noqa: E731
        return fp8_linear_bwd(dy, x, w, s(".x"), s(".w"), s(".dy"), self.recipe, self.wgrad)

    def next_scales(self, margin: int = 0):
        out = {}
        for k, a in self.amax.items():
            if k.endswith(".dy"):
                out[k] = gradient_scale(a, self.recipe, margin)
            else:
                out[k] = gradient_scale(a, "e4m3", margin)
        return out
