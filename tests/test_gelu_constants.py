"""The GEMM epilogue evaluates the exact-erf GELU through Abramowitz & Stegun formula 7.1.26.

The coefficients are read out of the CUDA source, so this checks the kernel's own constants:
the formula they define must stay within the published 1.5e-7 of erf (math.erf) on a dense
grid, and GELU built from it within 1e-7 * |x| of the exact x * Phi(x) (CPU only)."""
import math
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "diffusion_transformer_flux_gb300", "csrc", "gemm_kernel.cuh")


def _constants():
    src = open(SRC).read()
    vals = {}
    for name in ("kAsP", "kAsA1", "kAsA2", "kAsA3", "kAsA4", "kAsA5"):
        m = re.search(name + r"\s*=\s*([-+0-9.eE]+)f", src)
        assert m, name
        vals[name] = float(m.group(1))
    return vals


def _erf_as(z, c):
    t = 1.0 / (1.0 + c["kAsP"] * z)
    poly = t * (c["kAsA1"] + t * (c["kAsA2"] + t * (c["kAsA3"] + t * (c["kAsA4"] + t * c["kAsA5"]))))
    return 1.0 - poly * np.exp(-z * z)


def test_erf_formula_of_the_kernel_meets_the_published_bound():
    c = _constants()
    z = np.linspace(0.0, 8.0, 200001)
    ref = np.array([math.erf(v) for v in z])
    assert np.abs(_erf_as(z, c) - ref).max() <= 1.5e-7


def test_gelu_from_the_kernel_formula():
    c = _constants()
    x = np.linspace(-12.0, 12.0, 48001)
    z = np.abs(x) / math.sqrt(2.0)
    q = 1.0 - _erf_as(z, c)
    g = 0.5 * x * np.where(x >= 0, 2.0 - q, q)
    ref = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    assert np.all(np.abs(g - ref) <= 1e-7 * np.maximum(np.abs(x), 1.0))
