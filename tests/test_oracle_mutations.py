"""Planted mistakes in a copy of the oracle: each must make at least one pin fail (CPU only).

The pins are meant to catch a plausible error anywhere in the oracle.  This test copies
``oracle/``, the pin tests and the synthetic-input module to a temporary directory, plants one
mistake at a time (a dropped term, a wrong sign, exponent or index, a transposed operand, a
swapped order) and runs the pins there; every planted mistake must fail at least one of them.
A control run of the unmodified copy must pass, so that a broken copy cannot pass this test.
The oracle in the repository is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file under oracle/, what the mistake is, text, replacement)
MUTATIONS = [
    ("flux.py", "modulate drops the 1 + of the scale",
     "layernorm(x, eps) * (1.0 + _f64(scale)[:, None, :])", "layernorm(x, eps) * (_f64(scale)[:, None, :])"),
    ("flux.py", "gated residual subtracts",
     "return _f64(x) + _f64(gate)[:, None, :] * _f64(y)", "return _f64(x) - _f64(gate)[:, None, :] * _f64(y)"),
    ("flux.py", "RoPE frequency exponent halved",
     "inv_freq = float(theta) ** (-2.0 * i / d_a)", "inv_freq = float(theta) ** (-1.0 * i / d_a)"),
    ("flux.py", "RoPE rotation sign", "ra = a * cos - b * sin", "ra = a * cos + b * sin"),
    ("flux.py", "attention without 1/sqrt(d)",
     "s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(d)", "s = (q @ np.swapaxes(k, -1, -2))"),
    ("flux.py", "LayerNorm with the unbiased variance",
     "var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)",
     "var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    ("flux.py", "RMSNorm without its gain",
     "return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * _f64(g)",
     "return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)"),
    ("flux.py", "GELU with erf(x/2)", "0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))", "0.5 * x * (1.0 + _erf(x / 2.0))"),
    ("flux.py", "modulation chunks reversed",
     "return np.split(m, n_chunks, axis=-1)", "return np.split(m, n_chunks, axis=-1)[::-1]"),
    ("flux.py", "noise coefficients swapped",
     "return (1.0 - tt) * z0 + tt * z1", "return tt * z0 + (1.0 - tt) * z1"),
    ("flux.py", "loss summed instead of averaged",
     "return float(np.mean(diff * diff))", "return float(np.sum(diff * diff))"),
    ("flux.py", "unpatchify without the transpose",
     "return t.transpose(0, 2, 1).reshape(B, C, H, W)", "return t.reshape(B, C, H, W)"),
    ("flux.py", "timestep features sine first",
     "return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)",
     "return np.concatenate([np.sin(ang), np.cos(ang)], axis=1)"),
    ("flux.py", "embedder without its SiLU",
     "return linear(silu(linear(x, w1, b1, mm_cast)), w2, b2, mm_cast)",
     "return linear(linear(x, w1, b1, mm_cast), w2, b2, mm_cast)"),
    ("flux.py", "whole model joins the streams as [txt; img]",
     "c = np.concatenate([x_img, x_txt], axis=1)", "c = np.concatenate([x_txt, x_img], axis=1)"),
    ("flux.py", "parallel block drops the fc2 bias",
     'linear(om, w_cat, _f64(w["b_o"]) + _f64(w["b_2"]), mm_cast)', 'linear(om, w_cat, _f64(w["b_o"]), mm_cast)'),
    ("flux.py", "double block: the MLP gate on the attention branch",
     "x_img = gated_residual(x_img, mi[2], out_proj(", "x_img = gated_residual(x_img, mi[5], out_proj("),
    ("flux.py", "q normalised with the k gain",
     'q = rmsnorm(_heads(q, heads), w["g_q"], rms_eps)', 'q = rmsnorm(_heads(q, heads), w["g_k"], rms_eps)'),
    ("e4m3.py", "E4M3 ties rounded up instead of to even",
     "take_hi = (hi < len(_VALS)) & ((dhi < dlo) | ((dhi == dlo) & lo_odd))",
     "take_hi = (hi < len(_VALS)) & (dhi <= dlo)"),
    ("e5m2.py", "E5M2 exponent bias 16",
     "return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 15)", "return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 16)"),
    ("e5m2.py", "E5M2 ties rounded away from zero",
     "take_hi = (hi < len(_VALS)) & ((dhi < dlo) | ((dhi == dlo) & lo_odd))",
     "take_hi = (hi < len(_VALS)) & (dhi <= dlo)"),
    ("fp8_backward.py", "hybrid gradients cast to E4M3",
     "return e5m2_quantize, E5M2_MAX", "return e4m3_quantize, E5M2_MAX"),
    ("fp8_backward.py", "dgrad not divided by the weight scale",
     "dx = g @ e4m3_quantize(w * s_w) / (s_dy * s_w)", "dx = g @ e4m3_quantize(w * s_w) / s_dy"),
    ("fp8_backward.py", "FP8 wgrad on the unquantised input",
     "dw = g2.T @ e4m3_quantize(x2 * s_x) / (s_dy * s_x)", "dw = g2.T @ x2 / s_dy"),
    ("fp8_backward.py", "gradient scales against the E4M3 maximum under every recipe",
     "out[k] = gradient_scale(a, self.recipe, margin)", 'out[k] = gradient_scale(a, "e4m3", margin)'),
    ("fp8_recipes.py", "MX shared exponent one too high",
     "e = np.where(pos, k.astype(np.int64) - 1 - E4M3_EMAX, E8M0_MIN_EXP)",
     "e = np.where(pos, k.astype(np.int64) - E4M3_EMAX, E8M0_MIN_EXP)"),
    ("fp8_recipes.py", "MX elements multiplied by the block scale instead of divided",
     "p[..., sl] = e4m3_quantize(np.ldexp(part, -ej[..., None]))",
     "p[..., sl] = e4m3_quantize(np.ldexp(part, ej[..., None]))"),
    ("fp8_recipes.py", "MX linear takes the input's block exponent twice",
     "y = mxfp8_dequantize(px, ex, block) @ mxfp8_dequantize(pw, ew, block).T",
     "y = mxfp8_dequantize(px, 2 * ex, block) @ mxfp8_dequantize(pw, 0 * ew, block).T"),
    ("fp8_recipes.py", "blockwise weight tiles one row high",
     "ns, ks = _slices(w.shape[0], tile), _slices(w.shape[1], tile)",
     "ns, ks = _slices(w.shape[0], 1), _slices(w.shape[1], tile)"),
    ("fp8_recipes.py", "tensorwise input cast with the weight's scale",
     "sx, sw = tensorwise_scale(x, margin), tensorwise_scale(w, margin)",
     "sx, sw = tensorwise_scale(w, margin), tensorwise_scale(w, margin)"),
    ("flux.py", "whole model with the parallel switch still runs the sequential single block",
     "single = single_block_parallel if single_parallel else single_block", "single = single_block"),
    ("backward.py", "the whole-model backward's parallel single forward drops its MLP branch",
     'branch = linear_fwd(_merge(o), w["w_o"], w["b_o"]) + linear_fwd(u, w["w_2"], w["b_2"])\n    return',
     'branch = linear_fwd(_merge(o), w["w_o"], w["b_o"])\n    return'),
    ("fp8_attention.py", "FP8 attention without the division by the row sum",
     "return o / pt.sum(axis=-1, keepdims=True)", "return o"),
    ("fp8_attention.py", "FP8 attention casts the probabilities at scale 1",
     "def fp8_attention(q, k, v, s_q: float, s_k: float, s_v: float, s_p: float = E4M3_MAX):",
     "def fp8_attention(q, k, v, s_q: float, s_k: float, s_v: float, s_p: float = 1.0):"),
    ("backward.py", "RoPE backward rotates the same way",
     "return rope_rotate(dy, cos, -_f(sin), interleaved)", "return rope_rotate(dy, cos, _f(sin), interleaved)"),
    ("backward.py", "softmax backward without the row-sum term",
     "ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))", "ds = p * dp"),
    ("backward.py", "GELU derivative without u phi(u)",
     "return cdf + u * np.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)", "return cdf"),
    ("backward.py", "bias gradient averaged",
     "db = dy.reshape(-1, dy.shape[-1]).sum(axis=0)", "db = dy.reshape(-1, dy.shape[-1]).mean(axis=0)"),
    ("backward.py", "LayerNorm backward without the xhat term",
     "return r * (dxhat - dxhat.mean(axis=-1, keepdims=True)\n                - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))",
     "return r * (dxhat - dxhat.mean(axis=-1, keepdims=True))"),
]


def _pins(tests_dir):
    return sorted(os.path.join("tests", f) for f in os.listdir(tests_dir) if f.startswith("test_oracle_pins_"))


@pytest.fixture(scope="module")
def sandbox(tmp_path_factory):
    d = str(tmp_path_factory.mktemp("oracle_mutations"))
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(d, "tests"))
    for f in os.listdir(os.path.join(ROOT, "tests")):
        if f.startswith("test_oracle_pins_") or f == "conftest.py":
            shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(d, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(d, "tests", "golden"))
    pkg = os.path.join(d, "diffusion_transformer_flux_gb300")
    os.makedirs(pkg)
    for f in ("__init__.py", "synth.py"):
        shutil.copy(os.path.join(ROOT, "diffusion_transformer_flux_gb300", f), os.path.join(pkg, f))
    return d


def _run_pins(d):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                           *_pins(os.path.join(d, "tests"))], cwd=d, env=env, capture_output=True, text=True,
                          timeout=900)


def test_unmodified_copy_passes(sandbox):
    r = _run_pins(sandbox)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("fname,what,old,new", MUTATIONS, ids=[m[1] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(sandbox, fname, what, old, new):
    path = os.path.join(sandbox, "oracle", fname)
    with open(path) as f:
        src = f.read()
    assert src.count(old) == 1, f"the text to plant the mistake in was not found once: {what}"
    try:
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        r = _run_pins(sandbox)
    finally:
        with open(path, "w") as f:
            f.write(src)
    assert r.returncode != 0, f"no pin caught: {what}"
