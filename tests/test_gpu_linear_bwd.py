"""Backward of a linear layer through the C ABI (mmdit_linear_bwd) against the oracle's
chain-rule gradients: dx = dy W, dW = dy^T x, db = column sums of dy.

Shapes: a ragged token count (300 rows: the contraction of dW is padded to 304 with zeros),
the block's fc-sized linear (4608 x 3072 x 3072), fp32 (tf32 tensor cores), only some outputs
asked for, and an empty batch (dW and db become zero).  dx (bf16) and dW (fp32) are held to the
2e-2 x RMS bar against the float64 gradients of the same bf16 values; db, a sum of bf16 values
in fp32, to 1e-5 relative.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import synth
from oracle import backward as BW

from gpu_util import assert_parity, dev, host, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    dy = synth.bf16_round(rng.standard_normal((M, N)).astype(np.float32))
    x = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    w = synth.bf16_round((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    return dy, x, w


@pytest.mark.parametrize("act,M,N,K", [("bf16", 300, 256, 512), ("bf16", 4608, 3072, 3072), ("f32", 77, 64, 96)])
def test_linear_backward_matches_oracle(act, M, N, K):
    dy, x, w = _inputs(M, N, K, M + N)
    t = torch_dtype(act)
    dx = torch.empty(M, K, device="cuda", dtype=t)
    dw = torch.full((N, K), float("nan"), device="cuda")
    db = torch.full((N,), float("nan"), device="cuda")
    ws = L.mmdit_linear_bwd(dev(dy, t), dev(x, t), dev(w, t), dx, dw, db)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    rdx, rdw, rdb = BW.linear_bwd(dy, x, w)
    assert_parity(host(dx), rdx, 2e-2, f"dx {act} {M}x{N}x{K}", out_bf16=act == "bf16")
    assert_parity(host(dw), rdw, 2e-2, f"dW {act} {M}x{N}x{K}")
    np.testing.assert_allclose(host(db), rdb, rtol=1e-5, atol=1e-5 * np.abs(rdb).max())


def test_linear_backward_partial_outputs_and_empty_batch():
    dy, x, w = _inputs(130, 64, 96, 5)
    db = torch.empty(64, device="cuda")
    dx = torch.empty(130, 96, device="cuda", dtype=torch.bfloat16)
    # only db, then only dx (x and W not needed respectively)
    L.mmdit_linear_bwd(dev(dy), None, dev(w), None, None, db)
    L.mmdit_linear_bwd(dev(dy), None, dev(w), dx, None, None)
    torch.cuda.synchronize()
    rdx, _, rdb = BW.linear_bwd(dy, x, w)
    np.testing.assert_allclose(host(db), rdb, rtol=1e-5, atol=1e-5 * np.abs(rdb).max())
    assert_parity(host(dx), rdx, 2e-2, "dx alone", out_bf16=True)
    # no rows: the weight and bias gradients are zero
    dw0 = torch.full((64, 96), 7.0, device="cuda")
    db0 = torch.full((64,), 7.0, device="cuda")
    empty = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    L.mmdit_linear_bwd(empty, torch.empty(0, 96, device="cuda", dtype=torch.bfloat16), dev(w), None, dw0, db0)
    torch.cuda.synchronize()
    assert float(dw0.abs().max()) == 0.0 and float(db0.abs().max()) == 0.0
