"""The parallel-branch single block through the C ABI, against the oracle.

* small shapes (D 256, 2 heads), bf16 against the bf16-autocast oracle and fp32 against the
  float64 one, batch 1 and 2, with ragged sequence lengths;
* the Flux-sized block (4096 + 512 tokens, D 3072, 24 heads, F 12288) on sampled rows;
* with the MLP silenced (W_1 = 0, b_1 = 0, b_2 = 0) the GPU block equals the GPU sequential block
  whose MLP gate is zero, bit for bit: the two share every kernel of the attention half.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from oracle import flux as O

from gpu_util import BlockCase, assert_parity, dev, host, torch_dtype, upload_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _parallel_case(B, S_i, S_t, D, H, F, act, seed):
    c = BlockCase(B, S_i, S_t, D, H, F, act, seed=seed, single=True)
    c.w_img["w_mod"] = c.w_img["w_mod"][:3 * D].copy()
    c.w_img["b_mod"] = c.w_img["b_mod"][:3 * D].copy()
    return c


def _run(c, w=None):
    t = torch_dtype(c.act)
    cos = torch.empty(c.B, c.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(torch.from_numpy(c.ids).cuda(), (16, 56, 56), 10000.0, cos, sin)
    x = dev(c.x_joint(), t)
    y = torch.empty_like(x)
    ws = L.mmdit_single_block_parallel_fwd(c.dims, upload_weights(w or c.w_img, c.act), dev(c.vec, t), cos, sin, x, y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    return host(y), (cos, sin)


@pytest.mark.parametrize("B,S_i,S_t", [(1, 256, 32), (2, 300, 45)])
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_parallel_block_small(B, S_i, S_t, act):
    c = _parallel_case(B, S_i, S_t, 256, 2, 1024, act, seed=80 + B)
    got, _ = _run(c)
    ref = O.single_block_parallel(c.x_joint(), c.vec, c.cos, c.sin, c.w_img, c.H, mm_cast=c.mm_cast)
    assert_parity(got, ref, 2e-2, f"parallel single block {act} B={B}", out_bf16=act == "bf16")


def test_parallel_block_flux_sized_sampled_rows():
    c = _parallel_case(1, 4096, 512, 3072, 24, 12288, "bf16", seed=90)
    got, _ = _run(c)
    rng = np.random.default_rng(3)
    rows = np.sort(np.concatenate([rng.choice(4096, 192, replace=False), 4096 + rng.choice(512, 64, replace=False)]))
    ref = O.single_block_parallel(c.x_joint(), c.vec, c.cos, c.sin, c.w_img, c.H, mm_cast=O.round_bf16, rows=rows)
    assert_parity(got[:, rows], ref, 2e-2, "parallel single block, 4096+512 tokens", out_bf16=True)


def test_parallel_attention_half_equals_the_sequential_block():
    c = _parallel_case(2, 300, 45, 256, 2, 1024, "bf16", seed=95)
    D = c.D
    w = dict(c.w_img, w_1=np.zeros_like(c.w_img["w_1"]), b_1=np.zeros_like(c.w_img["b_1"]),
             b_2=np.zeros_like(c.w_img["b_2"]))
    par, (cos, sin) = _run(c, w)
    # the sequential block with chunks (shift, scale, gate, anything, anything, 0)
    ws6 = dict(w, w_mod=np.concatenate([w["w_mod"], w["w_mod"][:2 * D], np.zeros((D, D), np.float32)]),
               b_mod=np.concatenate([w["b_mod"], w["b_mod"][:2 * D], np.zeros(D, np.float32)]))
    x = dev(c.x_joint())
    y = torch.empty_like(x)
    ws = L.mmdit_single_block_fwd(c.dims, upload_weights(ws6, "bf16"), dev(c.vec), cos, sin, x, y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    np.testing.assert_array_equal(par, host(y))
