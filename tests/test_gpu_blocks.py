"""GPU parity of the double- and single-block forward against the fp64 oracle.

The bar (max |err| <= 2e-2 x output RMS) is checked against the oracle at the precision the
pages fix for training, bf16 autocast (every matrix-product operand rounded to bf16, all other
arithmetic in float64), allowing in addition half a bf16 ulp per element because the block's
output is itself stored in bf16.  The distance to the pure float64 oracle is checked too, at
the looser bound that bf16 operands allow (TOL_VS_FP64).  fp32 workloads (tf32 linears) are
held to the bar against the pure float64 oracle.

Small shapes (several tiles, ragged tails) are compared element by element on every output
and on the intermediates the workspace exposes (Q, K, V^T after RMSNorm/RoPE, the attention
output), so a failure names the step.  The Flux-sized workloads run in the launch
configuration the benchmark times and are compared on seeded samples of rows, which the
oracle computes exactly (every step after attention is row-wise).
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from oracle import flux as O

from gpu_util import TOL_VS_FP64, BlockCase, assert_parity, host, workspace_view

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _check_intermediates(case: BlockCase, ws):
    """Q, K (normalised and rotated), V^T and the attention output against the oracle at the
    case's precision; all four are stored in bf16 (half-ulp allowance)."""
    c = case.mm_cast
    offs = L.mmdit_block_workspace_offsets(case.dims, case.single)
    B, H, S, D = case.B, case.H, case.S, case.D
    S_pad = (S + 7) // 8 * 8
    qs, ks, vs = [], [], []
    streams = [(case.w_img, case.x_joint() if case.single else case.x_img)]
    if not case.single:
        streams.append((case.w_txt, case.x_txt))
    for w, x in streams:
        m = O.modulation(case.vec, w["w_mod"], w["b_mod"], mm_cast=c)
        q, k, v = O.qkv_heads(x, m[0], m[1], w, H, mm_cast=c)
        qs.append(q), ks.append(k), vs.append(v)
    q, k, v = (np.concatenate(a, axis=2) for a in (qs, ks, vs))
    cs, sn = case.cos[:, None], case.sin[:, None]
    q = O.apply_rope(q, cs, sn, case.interleaved)
    k = O.apply_rope(k, cs, sn, case.interleaved)
    gq = host(workspace_view(ws, offs[2], (B, H, S, 128), torch.bfloat16))
    gk = host(workspace_view(ws, offs[3], (B, H, S, 128), torch.bfloat16))
    gvt = host(workspace_view(ws, offs[4], (B, H, 128, S_pad), torch.float16))[..., :S]
    assert_parity(gq, q, 2e-2, "Q after RMSNorm + RoPE", out_bf16=True)
    assert_parity(gk, k, 2e-2, "K after RMSNorm + RoPE", out_bf16=True)
    assert_parity(gvt, np.swapaxes(v, -1, -2), 2e-2, "V^T", out_bf16=True)
    o = O.attention(q, k, v, c).transpose(0, 2, 1, 3).reshape(B, S, D)
    t = torch.float32 if case.act == "f32" else torch.bfloat16
    ob = case.act != "f32"
    rows_i = B * (S if case.single else case.S_i)
    go = host(workspace_view(ws, offs[5], (rows_i, D), t)).reshape(B, -1, D)
    if case.single:
        assert_parity(go, o, 2e-2, "attention output", out_bf16=ob)
    else:
        assert_parity(go, o[:, :case.S_i], 2e-2, "attention output (image rows)", out_bf16=ob)
        if case.S_t:
            got = host(workspace_view(ws, offs[6], (B * case.S_t, D), t)).reshape(B, -1, D)
            assert_parity(got, o[:, case.S_i:], 2e-2, "attention output (text rows)", out_bf16=ob)


def _check_outputs(case: BlockCase, got, rows=None):
    """The bar on every output, then the distance to the pure float64 oracle."""
    names = ["y"] if case.single else ["y_img", "y_txt"]
    xs = [case.x_joint()] if case.single else [case.x_img, case.x_txt]
    bf = case.act != "f32"
    if rows is None:
        ref, ref64 = case.oracle(case.mm_cast), case.oracle(None) if bf else None
        sel = [slice(None)] * len(names)
    else:
        ref = case.oracle_rows(*rows, mm_cast=case.mm_cast)
        ref64 = case.oracle_rows(*rows, mm_cast=None) if bf else None
        sel = list(rows)
    for i, (n, g, x) in enumerate(zip(names, got, xs)):
        r = ref[i]
        if r.size == 0:
            continue
        g, x = g[:, sel[i]], x[:, sel[i]]
        assert_parity(g, r, 2e-2, n, out_bf16=bf)
        # the residual dominates the output; the branch alone must also be close
        assert_parity(g - x, r - x, 0.1, n + " branch (y - x)", out_bf16=bf)
        if bf:
            assert_parity(g, ref64[i], TOL_VS_FP64, n + " vs float64 oracle", out_bf16=True)


# ----------------------------------------------------------------------------- small shapes
SMALL = [
    # B, S_i, S_t, D, H, F, act, interleaved, gelu_tanh
    (1, 256, 32, 256, 2, 1024, "f32", True, False),     # the tiny fp32 workload
    (2, 300, 45, 256, 2, 1024, "bf16", True, False),    # ragged tails, batch 2
    (1, 200, 77, 512, 4, 1536, "bf16", False, True),    # half-split RoPE, tanh GELU
    (3, 130, 0, 256, 2, 512, "bf16", True, False),      # no text tokens
]


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,act,inter,tanh", SMALL)
def test_double_block_small(B, S_i, S_t, D, H, F, act, inter, tanh):
    case = BlockCase(B, S_i, S_t, D, H, F, act, seed=S_i + D, std=0.05, interleaved=inter,
                     gelu_tanh=tanh)
    got, ws, _ = case.run_gpu()
    _check_outputs(case, got)
    _check_intermediates(case, ws)


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,act,inter,tanh", SMALL[:3])
def test_single_block_small(B, S_i, S_t, D, H, F, act, inter, tanh):
    case = BlockCase(B, S_i, S_t, D, H, F, act, seed=7 + S_i, std=0.05, single=True,
                     interleaved=inter, gelu_tanh=tanh)
    got, ws, _ = case.run_gpu()
    _check_outputs(case, got)
    _check_intermediates(case, ws)


def test_tiny_workload_with_flux_init():
    """The tiny fp32 workload exactly as configured: N(0, 0.02) weights, 16x16 image grid."""
    case = BlockCase(1, 256, 32, 256, 2, 1024, "f32", seed=1000, std=0.02, gain_jitter=0.0,
                     lat_hw=(16, 16))
    got, _, _ = case.run_gpu()
    for g, r in zip(got, case.oracle()):
        assert_parity(g, r, 2e-2, "tiny fp32 double block")


def test_block_output_may_alias_input():
    case = BlockCase(2, 130, 40, 256, 2, 1024, "bf16", seed=3, std=0.05)
    ref = case.oracle(case.mm_cast)
    t = torch.bfloat16
    from gpu_util import dev, upload_weights
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    xi, xt = dev(case.x_img, t), dev(case.x_txt, t)
    L.mmdit_double_block_fwd(case.dims, upload_weights(case.w_img, "bf16"),
                             upload_weights(case.w_txt, "bf16"), dev(case.vec, t), cos, sin, xi, xt,
                             xi, xt)
    torch.cuda.synchronize()
    assert_parity(host(xi), ref[0], 2e-2, "aliased y_img", out_bf16=True)
    assert_parity(host(xt), ref[1], 2e-2, "aliased y_txt", out_bf16=True)


@pytest.mark.parametrize("single", [False, True])
def test_precomputed_modulation_gives_identical_blocks(single):
    """A modulation computed ahead by mmdit_modulation_fwd and handed over through the weight
    set's `mod` gives the same bits as the block computing it itself."""
    case = BlockCase(2, 300, 45, 256, 2, 1024, "bf16", seed=19, std=0.05, single=single)
    from gpu_util import dev, upload_weights
    t = torch.bfloat16
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    vec = dev(case.vec, t)
    sets = [upload_weights(case.w_img, "bf16")] + ([] if single else [upload_weights(case.w_txt, "bf16")])
    outs = []
    for pre in (False, True):
        ws_ = [dict(w) for w in sets]
        if pre:
            for w in ws_:
                w["mod"] = torch.empty(case.B, 6 * case.D, device="cuda")
                L.mmdit_modulation_fwd(vec, w["w_mod"], w["b_mod"], w["mod"])
        if single:
            x = dev(case.x_joint(), t)
            y = torch.empty_like(x)
            L.mmdit_single_block_fwd(case.dims, ws_[0], vec, cos, sin, x, y)
            outs.append((y,))
        else:
            xi, xt = dev(case.x_img, t), dev(case.x_txt, t)
            yi, yt = torch.empty_like(xi), torch.empty_like(xt)
            L.mmdit_double_block_fwd(case.dims, ws_[0], ws_[1], vec, cos, sin, xi, xt, yi, yt)
            outs.append((yi, yt))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ----------------------------------------------------------------------------- Flux-sized workloads
def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(n, size=min(k, n), replace=False))
    return np.unique(np.concatenate([rows, [0, n - 1]]))


@pytest.mark.parametrize("B,lat,S_t", [(1, 64, 512), (4, 32, 512), (2, 64, 512)])
def test_double_block_flux_sized_sampled_rows(B, lat, S_t):
    """12B/535M block shapes (D 3072, 24 heads, F 12288) at 4096+512, 4x(1024+512) and
    2x(4096+512) tokens."""
    case = BlockCase(B, lat * lat, S_t, 3072, 24, 12288, "bf16", seed=1001 + B, std=0.02,
                     gain_jitter=0.0, lat_hw=(lat, lat))
    got, _, _ = case.run_gpu()
    _check_outputs(case, got, rows=(_sample(case.S_i, 96, 1), _sample(S_t, 32, 2)))


@pytest.mark.parametrize("B", [1, 2])
def test_single_block_flux_sized_sampled_rows(B):
    """The single block at 4096+512 tokens, batch 1 and 2 (the 535M-shaped and 1024 px
    workloads)."""
    case = BlockCase(B, 4096, 512, 3072, 24, 12288, "bf16", seed=1011 + B, std=0.02, gain_jitter=0.0,
                     lat_hw=(64, 64), single=True)
    got, _, _ = case.run_gpu()
    _check_outputs(case, got, rows=(_sample(case.S, 128, 3),))
