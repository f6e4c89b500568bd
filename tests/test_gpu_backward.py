"""GPU parity of the block backward (mmdit_double_block_bwd, mmdit_single_block_bwd) against the
float64 oracle of the chain rule (oracle.backward), on the same seeded inputs.

Every gradient the calls write is compared: the input streams' dx, dvec, and each stream's weight,
bias, gain and modulation gradients.  The bar comes from a numpy emulation of the GPU's roundings
(bf16 storage of every tensor the GPU stores in bf16, bf16 GEMM operands with fp32 accumulation,
fp16 P and dS in the attention backward) against the same float64 oracle: at these shapes the
emulated evaluation sits at most 1e-2 from it norm-wise and 0.17 x RMS in max norm (weight
gradients are sums over every row, so single entries carry the rounding of many products).  The
GPU is held to twice that: ||g - g64|| / ||g64|| <= 2e-2 and max|g - g64| <= 0.35 x RMS(g64).
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from oracle import backward as BW

from gpu_util import BlockCase, dev, host, upload_weights

pytestmark = pytest.mark.gpu
NORM_TOL = 2e-2
MAX_TOL = 0.35
NAMES = ("w_mod", "b_mod", "w_qkv", "b_qkv", "g_q", "g_k", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2")


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _check(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    nrm = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    rms = float(np.sqrt(np.mean(ref * ref)))
    mx = float(np.abs(got - ref).max()) / max(rms, 1e-300)
    assert nrm <= NORM_TOL, f"{what}: ||g - g64|| / ||g64|| = {nrm:.3e} > {NORM_TOL}"
    assert mx <= MAX_TOL, f"{what}: max|g - g64| / RMS = {mx:.3e} > {MAX_TOL}"
    return nrm, mx


def _grads_like(w):
    return {n: torch.full(tuple(np.shape(w[n])), float("nan"), device="cuda") for n in NAMES}


def _rope(case):
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    return cos, sin


def _dy(case, rng, shape):
    # gradient-sized values (the gradient scale of the attention backward keeps them in fp16 range)
    from diffusion_transformer_flux_gb300 import synth
    return synth.bf16_round(rng.standard_normal(shape).astype(np.float32) * 1e-3)


def _report(rows):
    worst = sorted(rows, key=lambda r: -r[1])[:4]
    print("[bwd] worst norm-wise: " + ", ".join(f"{n} {a:.2e} (max {m:.2e})" for n, a, m in worst))


@pytest.mark.parametrize("B,S_i,lat,S_t,D,H,F,interleaved,gelu_tanh", [
    (2, 256, 16, 45, 256, 2, 1024, True, False),
    (1, 100, 10, 20, 384, 3, 512, False, True),
])
def test_double_block_backward_matches_oracle(B, S_i, lat, S_t, D, H, F, interleaved, gelu_tanh):
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=90 + S_i, std=0.05, lat_hw=(lat, lat),
                     interleaved=interleaved, gelu_tanh=gelu_tanh)
    rng = np.random.default_rng(7 + S_i)
    dy_i, dy_t = _dy(case, rng, case.x_img.shape), _dy(case, rng, case.x_txt.shape)
    cos, sin = _rope(case)
    wi, wt = upload_weights(case.w_img, "bf16"), upload_weights(case.w_txt, "bf16")
    xi, xt = dev(case.x_img), dev(case.x_txt)
    dxi, dxt = torch.empty_like(xi), torch.empty_like(xt)
    dvec = torch.full((B, D), float("nan"), device="cuda")
    gi, gt = _grads_like(case.w_img), _grads_like(case.w_txt)
    ws = L.mmdit_double_block_bwd(case.dims, wi, wt, dev(case.vec), cos, sin, xi, xt, dev(dy_i), dev(dy_t),
                                  dxi, dxt, dvec, gi, gt)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    rdi, rdt, rdv, rgi, rgt = BW.double_block_backward(case.x_img, case.x_txt, case.vec, case.cos, case.sin,
                                                       case.w_img, case.w_txt, H, dy_i, dy_t,
                                                       interleaved, gelu_tanh)
    rows = [("dx_img", *_check(host(dxi), rdi, "dx_img")), ("dx_txt", *_check(host(dxt), rdt, "dx_txt")),
            ("dvec", *_check(host(dvec), rdv, "dvec"))]
    for name, g, r in (("img", gi, rgi), ("txt", gt, rgt)):
        for n in NAMES:
            rows.append((f"{name}.{n}", *_check(host(g[n]), r[n], f"{name}.{n}")))
    _report(rows)


@pytest.mark.parametrize("B,S_i,lat,S_t,D,H,F", [(2, 256, 16, 45, 256, 2, 1024), (1, 64, 8, 9, 512, 4, 1536)])
def test_single_block_backward_matches_oracle(B, S_i, lat, S_t, D, H, F):
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=95 + S_i, std=0.05, lat_hw=(lat, lat), single=True)
    rng = np.random.default_rng(11 + S_i)
    x = case.x_joint()
    dy = _dy(case, rng, x.shape)
    cos, sin = _rope(case)
    w = upload_weights(case.w_img, "bf16")
    gx = dev(x)
    dx = torch.empty_like(gx)
    dvec = torch.full((B, D), float("nan"), device="cuda")
    g = _grads_like(case.w_img)
    ws = L.mmdit_single_block_bwd(case.dims, w, dev(case.vec), cos, sin, gx, dev(dy), dx, dvec, g)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    rdx, rdv, rg = BW.single_block_backward(x, case.vec, case.cos, case.sin, case.w_img, H, dy)
    rows = [("dx", *_check(host(dx), rdx, "dx")), ("dvec", *_check(host(dvec), rdv, "dvec"))]
    for n in NAMES:
        rows.append((n, *_check(host(g[n]), rg[n], n)))
    _report(rows)


def test_backward_optional_outputs_and_repeat():
    """Gradients left out (NULL) are not written; two calls give the same dx and weight gradients
    (fixed-order reductions; dQ's atomic additions only move the last bits of fp32 values)."""
    case = BlockCase(1, 64, 16, 256, 2, 1024, "bf16", seed=3, std=0.05, lat_hw=(8, 8), single=True)
    rng = np.random.default_rng(5)
    x = case.x_joint()
    dy = dev(_dy(case, rng, x.shape))
    cos, sin = _rope(case)
    w = upload_weights(case.w_img, "bf16")
    gx = dev(x)
    dx1, dx2 = torch.empty_like(gx), torch.empty_like(gx)
    g1 = {"w_1": torch.zeros(1024, 256, device="cuda"), "b_mod": torch.zeros(6 * 256, device="cuda")}
    g2 = {"w_1": torch.zeros(1024, 256, device="cuda"), "b_mod": torch.zeros(6 * 256, device="cuda")}
    ws = L.mmdit_single_block_bwd(case.dims, w, dev(case.vec), cos, sin, gx, dy, dx1, None, g1)
    L.mmdit_single_block_bwd(case.dims, w, dev(case.vec), cos, sin, gx, dy, dx2, None, g2, ws=ws)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    # the MLP branch's gradients come before the attention backward: bit-equal
    assert torch.equal(g1["w_1"], g2["w_1"])
    # what depends on dQ (the attention branch's LayerNorm shift and scale, dx) can move in the
    # last bits with the order of dQ's atomic fp32 additions
    assert torch.allclose(g1["b_mod"], g2["b_mod"], rtol=1e-3, atol=1e-3 * float(g1["b_mod"].abs().max()))
    assert (host(dx1 - dx2) == 0).mean() > 0.9
    rdx, _, rg = BW.single_block_backward(x, case.vec, case.cos, case.sin, case.w_img, case.H, host(dy))
    _check(host(g1["w_1"]), rg["w_1"], "w_1")
    _check(host(g1["b_mod"]), rg["b_mod"], "b_mod")


def _close(a, b, what, rel=1e-5):
    a, b = host(a), host(b)
    scale = max(float(np.abs(b).max()), 1e-30)
    err = float(np.abs(a - b).max())
    assert err <= rel * scale, f"{what}: max diff {err:.3e} > {rel} x {scale:.3e}"


def test_training_pair_matches_the_one_call_backward():
    """mmdit_double_block_fwd_train gives the forward's outputs bit for bit, and
    mmdit_double_block_bwd_saved the one-call backward's gradients (the same kernels on the same
    values; only dQ's atomic accumulation order may move the last bits of the attention-side
    gradients).  Likewise for the single block."""
    B, S_i, S_t, D, H, F = 2, 256, 45, 256, 2, 1024
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=77, std=0.05, lat_hw=(16, 16))
    rng = np.random.default_rng(78)
    dy_i, dy_t = dev(_dy(case, rng, case.x_img.shape)), dev(_dy(case, rng, case.x_txt.shape))
    cos, sin = _rope(case)
    wi, wt = upload_weights(case.w_img, "bf16"), upload_weights(case.w_txt, "bf16")
    xi, xt, vec = dev(case.x_img), dev(case.x_txt), dev(case.vec)
    # reference: the forward, then the one-call backward
    yi, yt = torch.empty_like(xi), torch.empty_like(xt)
    L.mmdit_double_block_fwd(case.dims, wi, wt, vec, cos, sin, xi, xt, yi, yt)
    ref_dx = torch.empty_like(xi), torch.empty_like(xt)
    ref_dvec = torch.empty(B, D, device="cuda")
    ref_g = _grads_like(case.w_img), _grads_like(case.w_txt)
    L.mmdit_double_block_bwd(case.dims, wi, wt, vec, cos, sin, xi, xt, dy_i, dy_t, ref_dx[0], ref_dx[1], ref_dvec,
                             ref_g[0], ref_g[1])
    # the training pair
    ti, tt = torch.full_like(xi, float("nan")), torch.full_like(xt, float("nan"))
    saved = L.mmdit_double_block_fwd_train(case.dims, wi, wt, vec, cos, sin, xi, xt, ti, tt)
    dx = torch.empty_like(xi), torch.empty_like(xt)
    dvec = torch.empty(B, D, device="cuda")
    g = _grads_like(case.w_img), _grads_like(case.w_txt)
    L.mmdit_double_block_bwd_saved(case.dims, wi, wt, vec, cos, sin, xi, xt, dy_i, dy_t, dx[0], dx[1], saved, dvec,
                                   g[0], g[1])
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(saved) == 0
    assert torch.equal(ti, yi) and torch.equal(tt, yt)
    for s in range(2):
        # the MLP branch and the output projection come before the attention backward: bit-equal
        for n in ("w_1", "b_1", "w_2", "b_2", "w_o", "b_o"):
            assert torch.equal(g[s][n], ref_g[s][n]), n
        for n in NAMES:
            _close(g[s][n], ref_g[s][n], f"stream {s} {n}")
        _close(dx[s].float(), ref_dx[s].float(), f"dx stream {s}", rel=1e-2)  # a bf16 rounding may flip
    _close(dvec, ref_dvec, "dvec")
    # single block
    sc = BlockCase(1, 64, 16, 256, 2, 1024, "bf16", seed=79, std=0.05, lat_hw=(8, 8), single=True)
    x = dev(sc.x_joint())
    dy = dev(_dy(sc, rng, sc.x_joint().shape))
    cos1, sin1 = _rope(sc)
    w = upload_weights(sc.w_img, "bf16")
    y = torch.empty_like(x)
    L.mmdit_single_block_fwd(sc.dims, w, dev(sc.vec), cos1, sin1, x, y)
    rdx, rg = torch.empty_like(x), _grads_like(sc.w_img)
    L.mmdit_single_block_bwd(sc.dims, w, dev(sc.vec), cos1, sin1, x, dy, rdx, None, rg)
    ty = torch.full_like(x, float("nan"))
    saved1 = L.mmdit_single_block_fwd_train(sc.dims, w, dev(sc.vec), cos1, sin1, x, ty)
    tdx, tg = torch.empty_like(x), _grads_like(sc.w_img)
    L.mmdit_single_block_bwd_saved(sc.dims, w, dev(sc.vec), cos1, sin1, x, dy, tdx, saved1, None, tg)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(saved1) == 0
    assert torch.equal(ty, y)
    for n in NAMES:
        _close(tg[n], rg[n], f"single {n}")
