"""GPU parity of the individual entry points against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

from gpu_util import assert_parity, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


# ----------------------------------------------------------------------------- RoPE tables
@pytest.mark.parametrize("B,H,W,S_t", [(2, 8, 12, 20), (1, 128, 128, 512), (1, 1, 1, 0)])
def test_rope3d_tables(B, H, W, S_t):
    ids = synth.position_ids(B, H, W, S_t)
    ids[..., 0] = np.arange(ids.shape[1]) % 7  # exercise axis 0 too
    c_ref, s_ref = O.rope_cos_sin(ids)
    t_ids = torch.from_numpy(ids).cuda()
    cos = torch.empty(B, ids.shape[1], 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(t_ids, (16, 56, 56), 10000.0, cos, sin)
    torch.cuda.synchronize()
    assert np.abs(host(cos) - c_ref).max() < 2e-5
    assert np.abs(host(sin) - s_ref).max() < 2e-5


# ----------------------------------------------------------------------------- flow matching
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(3, 64, 20, 20), (4, 64, 32, 32), (1, 8, 1, 1)])
def test_flow_match_noise_and_loss(dtype, shape):
    rng = np.random.default_rng(5)
    z0, z1 = synth.latent_pair(rng, *shape)
    t = synth.timesteps(rng, shape[0], "logit_normal")
    pred = rng.standard_normal(shape).astype(np.float32)
    if dtype == torch.bfloat16:
        z0, z1, pred = synth.bf16_round(z0), synth.bf16_round(z1), synth.bf16_round(pred)
    d0, d1, dp = dev(z0, dtype), dev(z1, dtype), dev(pred, dtype)
    dt = torch.from_numpy(t).cuda()
    zt = torch.empty_like(d0)
    loss = torch.zeros(1, device="cuda")
    L.flow_match_noise_and_loss(d0, d1, dt, z_t=zt, pred=dp, loss=loss)
    torch.cuda.synchronize()
    ref_zt = O.flow_match_noise(z0, z1, t)
    # fp32 arithmetic: a few ulp of the inputs' magnitude; bf16 output: plus half an ulp of z_t
    bound = 2.0 ** -21 * (np.abs(z0) + np.abs(z1))
    if dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(ref_zt)
    assert np.all(np.abs(host(zt) - ref_zt) <= bound + 1e-30)
    ref_loss = O.flow_match_loss(pred, z0, z1)
    assert abs(loss.item() - ref_loss) <= 1e-4 * ref_loss
    # loss only, then noise only; the loss is deterministic call to call
    loss2 = torch.zeros(1, device="cuda")
    L.flow_match_noise_and_loss(d0, d1, dt, pred=dp, loss=loss2)
    zt2 = torch.zeros_like(d0)
    L.flow_match_noise_and_loss(d0, d1, dt, z_t=zt2)
    torch.cuda.synchronize()
    assert loss2.item() == loss.item()
    assert torch.equal(zt2, zt)


def test_flow_match_endpoints_on_gpu():
    rng = np.random.default_rng(6)
    z0, z1 = synth.latent_pair(rng, 2, 64, 8, 8)
    d0, d1 = dev(z0, torch.float32), dev(z1, torch.float32)
    zt = torch.empty_like(d0)
    L.flow_match_noise_and_loss(d0, d1, torch.tensor([0.0, 1.0], device="cuda"), z_t=zt)
    torch.cuda.synchronize()
    assert torch.equal(zt[0], d0[0]) and torch.equal(zt[1], d1[1])
    loss = torch.zeros(1, device="cuda")
    L.flow_match_noise_and_loss(d0, d1, torch.zeros(2, device="cuda"), pred=d1 - d0, loss=loss)
    torch.cuda.synchronize()
    assert loss.item() == 0.0


# ----------------------------------------------------------------------------- modulation GEMV
@pytest.mark.parametrize("act,B,rows,dim", [("bf16", 1, 6 * 3072, 3072), ("bf16", 3, 6 * 256, 256),
                                            ("bf16", 9, 2 * 512, 512), ("f32", 2, 6 * 256, 256)])
def test_modulation_matches_oracle(act, B, rows, dim):
    """SiLU(vec) w^T + b in fp32 accumulation; in bf16 mode SiLU(vec) is a bf16 operand of the
    linear (autocast), so the oracle at that precision is the reference.  Batch 9 runs two
    passes of the kernel (at most 8 batch rows each)."""
    rng = np.random.default_rng(rows + B)
    cast = synth.bf16_round if act == "bf16" else (lambda a: a.astype(np.float32))
    vec = cast(rng.standard_normal((B, dim)).astype(np.float32))
    w = cast((rng.standard_normal((rows, dim)) * 0.02).astype(np.float32))
    b = cast((rng.standard_normal(rows) * 0.02).astype(np.float32))
    t = torch.bfloat16 if act == "bf16" else torch.float32
    out = torch.empty(B, rows, device="cuda")
    L.mmdit_modulation_fwd(dev(vec, t), dev(w, t), dev(b, t), out)
    torch.cuda.synchronize()
    ref = np.concatenate(O.modulation(vec, w, b, n_chunks=1, mm_cast=O.round_bf16 if act == "bf16" else None),
                         axis=-1)
    # only the order of the fp32 accumulation differs from the oracle at the same precision
    assert_parity(host(out), ref, 1e-4, f"modulation {act} B={B} rows={rows}")


# ----------------------------------------------------------------------------- linear (GEMM core)
@pytest.mark.parametrize("act,M,N,K", [
    ("bf16", 300, 96, 200),      # ragged M, 32-wide tiles, K tail
    ("bf16", 257, 768, 3072),    # 256-wide tiles, several K slices
    ("bf16", 512, 3072, 4096),   # txt_in shape
    ("bf16", 4096, 64, 3072),    # narrow N
    ("f32", 130, 256, 72),       # tf32 path
    ("f32", 33, 1024, 256),
])
def test_linear_matches_oracle(act, M, N, K):
    rng = np.random.default_rng(M + N + K)
    cast = synth.bf16_round if act == "bf16" else (lambda a: a.astype(np.float32))
    x = cast(rng.standard_normal((M, K)).astype(np.float32))
    w = cast((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    b = cast((rng.standard_normal(N) * 0.05).astype(np.float32))
    t = torch.bfloat16 if act == "bf16" else torch.float32
    y = torch.empty(M, N, device="cuda", dtype=t)
    ws = L.mmdit_linear_fwd(dev(x, t), dev(w, t), dev(b, t), y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    tol = 2e-2 if act == "bf16" else 5e-3
    assert_parity(host(y), O.linear(x, w, b), tol, f"linear {act} {M}x{N}x{K}", out_bf16=act == "bf16")


# ----------------------------------------------------------------------------- attention
@pytest.mark.parametrize("B,H,S,qscale", [(1, 1, 1, 1.0), (2, 3, 128, 1.0), (2, 2, 300, 1.0),
                                         (1, 2, 1000, 6.0), (1, 24, 4608, 1.0)])
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_attention_matches_oracle(B, H, S, qscale, act):
    if act == "f32" and S > 1000:
        pytest.skip("one large case is enough")
    rng = np.random.default_rng(S + H)
    q = synth.bf16_round(rng.standard_normal((B, H, S, 128)).astype(np.float32) * qscale)
    k = synth.bf16_round(rng.standard_normal((B, H, S, 128)).astype(np.float32))
    v = synth.bf16_round(rng.standard_normal((B, H, S, 128)).astype(np.float32))
    t = torch.bfloat16 if act == "bf16" else torch.float32
    out = torch.empty(B, S, H * 128, device="cuda", dtype=t)
    ws = L.mmdit_attention_fwd(dev(q), dev(k), dev(v), out)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    # q, k, v are bf16 already; the bf16-autocast oracle keeps the softmax weights exact
    rows = np.random.default_rng(0).choice(S, 200, replace=False) if S > 1000 else np.arange(S)
    ref = O.attention(q[:, :, rows], k, v, O.round_bf16).transpose(0, 2, 1, 3).reshape(B, len(rows), H * 128)
    ref64 = O.attention(q[:, :, rows], k, v).transpose(0, 2, 1, 3).reshape(B, len(rows), H * 128)
    got = host(out)[:, rows]
    assert_parity(got, ref, 2e-2, f"attention B={B} H={H} S={S}", out_bf16=act == "bf16")
    assert_parity(got, ref64, 5e-2, f"attention B={B} H={H} S={S} vs float64")


@pytest.mark.parametrize("vscale", [6e4, 2.0 ** -10])
def test_attention_v_at_the_ends_of_its_fp16_range(vscale):
    """The PV product reads V in fp16 (the header states the range): V uniform in +-60000 (close to
    fp16's largest finite 65504) and V near 2^-10 (above fp16's smallest normal) both meet the bar
    against the oracle, which keeps V exact."""
    B, H, S = 1, 2, 700
    rng = np.random.default_rng(int(vscale) + 5)
    q = synth.bf16_round(rng.standard_normal((B, H, S, 128)).astype(np.float32))
    k = synth.bf16_round(rng.standard_normal((B, H, S, 128)).astype(np.float32))
    v = synth.bf16_round((rng.uniform(-1.0, 1.0, (B, H, S, 128)) * vscale).astype(np.float32))
    out = torch.empty(B, S, H * 128, device="cuda", dtype=torch.bfloat16)
    ws = L.mmdit_attention_fwd(dev(q), dev(k), dev(v), out)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    got = host(out)
    assert np.isfinite(got).all()
    ref = O.attention(q, k, v, O.round_bf16).transpose(0, 2, 1, 3).reshape(B, S, H * 128)
    assert_parity(got, ref, 2e-2, f"attention with |V| up to {vscale:g}", out_bf16=True)


# ----------------------------------------------------------------------------- embeddings / head
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_img_in_matches_oracle(act):
    rng = np.random.default_rng(8)
    B, Cc, Hh, Ww, D = 2, 64, 10, 12, 256
    z = rng.standard_normal((B, Cc, Hh, Ww)).astype(np.float32)
    cast = "bf16" if act == "bf16" else "f32"
    e = synth.embed_weights(rng, Cc, D, cast, std=0.1)
    t = torch.bfloat16 if act == "bf16" else torch.float32
    out = torch.empty(B, Hh * Ww, D, device="cuda", dtype=t)
    ws = L.mmdit_img_in_fwd(dev(z, torch.float32), dev(e["w"], t), dev(e["b"], t), out)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    zr = synth.bf16_round(z) if act == "bf16" else z  # tokens are held in the activation type
    assert_parity(host(out), O.img_in(zr, e["w"], e["b"]), 2e-2, "img_in", out_bf16=act == "bf16")


@pytest.mark.parametrize("act", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hh,Ww,D", [(2, 10, 12, 256), (1, 32, 32, 1024)])  # the second splits K
def test_final_layer_matches_oracle(act, B, Hh, Ww, D):
    rng = np.random.default_rng(9)
    Cc = 64
    cast = "bf16" if act == "bf16" else "f32"
    rnd = synth.bf16_round if act == "bf16" else (lambda a: a)
    x = rnd(rng.standard_normal((B, Hh * Ww, D)).astype(np.float32))
    vec = rnd(rng.standard_normal((B, D)).astype(np.float32))
    f = synth.final_layer_weights(rng, D, Cc, cast, std=0.1)
    t = torch.bfloat16 if act == "bf16" else torch.float32
    dims = L.make_dims(B, Hh * Ww, 0, D, D // 128, 4 * D, L.MMDIT_BF16 if act == "bf16" else L.MMDIT_F32)
    pred = torch.empty(B, Cc, Hh, Ww, device="cuda")
    ws = L.mmdit_final_layer_fwd(dims, Hh, Ww, dev(x, t), dev(vec, t), dev(f["w_ada"], t),
                                 dev(f["b_ada"], t), dev(f["w_out"], t), dev(f["b_out"], t), pred)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    cast = O.round_bf16 if act == "bf16" else None
    ref = O.final_layer(x, vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], Hh, Ww, mm_cast=cast)
    assert_parity(host(pred), ref, 2e-2, "final layer")


@pytest.mark.parametrize("act", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hh,Ww", [(2, 10, 12), (4, 32, 32)])
def test_img_in_noise_matches_oracle(act, B, Hh, Ww):
    """img_in of z_t formed while patchifying: z_t bit-equal to the standalone noise pass, the
    embedding against the oracle's img_in of the oracle's z_t."""
    rng = np.random.default_rng(18 + B)
    Cc, D = 64, 256
    z0, z1 = synth.latent_pair(rng, B, Cc, Hh, Ww)
    tt = synth.timesteps(rng, B, "logit_normal")
    cast = "bf16" if act == "bf16" else "f32"
    e = synth.embed_weights(rng, Cc, D, cast, std=0.1)
    t = torch.bfloat16 if act == "bf16" else torch.float32
    d0, d1, dt = dev(z0, torch.float32), dev(z1, torch.float32), dev(tt, torch.float32)
    out = torch.empty(B, Hh * Ww, D, device="cuda", dtype=t)
    zt = torch.full_like(d0, float("nan"))
    ws = L.mmdit_img_in_noise_fwd(d0, d1, dt, dev(e["w"], t), dev(e["b"], t), out, z_t=zt)
    zt_ref = torch.empty_like(d0)
    L.flow_match_noise_and_loss(d0, d1, dt, z_t=zt_ref)
    out_ref = torch.empty_like(out)
    L.mmdit_img_in_fwd(zt_ref, dev(e["w"], t), dev(e["b"], t), out_ref)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    assert torch.equal(zt, zt_ref), "z_t differs from the standalone noise pass"
    assert torch.equal(out, out_ref), "embedding differs from img_in of the same z_t"
    ztr = O.flow_match_noise(z0, z1, tt)
    assert_parity(host(zt), ztr, 1e-6, "z_t")
    zr = synth.bf16_round(ztr.astype(np.float32)) if act == "bf16" else ztr
    assert_parity(host(out), O.img_in(zr, e["w"], e["b"]), 2e-2, "img_in of z_t", out_bf16=act == "bf16")


@pytest.mark.parametrize("act", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hh,Ww,D", [(2, 10, 12, 256), (1, 32, 32, 1024), (4, 32, 32, 256),
                                       (1, 128, 128, 256)])  # split K, and the last one does not
def test_final_layer_loss_matches_oracle(act, B, Hh, Ww, D):
    """The output head with the loss fused on: pred equal to the plain head's, the loss within
    1e-5 of the oracle's MSE of that pred, and pred against the oracle's head; two calls in a row
    (the finishing kernel's ticket counter resets itself) give bit-equal losses."""
    rng = np.random.default_rng(19 + Hh)
    Cc = 64
    cast = "bf16" if act == "bf16" else "f32"
    rnd = synth.bf16_round if act == "bf16" else (lambda a: a)
    x = rnd(rng.standard_normal((B, Hh * Ww, D)).astype(np.float32))
    vec = rnd(rng.standard_normal((B, D)).astype(np.float32))
    f = synth.final_layer_weights(rng, D, Cc, cast, std=0.1)
    z0, z1 = synth.latent_pair(rng, B, Cc, Hh, Ww)
    t = torch.bfloat16 if act == "bf16" else torch.float32
    dims = L.make_dims(B, Hh * Ww, 0, D, D // 128, 4 * D, L.MMDIT_BF16 if act == "bf16" else L.MMDIT_F32)
    args = (dev(x, t), dev(vec, t), dev(f["w_ada"], t), dev(f["b_ada"], t), dev(f["w_out"], t),
            dev(f["b_out"], t))
    d0, d1 = dev(z0, torch.float32), dev(z1, torch.float32)
    pred = torch.full((B, Cc, Hh, Ww), float("nan"), device="cuda")
    loss = torch.full((2,), float("nan"), device="cuda")
    ws = L.mmdit_final_layer_loss_fwd(dims, Hh, Ww, *args, d0, d1, loss[0:1], pred=pred)
    L.mmdit_final_layer_loss_fwd(dims, Hh, Ww, *args, d0, d1, loss[1:2], ws=ws)  # no pred written
    pred_ref = torch.empty_like(pred)
    L.mmdit_final_layer_fwd(dims, Hh, Ww, *args, pred_ref)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    assert torch.equal(pred, pred_ref), "pred differs from the plain output head's"
    lv = loss.cpu().numpy()
    assert lv[0] == lv[1], f"two calls gave {lv[0]} and {lv[1]}"
    ref_loss = O.flow_match_loss(host(pred), z0, z1)
    assert abs(lv[0] - ref_loss) <= 1e-5 * ref_loss, (lv[0], ref_loss)
    mm = O.round_bf16 if act == "bf16" else None
    ref = O.final_layer(x, vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], Hh, Ww, mm_cast=mm)
    assert_parity(host(pred), ref, 2e-2, "final layer (loss variant)")
    # against the oracle head's own loss: the prediction's rounding moves the MSE by about twice
    # the relative error of the prediction (bf16 operands at the autocast precision; tf32 operands,
    # 2^-11 relative, against the pure float64 head for f32)
    ref_loss64 = O.flow_match_loss(ref, z0, z1)
    tol = 1e-3 if act == "bf16" else 5e-3
    assert abs(lv[0] - ref_loss64) <= tol * ref_loss64, (lv[0], ref_loss64)


@pytest.mark.parametrize("xdt,odt", [("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("B,R,D", [(2, 300, 3072), (1, 7, 8192), (3, 65, 256)])
def test_ln_modulate_matches_oracle(xdt, odt, B, R, D):
    rng = np.random.default_rng(B * R + D)
    x = rng.standard_normal((B, R, D)).astype(np.float32) * 3.0 + 0.5
    if xdt == "bf16":
        x = synth.bf16_round(x)
    mod = (rng.standard_normal((B, 6 * D)) * 0.3).astype(np.float32)  # [shift | scale | ...] per sample
    gx = dev(x, torch.bfloat16 if xdt == "bf16" else torch.float32)
    out = torch.empty(B, R, D, device="cuda", dtype=torch.bfloat16 if odt == "bf16" else torch.float32)
    gm = dev(mod, torch.float32)
    L.mmdit_ln_modulate_fwd(gx, gm[:, :D], gm[:, D:2 * D], out, 6 * D)
    torch.cuda.synchronize()
    ref = O.modulate(x, mod[:, :D], mod[:, D:2 * D])
    tol = 2e-2 if odt == "bf16" else 1e-5
    assert_parity(host(out), ref, tol, f"LayerNorm-modulate {xdt}->{odt}", out_bf16=odt == "bf16")


# ----------------------------------------------------------------------------- sampling step
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n,guided,inplace", [(8, True, False), (8 * 1001, False, False),
                                              (262144, True, True)])
def test_euler_cfg_step_matches_oracle(dtype, n, guided, inplace):
    rng = np.random.default_rng(n + guided)
    cast = synth.bf16_round if dtype == torch.bfloat16 else (lambda a: a.astype(np.float32))
    z, vc, vu = (cast(rng.standard_normal(n).astype(np.float32)) for _ in range(3))
    w, dt = 3.5, 0.05
    gz, gvc = dev(z, dtype), dev(vc, dtype)
    gvu = dev(vu, dtype) if guided else None
    out = gz if inplace else torch.empty_like(gz)
    L.flow_match_euler_step(gz, gvc, gvu, w, dt, out)
    torch.cuda.synchronize()
    ref = O.euler_step(z, O.cfg_combine(vc, vu, w) if guided else vc, dt)
    # fp32 arithmetic, then the output's own rounding
    assert_parity(host(out), ref, 1e-6, f"Euler step n={n}", out_bf16=dtype == torch.bfloat16)


def test_euler_steps_follow_the_straight_line_flow_on_gpu():
    """Ten Euler steps of 0.1 from z1 along v = z1 - z0 land on z0 (Euler is exact there)."""
    rng = np.random.default_rng(17)
    z0, z1 = synth.latent_pair(rng, 2, 64, 16, 16)
    v = dev((z1 - z0).astype(np.float32), torch.float32)
    z = dev(z1, torch.float32)
    for _ in range(10):
        L.flow_match_euler_step(z, v, None, 1.0, 0.1, z)
    torch.cuda.synchronize()
    assert_parity(host(z), z0, 1e-5, "z after ten Euler steps")
