"""The conditioning vector, the all-blocks modulation launch and the whole-model forward
through the C ABI, against the oracle on the same seeded inputs.

* conditioning: vec = timestep MLP(sinusoid(1000 t)) + vector MLP(y) (+ guidance term), bf16
  and fp32, with and without guidance, batch 1 and 3;
* mmdit_modulation_batched_fwd over 85 jobs of two row counts (more than one launch's worth)
  equals the per-job modulation bit for bit;
* the whole model at a small width (D 256, 2 heads, 2 double + 2 single blocks, 8 x 8 latents,
  16 text tokens), batch 1 (the streams inside the joint buffer) and batch 2 (joined by copies),
  bf16 against the bf16-autocast oracle over nine seeds and fp32 against the float64 oracle,
  within 2e-2 x RMS;
* the model with parallel-branch single blocks at the small width;
* a full-width stack (D 3072, 2 double + 2 single blocks, both single-block forms, 1024 + 512
  tokens) with every gate active, against the oracle's whole forward;
* the 12B stack at 512 px (19 double + 38 single blocks, 1024 + 512 tokens) with every gate at
  zero: the blocks pass the residual stream through, so the prediction is the output head of the
  embedded latents, which the oracle computes at full size.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

from gpu_util import assert_parity, dev, host, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _up(w, act):
    """Device copy of a (nested) weight structure of float32 arrays."""
    if isinstance(w, dict):
        return {k: _up(v, act) for k, v in w.items()}
    if isinstance(w, (list, tuple)):
        return type(w)(_up(v, act) for v in w)
    return dev(w, torch_dtype(act))


@pytest.mark.parametrize("act,D", [("bf16", 3072), ("f32", 256)])
@pytest.mark.parametrize("B,guided", [(1, False), (3, True)])
def test_conditioning_matches_oracle(act, D, B, guided):
    rng = np.random.default_rng(40 + B)
    cast = "f32" if act == "f32" else "bf16"
    w = {"time_in": synth.mlp_embedder_weights(rng, 256, D, cast, 0.05),
         "vector_in": synth.mlp_embedder_weights(rng, 768, D, cast, 0.05)}
    if guided:
        w["guidance_in"] = (synth.bf16_round(rng.standard_normal(D).astype(np.float32) * 0.1),
                            synth.bf16_round(rng.standard_normal(D).astype(np.float32) * 0.1))
    t = synth.timesteps(rng, B, "uniform")
    y = synth.bf16_round(rng.standard_normal((B, 768)).astype(np.float32))
    g = np.linspace(1.0, 4.0, B).astype(np.float32) if guided else None
    vec = torch.empty(B, D, device="cuda", dtype=torch_dtype(act))
    ws = L.mmdit_conditioning_fwd(dev(t, torch.float32), dev(y, torch_dtype(act)), _up(w, act), vec,
                                  guidance=None if g is None else dev(g, torch.float32))
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    mm = O.round_bf16 if act == "bf16" else None
    ref = O.conditioning_vec(t, y, w, g, mm_cast=mm)
    assert_parity(host(vec), ref, 2e-2, f"conditioning {act} B={B}", out_bf16=act == "bf16")
    if act == "f32":
        assert_parity(host(vec), ref, 1e-4, "conditioning f32 (tight)")


def test_batched_modulation_equals_per_job_modulation():
    rng = np.random.default_rng(7)
    B, D = 3, 512
    vec = dev(synth.bf16_round(rng.standard_normal((B, D)).astype(np.float32)))
    jobs, singles = [], []
    for i in range(85):
        rows = 6 * D if i % 3 else 2 * D
        w = torch.randn(rows, D, device="cuda").mul_(0.02).to(torch.bfloat16)
        b = torch.randn(rows, device="cuda").mul_(0.02).to(torch.bfloat16)
        jobs.append((w, b, torch.full((B, rows), float("nan"), device="cuda")))
        singles.append(torch.empty(B, rows, device="cuda"))
    L.mmdit_modulation_batched_fwd(vec, jobs)
    for (w, b, _), out in zip(jobs, singles):
        L.mmdit_modulation_fwd(vec, w, b, out)
    torch.cuda.synchronize()
    for (_, _, got), exp in zip(jobs, singles):
        assert torch.equal(got, exp)
    # and one job against the oracle
    w, b, got = jobs[4]
    ref = O.modulation(host(vec), host(w), host(b), 6, mm_cast=O.round_bf16)
    assert_parity(host(got), np.concatenate(ref, axis=-1), 2e-2, "batched modulation")


def _small_model(B, act, seed):
    rng = np.random.default_rng(seed)
    cast = "f32" if act == "f32" else "bf16"
    D, H, F, lat, S_t, txt_dim = 256, 2, 1024, 8, 16, 64
    w = synth.flux_weights(rng, D, H, F, 2, 2, txt_dim=txt_dim, vec_dim=64, dtype=cast, std=0.05)
    z = rng.standard_normal((B, 64, lat, lat)).astype(np.float32)
    txt = synth.bf16_round(rng.standard_normal((B, S_t, txt_dim)).astype(np.float32))
    t = synth.timesteps(rng, B, "uniform")
    y = synth.bf16_round(rng.standard_normal((B, 64)).astype(np.float32))
    ids = synth.position_ids(B, lat, lat, S_t)
    return w, z, txt, t, y, ids, (D, H, F, lat, S_t, txt_dim)


def _run_model(w, z, txt, t, y, ids, shape, B, act, n_double, n_single, guidance=None, single_parallel=False):
    D, H, F, lat, S_t, txt_dim = shape
    S = lat * lat + S_t
    cos = torch.empty(B, S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(torch.from_numpy(ids).cuda(), (16, 56, 56), 10000.0, cos, sin)
    dims = L.make_dims(B, lat * lat, S_t, D, H, F, L.MMDIT_BF16 if act == "bf16" else L.MMDIT_F32)
    cfg = L.make_flux_config(dims, n_double, n_single, lat, lat, 64, txt_dim, 256, y.shape[1],
                             single_parallel=single_parallel)
    pred = torch.empty(B, 64, lat, lat, device="cuda")
    ws = L.mmdit_flux_forward(cfg, w, dev(z, torch.float32), dev(txt, torch_dtype(act)), dev(t, torch.float32),
                              dev(y, torch_dtype(act)), cos, sin, pred, guidance=guidance)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    return host(pred)


# Seeds of the whole-model case: every one drawn is kept (5678 is the one that came out at
# 2.057e-2 x RMS while the embedders' hidden layer was stored in bf16).
MODEL_SEEDS = [(1, 61), (1, 5678), (1, 1), (1, 2), (1, 3), (1, 4), (2, 62), (2, 5), (2, 6)]


@pytest.mark.parametrize("B,seed", MODEL_SEEDS)
def test_small_model_matches_oracle_bf16(B, seed):
    w, z, txt, t, y, ids, shape = _small_model(B, "bf16", seed)
    got = _run_model(_up(w, "bf16"), z, txt, t, y, ids, shape, B, "bf16", 2, 2)
    ref = O.flux_forward(z, txt, t, y, ids, w, shape[1], mm_cast=O.round_bf16, store=O.round_bf16)
    e = assert_parity(got, ref, 2e-2, f"whole model bf16 B={B} seed {seed}")
    print(f"[model] bf16 B={B} seed {seed}: max|err|/RMS vs bf16-autocast oracle = {e:.3e}")


@pytest.mark.parametrize("B", [1, 2])
def test_small_model_matches_oracle_f32(B):
    w, z, txt, t, y, ids, shape = _small_model(B, "f32", 60 + B)
    got = _run_model(_up(w, "f32"), z, txt, t, y, ids, shape, B, "f32", 2, 2)
    ref = O.flux_forward(z, txt, t, y, ids, w, shape[1])
    assert_parity(got, ref, 2e-2, f"whole model f32 B={B}")


@pytest.mark.parametrize("B", [1, 2])
def test_small_model_with_parallel_single_blocks_matches_oracle(B):
    """The whole model with parallel-branch single blocks (the form whose parameter count matches
    the API reference's ~535 M / ~12 B), against the oracle's flux_forward(single_parallel=True)."""
    rng = np.random.default_rng(80 + B)
    D, H, F, lat, S_t, txt_dim = 256, 2, 1024, 8, 16, 64
    w = synth.flux_weights(rng, D, H, F, 2, 2, txt_dim=txt_dim, vec_dim=64, dtype="bf16", std=0.05,
                           single_parallel=True)
    z = rng.standard_normal((B, 64, lat, lat)).astype(np.float32)
    txt = synth.bf16_round(rng.standard_normal((B, S_t, txt_dim)).astype(np.float32))
    t = synth.timesteps(rng, B, "uniform")
    y = synth.bf16_round(rng.standard_normal((B, 64)).astype(np.float32))
    ids = synth.position_ids(B, lat, lat, S_t)
    got = _run_model(_up(w, "bf16"), z, txt, t, y, ids, (D, H, F, lat, S_t, txt_dim), B, "bf16", 2, 2,
                     single_parallel=True)
    ref = O.flux_forward(z, txt, t, y, ids, w, H, mm_cast=O.round_bf16, store=O.round_bf16,
                         single_parallel=True)
    e = assert_parity(got, ref, 2e-2, f"whole model, parallel single blocks, B={B}")
    print(f"[model] parallel single blocks B={B}: max|err|/RMS = {e:.3e}")
    # the switch reaches the single blocks: without them the prediction differs
    seq = O.flux_forward(z, txt, t, y, ids, dict(w, single=[]), H, mm_cast=O.round_bf16, store=O.round_bf16)
    assert np.abs(got - seq).max() > 1e-3


def test_small_model_without_single_blocks_and_text():
    # no single blocks: the head reads the double blocks' image stream directly
    w, z, txt, t, y, ids, shape = _small_model(2, "bf16", 71)
    w["single"] = []
    got = _run_model(_up(w, "bf16"), z, txt, t, y, ids, shape, 2, "bf16", 2, 0)
    ref = O.flux_forward(z, txt, t, y, ids, w, shape[1], mm_cast=O.round_bf16, store=O.round_bf16)
    assert_parity(got, ref, 2e-2, "whole model, double blocks only")


@pytest.mark.parametrize("single_parallel", [False, True])
def test_full_width_stack_matches_oracle(single_parallel):
    """A non-trivial stack at the 12B block width: D 3072, 24 heads, F 12288, 2 double + 2 single
    blocks (sequential or parallel-branch) at 32 x 32 latents and 512 text tokens, batch 1,
    against the oracle's whole forward at the bf16-autocast precision (every gate active)."""
    B, lat, S_t, D, H, F, txt_dim = 1, 32, 512, 3072, 24, 12288, 4096
    rng = np.random.default_rng(3000 + single_parallel)
    w = synth.flux_weights(rng, D, H, F, 2, 2, txt_dim=txt_dim, vec_dim=768, dtype="bf16", std=0.02,
                           single_parallel=single_parallel)
    z = rng.standard_normal((B, 64, lat, lat)).astype(np.float32)
    txt = synth.bf16_round(rng.standard_normal((B, S_t, txt_dim)).astype(np.float32))
    t = synth.timesteps(rng, B, "uniform")
    y = synth.bf16_round(rng.standard_normal((B, 768)).astype(np.float32))
    ids = synth.position_ids(B, lat, lat, S_t)
    got = _run_model(_up(w, "bf16"), z, txt, t, y, ids, (D, H, F, lat, S_t, txt_dim), B, "bf16", 2, 2,
                     single_parallel=single_parallel)
    ref = O.flux_forward(z, txt, t, y, ids, w, H, mm_cast=O.round_bf16, store=O.round_bf16,
                         single_parallel=single_parallel)
    # 3e-2: at the 12B width a numpy emulation of the GPU's roundings alone (fp32 accumulation,
    # bf16 storage of every tensor the GPU stores in bf16, fp16 softmax weights) sits 2.2-2.7e-2
    # x RMS from the bf16-autocast oracle per block on the benchmark's inputs (2.07e-2 with exact
    # softmax weights); the small-width model above holds 2e-2
    e = assert_parity(got, ref, 3e-2, f"full-width stack (parallel={single_parallel})")
    print(f"[model] full-width 2 + 2 stack, parallel={single_parallel}: max|err|/RMS = {e:.3e}")


def _zero_gate_rows(w_mod, b_mod, D):
    for c in (2, 5):
        w_mod[c * D:(c + 1) * D] = 0
        b_mod[c * D:(c + 1) * D] = 0


def test_12b_stack_at_512px_with_zero_gates_is_the_head_of_the_embedded_latents():
    B, lat, S_t, D, H, F, txt_dim = 1, 32, 512, 3072, 24, 12288, 4096
    rng = np.random.default_rng(1002)
    # small weights (embedders, head) from numpy for the oracle; block weights drawn on the device
    w_small = {"img_in": tuple(synth.embed_weights(rng, 64, D).values()),
               "txt_in": tuple(synth.embed_weights(rng, txt_dim, D).values()),
               "time_in": synth.mlp_embedder_weights(rng, 256, D),
               "vector_in": synth.mlp_embedder_weights(rng, 768, D),
               "final": synth.final_layer_weights(rng, D, 64)}
    w = _up(w_small, "bf16")
    gen = torch.Generator(device="cuda").manual_seed(2002)

    def stream():
        def n(*shape):
            return (torch.randn(*shape, device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
        s = {"w_mod": n(6 * D, D), "b_mod": n(6 * D), "w_qkv": n(3 * D, D), "b_qkv": n(3 * D),
             "g_q": torch.ones(128, device="cuda", dtype=torch.bfloat16),
             "g_k": torch.ones(128, device="cuda", dtype=torch.bfloat16),
             "w_o": n(D, D), "b_o": n(D), "w_1": n(F, D), "b_1": n(F), "w_2": n(D, F), "b_2": n(D)}
        _zero_gate_rows(s["w_mod"], s["b_mod"], D)
        return s

    w["double"] = [(stream(), stream()) for _ in range(19)]
    w["single"] = [stream() for _ in range(38)]
    z = rng.standard_normal((B, 64, lat, lat)).astype(np.float32)
    txt = synth.bf16_round(rng.standard_normal((B, S_t, txt_dim)).astype(np.float32))
    t = synth.timesteps(rng, B, "uniform")
    y = synth.bf16_round(rng.standard_normal((B, 768)).astype(np.float32))
    ids = synth.position_ids(B, lat, lat, S_t)
    got = _run_model(w, z, txt, t, y, ids, (D, H, F, lat, S_t, txt_dim), B, "bf16", 19, 38)
    vec = O.round_bf16(O.conditioning_vec(t, y, w_small, mm_cast=O.round_bf16))
    x_img = O.round_bf16(O.img_in(z, *w_small["img_in"], mm_cast=O.round_bf16))
    f = w_small["final"]
    ref = O.final_layer(x_img, vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], lat, lat, mm_cast=O.round_bf16)
    assert_parity(got, ref, 2e-2, "12B stack with zero gates")
