#!/usr/bin/env python3
"""Benchmark of the Flux MMDiT block forward hot path on GB300 (one process per GPU).

One step is one pass of the whole hot path on the 535M-shaped Flux workload (hidden 3072,
24 heads x 128, MLP 12288, 4096 image tokens from 64x64x64 latents + 512 text tokens from a
[1, 512, 4096] text embedding, batch 1):

    rope3d_freqs -> img_in of z_t (the flow-matching noise formed while patchifying) -> txt_in
    -> double block -> single block -> output head with the flow-matching loss fused on

all through the C ABI of libmmdit.so, with inputs resident in HBM when the timed region
starts (``value``) or copied from pinned host memory inside it (``e2e``).  Other workloads:
the same step at batch 2 with 4096 + 512 tokens (the metric's second point), the double block
at batch 4 with 1024 + 512 tokens, the blocks at 16384 + 512 tokens with E4M3 linears, and the
whole Flux 12B forward.  Every AdaLN modulation of the step (the blocks' and the output head's)
is computed first, in one batched GEMV launch (mmdit_modulation_batched_fwd).  The metric is the
dense-contraction throughput of the two blocks (2 * B * S * D * (3D + D + 2F) + 4 * B * S^2 *
d * H floating-point operations per block) divided by the time of the whole step, reported
in TFLOP/s and as a fraction of the measured bf16 tensor peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (the forward has no exchange step);
``value`` is the work of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MMDiT block fwd TFLOP/s & % of GB300 bf16 tensor peak at 4096+512 tokens"
WORKLOAD = "flux535m_bf16"
C3_WORKLOAD = "flux12b_512px_bf16"
C4_WORKLOAD = "flux12b_1024px_bf16"
FP8_WORKLOAD = "flux12b_2048px_fp8"
MODEL_WORKLOAD = "flux12b_512px_model"
AXES = (16, 56, 56)
THETA = 10000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=5)
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain per-call launches instead of a CUDA-graph replay of the step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time of the oracle baseline sample")
    ap.add_argument("--workload", choices=[WORKLOAD, C3_WORKLOAD, C4_WORKLOAD, FP8_WORKLOAD, MODEL_WORKLOAD],
                    default=WORKLOAD,
                    help=f"{WORKLOAD}: the hot-path step above (the headline); {C4_WORKLOAD}: the same "
                         "step at batch 2 with N(0, 1) text tokens of width D and logit-normal t (the "
                         f"metric's second point); {C3_WORKLOAD}: the double block alone at batch 4, "
                         f"1024 + 512 tokens, with the noise, output head and loss; {FP8_WORKLOAD}: the "
                         "double + single block at 16384 + 512 tokens with E4M3 linears; "
                         f"{MODEL_WORKLOAD}: the whole Flux 12B forward (19 double + 38 single "
                         "blocks) at 1024 + 512 tokens through mmdit_flux_forward")
    ap.add_argument("--fp8-recipe", choices=["delayed", "tensorwise", "blockwise", "mxfp8"], default="delayed",
                    help=f"the scaling recipe of the E4M3 linears in {FP8_WORKLOAD}: per-tensor delayed "
                         "scaling (the FP8 page's default), per-tensor current scaling, per-tile "
                         "current scaling (1 x 128 inputs, 128 x 128 weights), or MXFP8 (a power-of-two "
                         "scale per 32 elements along K; its products run on the bf16 tensor cores)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    return args


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(dist, x: float, device="cpu") -> float:
    """The largest of every rank's x (the slowest rank's time); x itself on one process."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, steps: int, world: int, seconds: float) -> float:
    """Work of all ranks (each runs the same step on its own replica) over the slowest time."""
    return world * flops_per_rank_step * steps / seconds / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured (MEASURED_PEAKS.json)"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- workload
def block_flops(B, S, D, F, H, d=128):
    return 2 * B * S * D * (3 * D + D + 2 * F) + 4 * B * S * S * d * H


class HostWorkload:
    """Seeded host-side inputs and weights (float32 arrays holding bf16-rounded values).  The text
    tokens are a [B, S_t, 4096] embedding fed through txt_in where the workload names that source,
    else N(0, 1) at width D (the block input itself)."""

    def __init__(self, wl):
        from diffusion_transformer_flux_gb300 import synth
        self.wl = wl
        B, D, H, F = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden
        rng_in = np.random.Generator(np.random.PCG64(1000 + wl.index))
        rng_w = np.random.Generator(np.random.PCG64(2000 + wl.index))
        self.z0, self.z1 = synth.latent_pair(rng_in, B, wl.channels, wl.lat_h, wl.lat_w)
        self.t = synth.timesteps(rng_in, B, wl.t_dist)
        txt_w = wl.ctx_dim if wl.txt_from_ctx else D
        self.txt = synth.bf16_round(rng_in.standard_normal((B, wl.seq_txt, txt_w), dtype=np.float32))
        self.vec = synth.bf16_round(rng_in.standard_normal((B, D), dtype=np.float32))
        self.ids = synth.position_ids(B, wl.lat_h, wl.lat_w, wl.seq_txt)
        self.img_in = synth.embed_weights(rng_w, wl.channels, D, "bf16")
        self.txt_in = synth.embed_weights(rng_w, wl.ctx_dim, D, "bf16") if wl.txt_from_ctx else None
        self.w_dimg = synth.stream_weights(rng_w, D, H, 128, F, "bf16")
        self.w_dtxt = synth.stream_weights(rng_w, D, H, 128, F, "bf16")
        self.has_single = "single" in wl.blocks
        self.w_single = synth.stream_weights(rng_w, D, H, 128, F, "bf16") if self.has_single else None
        self.final = synth.final_layer_weights(rng_w, D, wl.channels, "bf16")


class BatchedModulation:
    """Every AdaLN modulation of the step (the blocks' six-chunk modulations, the output head's shift
    and scale) in one launch at the start of the step, on the step's stream: they depend only on vec
    and the weights, and one launch streams the weights at close to the HBM rate.  (Run on a second
    stream beside the RoPE tables and the embeddings, the GEMV's blocks hold every SM while those
    short launches wait, and the pair took longer than the two in sequence.)  The blocks then read
    them through the weight sets' `mod` entries."""

    def __init__(self, torch, L, vec, weight_sets, device):
        self.torch, self.L, self.vec = torch, L, vec
        # [(name, w_mod, b_mod), ...] in the order the steps need them
        self.sets = weight_sets
        B = vec.shape[0]
        self.mods = {n: torch.empty(B, w.shape[0], device=device) for n, w, _ in weight_sets}

    def compute(self):
        self.L.mmdit_modulation_batched_fwd(self.vec, [(w, b, self.mods[n]) for n, w, b in self.sets])

    def weights(self, name, w):
        return dict(w, mod=self.mods[name])


class DeviceStep:
    """Device buffers, weights and workspaces of one replica, and the step itself."""

    def __init__(self, hw: HostWorkload, device, keep_pred=False):
        import torch
        from diffusion_transformer_flux_gb300 import _lib as L
        self.L, self.torch = L, torch
        wl = hw.wl
        self.wl = wl
        B, D, H, F, S_i, S_t = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden, wl.seq_img, wl.seq_txt
        S = S_i + S_t
        bf = torch.bfloat16

        def dev(a, dt=bf):
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device).to(dt)

        def devw(w):
            return {k: dev(v) for k, v in w.items()}

        self.z0, self.z1 = dev(hw.z0, torch.float32), dev(hw.z1, torch.float32)
        self.t = dev(hw.t, torch.float32)
        self.txt, self.vec = dev(hw.txt), dev(hw.vec)
        self.ids = dev(hw.ids, torch.float32)
        self.img_in = devw(hw.img_in)
        self.txt_in = devw(hw.txt_in) if hw.txt_in is not None else None
        self.w_dimg, self.w_dtxt = devw(hw.w_dimg), devw(hw.w_dtxt)
        self.w_single = devw(hw.w_single) if hw.has_single else None
        self.final = devw(hw.final)
        self.cos = torch.empty(B, S, 64, device=device)
        self.sin = torch.empty_like(self.cos)
        # Activations.  Batch 1: [img; txt] is one contiguous buffer per stage, so the double block's
        # streams are views of it and the single block reads it directly.  Batch > 1: the streams are
        # separate [B, S_s, D] buffers, joined into [B, S, D] (and the image rows taken back out) by
        # strided copies on the copy engine (mmdit_copy_rows).
        self.joint = B == 1
        if self.joint:
            self.X = torch.empty(B, S, D, device=device, dtype=bf)   # embeddings [img; txt]
            self.Y = torch.empty_like(self.X)                        # double-block output
            self.Z = torch.empty_like(self.X)                        # single-block output
            self.x_img, self.x_txt = self.X[:, :S_i], self.X[:, S_i:]
            self.y_img, self.y_txt = self.Y[:, :S_i], self.Y[:, S_i:]
        else:
            self.x_img = torch.empty(B, S_i, D, device=device, dtype=bf)
            self.x_txt = torch.empty(B, S_t, D, device=device, dtype=bf)
            self.y_img, self.y_txt = torch.empty_like(self.x_img), torch.empty_like(self.x_txt)
            # the single block's input and output, and the image rows the head reads
            self.C = torch.empty(B, S, D, device=device, dtype=bf) if hw.has_single else None
            self.Zc = torch.empty_like(self.C) if hw.has_single else None
            self.z_img = torch.empty_like(self.x_img) if hw.has_single else None
        if not wl.txt_from_ctx:
            self.x_txt = self.txt  # the text tokens are the block input itself
            if self.joint:
                raise ValueError("batch-1 workloads take their text through txt_in")
        self.loss = torch.zeros(1, device=device)
        # the prediction is written only when asked for (the step's result is the loss)
        self.pred = torch.empty_like(self.z0) if keep_pred else None
        self.dims = L.make_dims(B, S_i, S_t, D, H, F, L.MMDIT_BF16)
        self.embed_stream = torch.cuda.Stream(device)
        self.copy_stream = torch.cuda.Stream(device)
        self.dims_final = L.make_dims(B, S_i, 0, D, H, F, L.MMDIT_BF16)
        ws_block = max(L.mmdit_double_block_workspace_size(self.dims),
                       L.mmdit_single_block_workspace_size(self.dims))
        self.ws_block = L.workspace(ws_block, device)
        self.ws_lin = (L.workspace(L.mmdit_linear_workspace_size(L.MMDIT_BF16, B * S_t, D, wl.ctx_dim), device)
                       if self.txt_in is not None else None)
        self.ws_img = L.workspace(L.mmdit_img_in_workspace_size(L.MMDIT_BF16, B, wl.channels, wl.lat_h,
                                                                wl.lat_w), device)
        self.ws_final = L.workspace(L.mmdit_final_layer_loss_workspace_size(self.dims_final, wl.channels), device)
        self.S, self.S_i, self.B, self.D = S, S_i, B, D
        sets = [("dimg", self.w_dimg["w_mod"], self.w_dimg["b_mod"]),
                ("dtxt", self.w_dtxt["w_mod"], self.w_dtxt["b_mod"])]
        if hw.has_single:
            sets.append(("single", self.w_single["w_mod"], self.w_single["b_mod"]))
        sets.append(("head", self.final["w_ada"], self.final["b_ada"]))
        self.mods = BatchedModulation(torch, L, self.vec, sets, device)
        n_blocks = 2 if hw.has_single else 1
        self.flops_blocks = n_blocks * block_flops(B, S, D, F, H)
        self.flops_dense = (self.flops_blocks + 2 * B * S_i * wl.channels * D
                            + (2 * B * S_t * wl.ctx_dim * D if wl.txt_from_ctx else 0)
                            + 2 * B * S_i * D * wl.channels)

    def _rows(self, dst, src, rows_per_sample, dst_off=0, src_off=0):
        """Copy rows_per_sample token rows of each sample between [B, ., D] bf16 buffers."""
        e = 2 * self.D
        self.L.mmdit_copy_rows(dst.data_ptr() + dst_off * e, dst.shape[1] * e, src.data_ptr() + src_off * e,
                               src.shape[1] * e, rows_per_sample * e, self.B)

    def step(self, before_embed=None):
        """One pass of the hot path; every computation runs in libmmdit.so kernels.
        `before_embed`, if given, runs on the host after the modulations are enqueued and before
        anything that reads the other inputs (the end-to-end step waits there for its copies)."""
        L, wl, side = self.L, self.wl, self.mods
        S_i = self.S_i
        side.compute()  # every modulation of the step, one launch
        main = self.torch.cuda.current_stream()
        if before_embed is not None:
            before_embed()
        # img_in on a second stream beside the RoPE tables and txt_in: neither fills the GPU alone
        self.embed_stream.wait_stream(main)
        with self.torch.cuda.stream(self.embed_stream):
            # z_t = (1 - t) z0 + t z1 formed while patchifying, then projected
            L.mmdit_img_in_noise_fwd(self.z0, self.z1, self.t, self.img_in["w"], self.img_in["b"], self.x_img,
                                     ws=self.ws_img)
        L.rope3d_freqs(self.ids, AXES, THETA, self.cos, self.sin)
        if self.txt_in is not None:
            L.mmdit_linear_fwd(self.txt, self.txt_in["w"], self.txt_in["b"], self.x_txt, ws=self.ws_lin)
        main.wait_stream(self.embed_stream)
        L.mmdit_double_block_fwd(self.dims, side.weights("dimg", self.w_dimg), side.weights("dtxt", self.w_dtxt),
                                 self.vec, self.cos, self.sin, self.x_img, self.x_txt,
                                 self.y_img, self.y_txt, ws=self.ws_block)
        head_in = self.y_img
        if self.w_single is not None:
            if self.joint:
                L.mmdit_single_block_fwd(self.dims, side.weights("single", self.w_single), self.vec, self.cos,
                                         self.sin, self.Y, self.Z, ws=self.ws_block)
                head_in = self.Z[:, :S_i]
            else:
                self._rows(self.C, self.y_img, S_i)
                self._rows(self.C, self.y_txt, self.S - S_i, dst_off=S_i)
                L.mmdit_single_block_fwd(self.dims, side.weights("single", self.w_single), self.vec, self.cos,
                                         self.sin, self.C, self.Zc, ws=self.ws_block)
                self._rows(self.z_img, self.Zc, S_i)
                head_in = self.z_img
        # output head (its shift and scale from the batched modulation launch) with the
        # flow-matching loss fused onto its last kernel
        L.mmdit_final_layer_loss_fwd(self.dims_final, wl.lat_h, wl.lat_w, head_in, self.vec,
                                     self.final["w_ada"], self.final["b_ada"], self.final["w_out"],
                                     self.final["b_out"], self.z0, self.z1, self.loss, pred=self.pred,
                                     mod=side.mods["head"], ws=self.ws_final)

    input_names = ("z0", "z1", "t", "txt", "vec", "ids")

    def workspaces(self):
        return tuple(w for w in (self.ws_block, self.ws_lin, self.ws_img, self.ws_final) if w is not None)

    def result(self):
        """The step's result read back by the end-to-end leg (the loss)."""
        return self.loss

    def step_from_host(self, pinned: dict, result_host):
        """The same step with this step's inputs copied from pinned host memory and the result
        read back.  The copies run on a copy stream that starts after everything before the
        step: vec first, on which the modulations (the step's first launch) wait alone, then the
        rest, on which the embeddings wait; the loss comes back on the step's stream."""
        torch = self.torch
        main = torch.cuda.current_stream()
        cs = self.copy_stream
        cs.wait_stream(main)
        with torch.cuda.stream(cs):
            self.vec.copy_(pinned["vec"], non_blocking=True)
            vec_in = torch.cuda.Event()
            vec_in.record(cs)
            for name, src in pinned.items():
                if name != "vec":
                    getattr(self, name).copy_(src, non_blocking=True)
            all_in = torch.cuda.Event()
            all_in.record(cs)
        main.wait_event(vec_in)
        self.step(before_embed=lambda: main.wait_event(all_in))
        result_host.copy_(self.result(), non_blocking=True)

    def copy_then_step(self, pinned: dict, result_host):
        """The step with every input copied from pinned host memory first and the result read
        back, all on the current stream."""
        for name, src in pinned.items():
            getattr(self, name).copy_(src, non_blocking=True)
        self.step()
        result_host.copy_(self.result(), non_blocking=True)


class Fp8BlockStep(DeviceStep):
    """The 12B block shapes at 2048 px with E4M3 linears: rope3d_freqs, then a double and a
    single block whose four linears per stream run on E4M3 operands with delayed per-tensor
    scaling (the blocks cast their weights at every call, as training does after each
    optimizer step).  The workload names no text or image source, so the block inputs are
    N(0, 1) at width D.  Each step records its amax into history column 0 (most_recent reads
    only the latest), so that a captured graph replays the same step."""

    def __init__(self, wl, device, recipe="delayed"):
        import torch
        from diffusion_transformer_flux_gb300 import _lib as L
        from diffusion_transformer_flux_gb300 import synth
        self.L, self.torch, self.wl = L, torch, wl
        B, D, H, F, S_i, S_t = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden, wl.seq_img, wl.seq_txt
        assert B == 1, "the concatenated-sequence views below assume batch 1"
        S = S_i + S_t
        bf = torch.bfloat16
        inp = synth.block_inputs(B, S_i, S_t, D, "bf16", 1000 + wl.index, (wl.lat_h, wl.lat_w))
        rng_w = np.random.Generator(np.random.PCG64(2000 + wl.index))
        ws_ = [synth.stream_weights(rng_w, D, H, 128, F, "bf16") for _ in range(3)]

        def dev(a, dt=bf):
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device).to(dt)

        self.w_dimg, self.w_dtxt, self.w_single = ({k: dev(v) for k, v in w.items()} for w in ws_)
        self.X = dev(np.concatenate([inp.x_img, inp.x_txt], axis=1))
        self.vec = dev(inp.vec)
        self.ids = dev(inp.ids, torch.float32)
        self.Y = torch.empty_like(self.X)
        self.Z = torch.empty_like(self.X)
        self.cos = torch.empty(B, S, 64, device=device)
        self.sin = torch.empty_like(self.cos)
        self.hist_d = torch.zeros(16, 1024, device=device)
        self.scale_d = torch.ones(16, device=device)
        self.hist_s = torch.zeros(8, 1024, device=device)
        self.scale_s = torch.ones(8, device=device)
        self.fp8_d = L.make_fp8_state(self.hist_d, self.scale_d, pos=0)
        self.fp8_s = L.make_fp8_state(self.hist_s, self.scale_s, pos=0)
        mode = {"delayed": L.MMDIT_GEMM_FP8_E4M3, "tensorwise": L.MMDIT_GEMM_FP8_TENSORWISE,
                "blockwise": L.MMDIT_GEMM_FP8_BLOCKWISE, "mxfp8": L.MMDIT_GEMM_FP8_MXFP8}[recipe]
        if recipe in ("blockwise", "mxfp8"):  # per-tile or per-block scales of this call only: no state
            self.fp8_d = self.fp8_s = None
        self.recipe = recipe
        self.dims = L.make_dims(B, S_i, S_t, D, H, F, L.MMDIT_BF16, gemm=mode)
        ws_block = max(L.mmdit_double_block_workspace_size(self.dims),
                       L.mmdit_single_block_workspace_size(self.dims))
        self.ws_block = L.workspace(ws_block, device)
        self.S, self.S_i = S, S_i
        self.mods = BatchedModulation(torch, L, self.vec,
                                   [(n, w["w_mod"], w["b_mod"]) for n, w in (("dimg", self.w_dimg),
                                                                            ("dtxt", self.w_dtxt),
                                                                            ("single", self.w_single))], device)
        self.flops_blocks = 2 * block_flops(B, S, D, F, H)
        self.flops_dense = self.flops_blocks
        self.flops_linears = 2 * 2 * B * S * D * (3 * D + D + 2 * F)

    input_names = ("X", "vec", "ids")
    step_from_host = DeviceStep.copy_then_step

    def workspaces(self):
        return (self.ws_block,)

    def result(self):
        """The image rows of the single block's output (what a caller keeps)."""
        return self.Z[:, :self.S_i]

    def step(self):
        L, S_i, side = self.L, self.S_i, self.mods
        side.compute()
        L.rope3d_freqs(self.ids, AXES, THETA, self.cos, self.sin)
        L.mmdit_double_block_fwd(self.dims, side.weights("dimg", self.w_dimg), side.weights("dtxt", self.w_dtxt),
                                 self.vec, self.cos, self.sin, self.X[:, :S_i], self.X[:, S_i:],
                                 self.Y[:, :S_i], self.Y[:, S_i:], ws=self.ws_block, fp8=self.fp8_d)
        L.mmdit_single_block_fwd(self.dims, side.weights("single", self.w_single), self.vec, self.cos,
                                 self.sin, self.Y, self.Z, ws=self.ws_block, fp8=self.fp8_s)


class ModelStep(DeviceStep):
    """The whole Flux 12B forward at 512 px through mmdit_flux_forward: rope3d_freqs, the
    flow-matching noise, the model (conditioning vector from t and a pooled text vector, every
    block's modulation in one launch, img_in, txt_in, 19 double and 38 single blocks, the output
    head), the flow-matching loss.  Batch 1, 32 x 32 x 64 latents, a [1, 512, 4096] text
    embedding and a [1, 768] pooled vector, N(0, 1).  The block weights (26 GB of bf16) are
    drawn on the device from a seeded torch generator, N(0, 0.02), gains 1; the embedders and
    the head from the seeded numpy generator."""

    def __init__(self, wl, device):
        import torch
        from diffusion_transformer_flux_gb300 import _lib as L
        from diffusion_transformer_flux_gb300 import synth
        self.L, self.torch, self.wl = L, torch, wl
        B, D, H, F, S_i, S_t = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden, wl.seq_img, wl.seq_txt
        S = S_i + S_t
        bf = torch.bfloat16
        rng_in = np.random.Generator(np.random.PCG64(1000 + wl.index))
        rng_w = np.random.Generator(np.random.PCG64(2000 + wl.index))

        def dev(a, dt=bf):
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device).to(dt)

        z0, z1 = synth.latent_pair(rng_in, B, wl.channels, wl.lat_h, wl.lat_w)
        self.z0, self.z1 = dev(z0, torch.float32), dev(z1, torch.float32)
        self.t = dev(synth.timesteps(rng_in, B, wl.t_dist), torch.float32)
        self.txt = dev(synth.bf16_round(rng_in.standard_normal((B, S_t, wl.ctx_dim), dtype=np.float32)))
        self.y = dev(synth.bf16_round(rng_in.standard_normal((B, wl.vec_dim), dtype=np.float32)))
        self.ids = dev(synth.position_ids(B, wl.lat_h, wl.lat_w, S_t), torch.float32)
        w = {"img_in": tuple(dev(a) for a in synth.embed_weights(rng_w, wl.channels, D).values()),
             "txt_in": tuple(dev(a) for a in synth.embed_weights(rng_w, wl.ctx_dim, D).values()),
             "time_in": tuple(dev(a) for a in synth.mlp_embedder_weights(rng_w, 256, D)),
             "vector_in": tuple(dev(a) for a in synth.mlp_embedder_weights(rng_w, wl.vec_dim, D)),
             "final": {k: dev(v) for k, v in synth.final_layer_weights(rng_w, D, wl.channels).items()}}
        gen = torch.Generator(device=device).manual_seed(2000 + wl.index)

        def n(*shape):
            return (torch.randn(*shape, device=device, generator=gen) * 0.02).to(bf)

        def stream():
            one = torch.ones(128, device=device, dtype=bf)
            return {"w_mod": n(6 * D, D), "b_mod": n(6 * D), "w_qkv": n(3 * D, D), "b_qkv": n(3 * D),
                    "g_q": one, "g_k": one.clone(), "w_o": n(D, D), "b_o": n(D), "w_1": n(F, D), "b_1": n(F),
                    "w_2": n(D, F), "b_2": n(D)}

        w["double"] = [(stream(), stream()) for _ in range(wl.n_double)]
        w["single"] = [stream() for _ in range(wl.n_single)]
        self.weights = w
        self.fw = L.make_flux_w(w)
        dims = L.make_dims(B, S_i, S_t, D, H, F, L.MMDIT_BF16)
        self.cfg = L.make_flux_config(dims, wl.n_double, wl.n_single, wl.lat_h, wl.lat_w, wl.channels,
                                      wl.ctx_dim, 256, wl.vec_dim)
        self.ws_model = L.workspace(L.mmdit_flux_workspace_size(self.cfg), device)
        self.ws_flow = L.workspace(L.flow_match_workspace_size(B, self.z0[0].numel()), device)
        self.cos = torch.empty(B, S, 64, device=device)
        self.sin = torch.empty_like(self.cos)
        self.zt = torch.empty_like(self.z0)
        self.pred = torch.empty_like(self.z0)
        self.loss = torch.zeros(1, device=device)
        self.S, self.S_i = S, S_i
        n_blocks = wl.n_double + wl.n_single
        self.flops_blocks = n_blocks * block_flops(B, S, D, F, H)
        self.flops_dense = (self.flops_blocks + 2 * B * S_i * wl.channels * D + 2 * B * S_t * wl.ctx_dim * D
                            + 2 * B * S_i * D * wl.channels)

    input_names = ("z0", "z1", "t", "txt", "y", "ids")
    step_from_host = DeviceStep.copy_then_step

    def workspaces(self):
        return (self.ws_model, self.ws_flow)

    def step(self):
        L = self.L
        L.rope3d_freqs(self.ids, AXES, THETA, self.cos, self.sin)
        L.flow_match_noise_and_loss(self.z0, self.z1, self.t, z_t=self.zt, ws=self.ws_flow)
        L.mmdit_flux_forward(self.cfg, self.fw, self.zt, self.txt, self.t, self.y, self.cos, self.sin,
                             self.pred, ws=self.ws_model)
        L.flow_match_noise_and_loss(self.z0, self.z1, self.t, pred=self.pred, loss=self.loss,
                                    ws=self.ws_flow)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while running."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, period_ms=20):
        self.uuid = uuid
        self.proc = None
        self.period_ms = period_ms

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        rows = [[c.strip() for c in ln.split(",")] for ln in getattr(self, "lines", [])]
        if self.uuid:
            mine = [r for r in rows if r and self.uuid in r[0]]
            rows = mine or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons, power = [], [], set(), []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ----------------------------------------------------------------------------- per-kernel roofline
def kernel_work(label: str, wl, recipe: str = "delayed"):
    """(bound, algorithmic amount per launch, unit) of one library step, from the workload shapes.
    The FP8 casts move 3 B per element (bf16 in, E4M3 out) under the E4M3 recipes and 4 B under
    MXFP8 (bf16 in, the represented values out in bf16)."""
    B, D, F, H = wl.batch, wl.hidden, wl.mlp_hidden, wl.heads
    S_i, S_t = wl.seq_img, wl.seq_txt
    S = S_i + S_t
    rows = {"img": B * S_i, "txt": B * S_t}
    parts = label.split(".")
    if parts[0] in ("double", "single"):
        r = B * S if parts[0] == "single" else rows[parts[-1]] if parts[-1] in rows else B * S
        op = parts[1]
        if op == "qkv":
            return "tensor", 2.0 * r * D * 3 * D, "FLOP"
        if op == "out":
            return "tensor", 2.0 * r * D * D, "FLOP"
        if op in ("fc1", "fc2"):
            return "tensor", 2.0 * r * D * F, "FLOP"
        if op == "attention":
            return "tensor", 4.0 * B * S * S * 128 * H, "FLOP"
        if op == "modulation":
            sets = 2 if label == "double.modulation" else 1
            return "hbm", sets * (6.0 * D * D * 2 + B * 6 * D * 4) + B * D * 2, "B"
        e_mm = 1 if wl.dtype == "fp8" else 2  # bytes per element of the linears' inputs
        if op == "ln1":
            return "hbm", r * D * 2 + r * D * e_mm, "B"
        if op == "ln2":
            return "hbm", r * D * 4 + r * D * e_mm, "B"
        cast_b = 4.0 if recipe == "mxfp8" else 3.0
        if op == "fp8_cast_w":  # every weight of the block's streams
            sets = 2 if parts[0] == "double" else 1
            return "hbm", sets * cast_b * (4 * D * D + 2 * F * D), "B"
        if op in ("fp8_cast_o", "fp8_cast_h1", "fp8_cast_h2"):  # a D-wide input of every row
            return "hbm", cast_b * B * S * D, "B"
        if op == "fp8_cast_u":  # the fc2 input of every row
            return "hbm", cast_b * B * S * F, "B"
        if op == "fp8_scale":
            return "latency", 0.0, ""
    n_lat = B * wl.channels * S_i
    if label == "conditioning":  # the two embedders' weights
        return "hbm", 2.0 * (256 * D + wl.vec_dim * D + 2 * D * D), "B"
    if label == "modulation.batched":  # every block stream's 6D x D modulation weights
        n_mod = (2 * wl.n_double + wl.n_single if "model" in wl.blocks
                 else 2 + (1 if "single" in wl.blocks else 0))
        # the bf16 steps that end in the output head add its 2D x D shift-and-scale weights
        head = 2.0 * D * D * 2 + B * 2 * D * 4 if ("model" not in wl.blocks and wl.dtype != "fp8") else 0.0
        return "hbm", n_mod * (6.0 * D * D * 2 + B * 6 * D * 4) + head + B * D * 2, "B"
    if label == "modulation":  # one block stream's 6D x D weights (mmdit_modulation_fwd)
        return "hbm", 6.0 * D * D * 2 + B * 6 * D * 4 + B * D * 2, "B"
    if label == "rope3d_freqs":
        return "hbm", B * S * 3 * 4 + 2.0 * B * S * 64 * 4, "B"
    if label in ("flow_match.noise", "flow_match.loss"):
        return "hbm", 3.0 * n_lat * 4, "B"
    if label in ("img_in", "img_in_noise"):  # (the noised variant forms z_t while patchifying)
        return "tensor", 2.0 * B * S_i * wl.channels * D, "FLOP"
    if label == "linear":
        return "tensor", 2.0 * B * S_t * wl.ctx_dim * D, "FLOP"
    if label in ("final_layer", "final_layer_loss"):  # (the loss variant adds the fused MSE)
        return "tensor", 2.0 * B * S_i * D * wl.channels, "FLOP"
    return "unknown", 0.0, ""


def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "diffusion_transformer_flux_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(label: str, workload: str):
    """DRAM bytes per launch of `label` in `workload` from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_digest") != source_digest():
        return None
    v = t.get("workloads", {}).get(workload, {}).get(label)
    return float(v) if v is not None else None


# ----------------------------------------------------------------------------- oracle baseline
def oracle_sample(hw: HostWorkload, n_img_rows: int, n_txt_rows: int, seed: int):
    """One bounded sample of the workload computed by the fp64 oracle: the image and text
    embeddings, then the double block's output at seeded rows (its keys and values need every
    token).  Returns the dense floating-point operations the oracle executed."""
    from oracle import flux as O
    wl = hw.wl
    B, D, H, F, S_i, S_t = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden, wl.seq_img, wl.seq_txt
    S = S_i + S_t
    rng = np.random.default_rng(seed)
    ri = rng.choice(S_i, n_img_rows, replace=False)
    rt = rng.choice(S_t, n_txt_rows, replace=False)
    zt = O.flow_match_noise(hw.z0, hw.z1, hw.t)
    x_img = O.img_in(zt, hw.img_in["w"], hw.img_in["b"])
    x_txt = O.txt_in(hw.txt, hw.txt_in["w"], hw.txt_in["b"]) if hw.txt_in is not None else hw.txt
    cos, sin = O.rope_cos_sin(hw.ids)
    O.double_block_rows(x_img, x_txt, hw.vec, cos, sin, hw.w_dimg, hw.w_dtxt, H, ri, rt)
    nr = B * (n_img_rows + n_txt_rows)
    return (2.0 * B * S_i * wl.channels * D + (2.0 * B * S_t * wl.ctx_dim * D if hw.txt_in is not None else 0.0)
            + 2 * 2.0 * B * D * 6 * D                       # two modulation linears
            + 2.0 * B * S * D * 3 * D + 2.0 * nr * D * 3 * D  # K/V for all tokens, Q for the rows
            + 4.0 * nr * S * 128 * H + 2.0 * nr * D * D + 4.0 * nr * D * F)


def oracle_full_step(hw: HostWorkload):
    """The whole step computed by the fp64 oracle (no rounding anywhere): noise, img_in, the text
    tokens (txt_in where the workload has it), the double block, the single block where the
    workload has one, the output head and the flow-matching loss.  Returns (the blocks' dense
    floating-point operations, the loss)."""
    from oracle import flux as O
    wl = hw.wl
    B, D, H, F, S_i, S_t = wl.batch, wl.hidden, wl.heads, wl.mlp_hidden, wl.seq_img, wl.seq_txt
    zt = O.flow_match_noise(hw.z0, hw.z1, hw.t)
    x_img = O.img_in(zt, hw.img_in["w"], hw.img_in["b"])
    x_txt = O.txt_in(hw.txt, hw.txt_in["w"], hw.txt_in["b"]) if hw.txt_in is not None else hw.txt
    cos, sin = O.rope_cos_sin(hw.ids)
    y_img, y_txt = O.double_block(x_img, x_txt, hw.vec, cos, sin, hw.w_dimg, hw.w_dtxt, H)
    n_blocks = 1
    if hw.has_single:
        c = O.single_block(np.concatenate([y_img, y_txt], axis=1), hw.vec, cos, sin, hw.w_single, H)
        y_img = c[:, :S_i]
        n_blocks = 2
    f = hw.final
    pred = O.final_layer(y_img, hw.vec, f["w_ada"], f["b_ada"], f["w_out"], f["b_out"], wl.lat_h, wl.lat_w)
    return n_blocks * block_flops(B, S_i + S_t, D, F, H), O.flow_match_loss(pred, hw.z0, hw.z1)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measure_euler_step(L, torch, device, hbm_peak, n=1 << 26, reps=10):
    """The sampling step (flow_match_euler_step: guidance combine + Euler update) on n fp32
    elements, 4 * n * 4 bytes per call (z, v_cond, v_uncond read; z_out written), inputs far
    larger than L2; CUDA events around `reps` calls after one warm-up."""
    z, vc, vu = (torch.randn(n, device=device) for _ in range(3))
    out = torch.empty_like(z)
    L.flow_match_euler_step(z, vc, vu, 3.5, 0.05, out)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.flow_match_euler_step(z, vc, vu, 3.5, 0.05, out)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / reps
    gbs = 16.0 * n / us / 1e3
    del z, vc, vu, out
    return {"kernel": "flow_match.euler_step", "n": n, "dtype": "f32", "bytes_per_call": 16 * n,
            "avg_us": round(us, 2), "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4)}


def _time_calls(torch, fn, reps):
    """Average microseconds of fn over `reps` calls after one warm-up (CUDA events)."""
    fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def measure_fp8_peak(torch, device, n=8192, reps=10):
    """Dense E4M3 tensor throughput of this GPU: torch._scaled_mm (cuBLASLt) on n^3 E4M3 operands
    with bf16 output, best of `reps` single calls timed with CUDA events (the bf16 peak's
    protocol).  None if the call is not available."""
    try:
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        one = torch.ones((), device=device)
        bt = b.t()  # column-major second operand, as the call wants

        def mm():
            return torch._scaled_mm(a, bt, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        mm()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return {"tflops": round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1), "n": n,
                "how": f"torch._scaled_mm E4M3 {n}^3, bf16 out, best of {reps} (CUDA events)"}
    except Exception as exc:  # noqa: BLE001 - any failure leaves the nominal ratio in place
        return {"tflops": None, "error": f"{type(exc).__name__}: {exc}"[:200]}


def measure_hbm_sweeps(L, torch, device, hbm_peak, reps=10):
    """The element-wise passes at inputs far larger than L2 (>= 256 MB per operand), against the HBM
    peak: the flow-matching noise (z0, z1 read; z_t written) and loss (z0, z1, pred read) over
    2^26 fp32 elements, and LayerNorm-modulate over 65536 x 4096 bf16 rows (x read, out written)
    and over 32768 x 4096 fp32 rows (the blocks' fp32 residual) to bf16."""
    out = []
    n = 1 << 26
    z0, z1 = torch.randn(n, device=device), torch.randn(n, device=device)
    t = torch.rand(1, device=device)
    zt, pred, loss = torch.empty_like(z0), torch.randn(n, device=device), torch.zeros(1, device=device)
    ws = L.workspace(L.flow_match_workspace_size(1, n), device)
    for label, kw, nbytes in (("flow_match.noise", dict(z_t=zt), 12 * n),
                              ("flow_match.loss", dict(pred=pred, loss=loss), 12 * n)):
        us = _time_calls(torch, lambda: L.flow_match_noise_and_loss(z0.view(1, n), z1.view(1, n), t, ws=ws, **kw),
                         reps)
        gbs = nbytes / us / 1e3
        out.append({"kernel": label, "bytes_per_call": nbytes, "avg_us": round(us, 2),
                    "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4)})
    del z0, z1, zt, pred
    D = 4096
    mod = torch.randn(1, 6 * D, device=device) * 0.1
    for rows, xdt, label in ((65536, torch.bfloat16, "ln_modulate bf16 -> bf16"),
                             (32768, torch.float32, "ln_modulate fp32 -> bf16")):
        x = torch.randn(1, rows, D, device=device).to(xdt)
        y = torch.empty(1, rows, D, device=device, dtype=torch.bfloat16)
        nbytes = rows * D * (x.element_size() + 2)
        us = _time_calls(torch, lambda: L.mmdit_ln_modulate_fwd(x, mod[:, :D], mod[:, D:2 * D], y, 6 * D), reps)
        gbs = nbytes / us / 1e3
        out.append({"kernel": label, "rows": rows, "dim": D, "bytes_per_call": nbytes, "avg_us": round(us, 2),
                    "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4)})
        del x, y
    return out


def measure_parallel_block(st, L, torch, peak, reps=10):
    """The parallel-branch single block (mmdit_single_block_parallel_fwd) at the step's shapes:
    the single block's weights with their first three modulation chunks, CUDA events around
    `reps` calls after one warm-up (283 MB of weights per call, more than L2 holds)."""
    wl = st.wl
    D = wl.hidden
    w = dict(st.w_single, w_mod=st.w_single["w_mod"][:3 * D], b_mod=st.w_single["b_mod"][:3 * D])
    L.mmdit_single_block_parallel_fwd(st.dims, w, st.vec, st.cos, st.sin, st.Y, st.Z, ws=st.ws_block)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.mmdit_single_block_parallel_fwd(st.dims, w, st.vec, st.cos, st.sin, st.Y, st.Z, ws=st.ws_block)
    b.record()
    torch.cuda.synchronize()
    if L.mmdit_workspace_status(st.ws_block) != 0:
        raise RuntimeError("a kernel gave up a bounded wait in the parallel block")
    us = a.elapsed_time(b) * 1e3 / reps
    flops = block_flops(wl.batch, wl.seq, D, wl.mlp_hidden, wl.heads)
    return {"block": "single block with parallel branches", "tokens": wl.seq, "avg_us": round(us, 2),
            "achieved_tflops": round(flops / us / 1e6, 1), "frac": round(flops / us / 1e6 / peak, 4)}


def measure_block_bwd(st, L, torch, peak, reps=3):
    """The double block's backward (mmdit_double_block_bwd) at the step's shapes, every gradient
    requested (both streams' fp32 weight gradients, dvec, dx): CUDA events around `reps` calls
    after one warm-up.  Work counted: the backward's contractions, 2 x the block's GEMM FLOPs (dx
    and dW of each linear) + 2.5 x its attention FLOPs (QK^T recomputed, dO V^T, P^T dO, dS K,
    dS^T Q); the call also recomputes the forward (activation recomputation), which is not
    counted, so the figure is conservative."""
    wl = st.wl
    B, D, F, H, S_i, S_t = wl.batch, wl.hidden, wl.mlp_hidden, wl.heads, wl.seq_img, wl.seq_txt
    S = S_i + S_t
    gen = torch.Generator(device=st.vec.device).manual_seed(7)
    dy_i = (torch.randn(B, S_i, D, device=st.vec.device, generator=gen) * 1e-3).to(torch.bfloat16)
    dy_t = (torch.randn(B, S_t, D, device=st.vec.device, generator=gen) * 1e-3).to(torch.bfloat16)
    dx_i, dx_t = torch.empty_like(dy_i), torch.empty_like(dy_t)
    dvec = torch.empty(B, D, device=st.vec.device)
    grads = [{n: torch.empty(tuple(w[n].shape), device=st.vec.device) for n in L.STREAM_W_FIELDS}
             for w in (st.w_dimg, st.w_dtxt)]
    args = (st.dims, st.w_dimg, st.w_dtxt, st.vec, st.cos, st.sin, st.x_img, st.x_txt, dy_i, dy_t, dx_i, dx_t, dvec,
            grads[0], grads[1])
    ws = L.mmdit_double_block_bwd(*args)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.mmdit_double_block_bwd(*args, ws=ws)
    b.record()
    torch.cuda.synchronize()
    if L.mmdit_workspace_status(ws) != 0:
        raise RuntimeError("a kernel gave up a bounded wait in the block backward")
    us = a.elapsed_time(b) * 1e3 / reps
    gemm = 2 * B * S * D * (3 * D + D + 2 * F)
    attn = 4 * B * S * S * 128 * H
    flops = 2 * gemm + 2.5 * attn
    # one more call with the library's per-step events: the attention backward's own time
    L.mmdit_profile_enable(True)
    L.mmdit_double_block_bwd(*args, ws=ws)
    steps = L.mmdit_profile_collect()
    L.mmdit_profile_enable(False)
    attn_us = 1e3 * sum(ms for n, ms in steps if n == "bwd.attention")
    del grads, ws
    return {"op": "double block backward (all gradients, forward recomputed inside)", "tokens": S,
            "avg_us": round(us, 2), "flops_counted": flops, "achieved_tflops": round(flops / us / 1e6, 1),
            "frac": round(flops / us / 1e6 / peak, 4),
            "attention_backward": {"avg_us": round(attn_us, 2), "flops": 2.5 * attn,
                                   "achieved_tflops": round(2.5 * attn / attn_us / 1e6, 1) if attn_us else None,
                                   "frac": round(2.5 * attn / attn_us / 1e6 / peak, 4) if attn_us else None}}


def measure_block_train(st, L, torch, peak, reps=3):
    """One double block's share of a training step at the step's shapes, two ways: the forward
    (mmdit_double_block_fwd) then the one-call backward, which recomputes the forward; and the
    training pair (mmdit_double_block_fwd_train, which keeps what the backward reads, then
    mmdit_double_block_bwd_saved).  CUDA events around `reps` of each after one warm-up; the
    work counted is the forward's contractions plus the backward's (2 x the GEMMs + 2.5 x the
    attention), the same for both."""
    wl = st.wl
    B, D, F, H, S_i, S_t = wl.batch, wl.hidden, wl.mlp_hidden, wl.heads, wl.seq_img, wl.seq_txt
    S = S_i + S_t
    dev = st.vec.device
    gen = torch.Generator(device=dev).manual_seed(8)
    dy_i = (torch.randn(B, S_i, D, device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
    dy_t = (torch.randn(B, S_t, D, device=dev, generator=gen) * 1e-3).to(torch.bfloat16)
    y_i, y_t = torch.empty_like(dy_i), torch.empty_like(dy_t)
    dx_i, dx_t = torch.empty_like(dy_i), torch.empty_like(dy_t)
    dvec = torch.empty(B, D, device=dev)
    grads = [{n: torch.empty(tuple(w[n].shape), device=dev) for n in L.STREAM_W_FIELDS}
             for w in (st.w_dimg, st.w_dtxt)]
    common = (st.dims, st.w_dimg, st.w_dtxt, st.vec, st.cos, st.sin, st.x_img, st.x_txt)
    ws_f = L.workspace(L.mmdit_double_block_workspace_size(st.dims), dev)
    ws_b = L.workspace(L.mmdit_double_block_bwd_workspace_size(st.dims), dev)

    def recompute():
        L.mmdit_double_block_fwd(*common, y_i, y_t, ws=ws_f)
        L.mmdit_double_block_bwd(*common, dy_i, dy_t, dx_i, dx_t, dvec, grads[0], grads[1], ws=ws_b)

    def pair():
        L.mmdit_double_block_fwd_train(*common, y_i, y_t, saved=ws_b)
        L.mmdit_double_block_bwd_saved(*common, dy_i, dy_t, dx_i, dx_t, ws_b, dvec, grads[0], grads[1])

    out = {}
    for name, fn in (("forward + one-call backward", recompute), ("training pair", pair)):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        if L.mmdit_workspace_status(ws_b) != 0:
            raise RuntimeError("a kernel gave up a bounded wait in the block training step")
        out[name] = a.elapsed_time(b) * 1e3 / reps
    gemm = 2 * B * S * D * (3 * D + D + 2 * F)
    attn = 4 * B * S * S * 128 * H
    flops = (gemm + attn) + (2 * gemm + 2.5 * attn)
    del grads, ws_f, ws_b
    return {"op": "double block forward + backward (all gradients)", "tokens": S, "flops_counted": flops,
            **{k: {"avg_us": round(v, 2), "achieved_tflops": round(flops / v / 1e6, 1),
                   "frac": round(flops / v / 1e6 / peak, 4)} for k, v in out.items()}}


def measure_blockwise_linear(L, torch, device, M=4608, N=12288, K=3072, reps=5):
    """The blockwise FP8 linear (mmdit_fp8_blockwise_linear_fwd: per-tile E4M3 casts of x and W in
    the call, then the slice-scaled GEMM) at the fc1 shape: 2 M N K FLOPs per call, CUDA events
    around `reps` calls after one warm-up."""
    x = torch.randn(M, K, device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, device=device) * 0.02).to(torch.bfloat16)
    b = torch.zeros(N, device=device, dtype=torch.bfloat16)
    y = torch.empty(M, N, device=device, dtype=torch.bfloat16)
    ws = L.mmdit_fp8_blockwise_linear_fwd(x, w, b, y)
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.mmdit_fp8_blockwise_linear_fwd(x, w, b, y, ws=ws)
    e.record()
    torch.cuda.synchronize()
    if L.mmdit_workspace_status(ws) != 0:
        raise RuntimeError("a kernel gave up a bounded wait in the blockwise FP8 linear")
    us = a.elapsed_time(e) * 1e3 / reps
    return {"op": "blockwise FP8 linear (casts of x and W included)", "M": M, "N": N, "K": K,
            "avg_us": round(us, 2), "achieved_tflops": round(2.0 * M * N * K / us / 1e6, 1)}


def measure_mx_linear(L, torch, device, M=4608, N=12288, K=3072, reps=5):
    """The MXFP8 linear (mmdit_fp8_mxfp8_linear_fwd: the MX casts of x and W in the call, then the
    bf16 GEMM of their represented values) at the fc1 shape: 2 M N K FLOPs per call, CUDA events
    around `reps` calls after one warm-up."""
    x = torch.randn(M, K, device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, device=device) * 0.02).to(torch.bfloat16)
    b = torch.zeros(N, device=device, dtype=torch.bfloat16)
    y = torch.empty(M, N, device=device, dtype=torch.bfloat16)
    ws = L.mmdit_fp8_mxfp8_linear_fwd(x, w, b, y)
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.mmdit_fp8_mxfp8_linear_fwd(x, w, b, y, ws=ws)
    e.record()
    torch.cuda.synchronize()
    if L.mmdit_workspace_status(ws) != 0:
        raise RuntimeError("a kernel gave up a bounded wait in the MXFP8 linear")
    us = a.elapsed_time(e) * 1e3 / reps
    return {"op": "MXFP8 linear (casts of x and W included; bf16 tensor cores)", "M": M, "N": N, "K": K,
            "avg_us": round(us, 2), "achieved_tflops": round(2.0 * M * N * K / us / 1e6, 1)}


def measure_linear_bwd(L, torch, device, peak, M=4608, N=12288, K=3072, reps=5):
    """The backward of the block's fc1-shaped linear (mmdit_linear_bwd: dx and dW through the
    tensor-core GEMM reading W, dy and x MN-major as stored, db): 4 M N K FLOPs per call, CUDA
    events around `reps` calls after one warm-up."""
    dy = torch.randn(M, N, device=device).to(torch.bfloat16)
    x = torch.randn(M, K, device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, device=device) * 0.02).to(torch.bfloat16)
    dx = torch.empty(M, K, device=device, dtype=torch.bfloat16)
    dw = torch.empty(N, K, device=device)
    db = torch.empty(N, device=device)
    ws = L.mmdit_linear_bwd(dy, x, w, dx, dw, db)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        L.mmdit_linear_bwd(dy, x, w, dx, dw, db, ws=ws)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / reps
    flops = 4.0 * M * N * K
    return {"op": "linear backward (dx, dW, db)", "M": M, "N": N, "K": K, "avg_us": round(us, 2),
            "achieved_tflops": round(flops / us / 1e6, 1), "frac": round(flops / us / 1e6 / peak, 4)}


def run_cpu_baseline_full(hw: HostWorkload):
    """One full step of the fp64 oracle, timed; its loss checks the GPU's."""
    t0 = time.perf_counter()
    flops, loss = oracle_full_step(hw)
    dt = time.perf_counter() - t0
    blocks = "double and single blocks" if hw.has_single else "double block"
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"1 x the whole step in the fp64 oracle at full size ({wl_desc(hw.wl)}, batch "
                       f"{hw.wl.batch}): noise, img_in, text tokens, the full {blocks}, output head, "
                       "loss; the value counts the blocks' dense FLOPs over the step's time"),
            "seconds": round(dt, 2)}, loss


def run_cpu_baseline(hw: HostWorkload, min_seconds: float, rows=(32, 8)):
    flops, n, t0 = 0.0, 0, time.perf_counter()
    while True:
        flops += oracle_sample(hw, rows[0], rows[1], seed=n)
        n += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"{n} x (fp64 oracle: flow-matching noise, img_in, txt_in, then the "
                       f"{wl_desc(hw.wl)} double block at {rows[0]} image + {rows[1]} text rows with "
                       "keys/values for all tokens)"), "seconds": round(dt, 2)}


def wl_desc(wl):
    return f"{wl.seq_img}+{wl.seq_txt}-token D{wl.hidden} F{wl.mlp_hidden}"


def run_reference(args):
    """The oracle on the host cores, on this workload, one bounded sample per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from diffusion_transformer_flux_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    hw = HostWorkload(wl)
    rows = (8, 2)
    for i in range(args.warmup):
        oracle_sample(hw, *rows, seed=i)
    flops, t0 = 0.0, time.perf_counter()
    for i in range(args.steps):
        flops += oracle_sample(hw, *rows, seed=1000 + i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"per step: fp64 oracle flow-matching noise, img_in, txt_in and the {wl_desc(wl)} "
              f"double block at {rows[0]} image + {rows[1]} text rows (keys/values for all tokens)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64; N(0,0.02) weights, N(0,1) activations and latents)",
            "config": {"workload": WORKLOAD, "global_batch": wl.batch, "seq_len": wl.seq,
                       "tokens": f"{wl.seq_img} image + {wl.seq_txt} text", "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, local = dist_env()
    import torch
    from diffusion_transformer_flux_gb300 import _lib as L
    from diffusion_transformer_flux_gb300 import synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    L.load()
    wl = synth.WORKLOADS[args.workload]
    fp8 = wl.dtype == "fp8"
    model = args.workload == MODEL_WORKLOAD
    hw = None if (fp8 or model) else HostWorkload(wl)
    st = (Fp8BlockStep(wl, device, args.fp8_recipe) if fp8 else ModelStep(wl, device) if model
          else DeviceStep(hw, device))
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > 129 MB of L2

    def barrier():
        if dist is not None:
            dist.barrier()


    def timed(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        barrier()
        torch.cuda.synchronize()
        L.mmdit_launch_count_reset()
        for i in range(k):
            flush.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        launches = L.mmdit_launch_count()
        barrier()
        return [a.elapsed_time(b) for a, b in evs], launches

    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    for ws in st.workspaces():
        if L.mmdit_workspace_status(ws) != 0:
            raise RuntimeError("a kernel gave up a bounded wait during warm-up")

    # library launches of one step, counted on a plain (uncaptured) step
    L.mmdit_launch_count_reset()
    st.step()
    torch.cuda.synchronize()
    launches_per_step = L.mmdit_launch_count()
    step_fn = st.step
    if not args.no_graph:
        # the whole step as one CUDA graph (captured on a side stream after warm-up there)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                st.step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            st.step()
        torch.cuda.synchronize()
        step_fn = graph.replay
        for _ in range(args.warmup):
            step_fn()
        torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "") or "") or None
    with ClockSampler(uuid) as clk:
        ms, _ = timed(step_fn, args.steps)
    launches = launches_per_step * args.steps
    clocks = clk.summary()
    if not bool(torch.isfinite(st.result()).all()):
        raise RuntimeError("non-finite result")
    for ws in st.workspaces():
        if L.mmdit_workspace_status(ws) != 0:
            raise RuntimeError("a kernel gave up a bounded wait in the timed steps")
    total_s = max_over_ranks(dist, sum(ms) / 1e3, device)
    value = whole_job_tflops(st.flops_blocks, args.steps, world, total_s)

    # end to end: this step's inputs from pinned host memory, the loss back to the host
    pinned = {n: getattr(st, n).detach().cpu().pin_memory() for n in st.input_names}
    res = st.result()
    result_host = torch.empty(res.shape, dtype=res.dtype, pin_memory=True)
    for _ in range(2):
        st.step_from_host(pinned, result_host)
    ms_e2e, _ = timed(lambda: st.step_from_host(pinned, result_host), args.steps)
    e2e_s = max_over_ranks(dist, sum(ms_e2e) / 1e3, device)
    # the end-to-end step's result against a plain step of the same (now resident) inputs
    torch.cuda.synchronize()
    e2e_result = result_host.clone()
    st.step()
    torch.cuda.synchronize()
    if not torch.equal(e2e_result, st.result().cpu()):
        raise RuntimeError("the end-to-end step's result differs from the plain step's")
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = result_host.numel() * result_host.element_size()

    # per-kernel durations from CUDA events the library records around each of its steps
    L.mmdit_profile_enable(True)
    for _ in range(args.profile_steps):
        flush.zero_()
        st.step()
    recs = L.mmdit_profile_collect()
    L.mmdit_profile_enable(False)
    agg = {}
    for name, t in recs:
        a = agg.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += t
    prof_total = sum(v[1] for v in agg.values()) or 1.0
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # E4M3 contractions: this GPU's measured E4M3 GEMM throughput where it could be taken, else
    # the measured bf16 peak times the nominal dense fp8 : bf16 ratio (2)
    fp8_meas = measure_fp8_peak(torch, device) if fp8 else None
    fp8_measured = bool(fp8_meas and fp8_meas.get("tflops"))
    fp8_peak = float(fp8_meas["tflops"]) if fp8_measured else 2.0 * bf16_peak

    def peak_of(name):
        is_linear = name.split(".")[-1] in ("qkv", "out", "fc1", "fc2")
        # the MXFP8 recipe multiplies its represented values on the bf16 tensor cores
        return fp8_peak if (fp8 and is_linear and args.fp8_recipe != "mxfp8") else bf16_peak

    per_kernel = []
    for name, (n, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        bound, amount, unit = kernel_work(name, wl, args.fp8_recipe)
        avg_s = t / n / 1e3
        row = {"kernel": name, "launches": n, "avg_us": round(avg_s * 1e6, 2), "share": round(t / prof_total, 4),
               "bound": bound}
        if bound == "tensor":
            row["achieved_tflops"] = round(amount / avg_s / 1e12, 1)
            row["frac"] = round(amount / avg_s / 1e12 / peak_of(name), 4)
        elif bound == "hbm":
            row["achieved_gbs"] = round(amount / avg_s / 1e9, 1)
            row["frac"] = round(amount / avg_s / 1e9 / hbm_peak, 4)
        per_kernel.append(row)
    dom = per_kernel[0]
    bound, amount, unit = kernel_work(dom["kernel"], wl, args.fp8_recipe)
    dom_s = dom["avg_us"] / 1e6
    if bound == "tensor":
        ach, peak, runit = amount / dom_s / 1e12, peak_of(dom["kernel"]), "TFLOP/s"
    else:
        ach, peak, runit = amount / dom_s / 1e9, hbm_peak, "GB/s"
    roofline = {"kernel": dom["kernel"], "bound": bound, "achieved": round(ach, 2), "peak": peak,
                "unit": runit, "frac": round(ach / peak, 4), "traffic": committed_traffic(dom["kernel"], args.workload),
                "algorithmic_per_launch": amount, "algorithmic_unit": unit,
                "peak_source": f"{peak_src}: {'bf16_tflops (burst)' if bound == 'tensor' else 'hbm_gbs'}"}
    if peak != bf16_peak and bound == "tensor":
        roofline["peak_source"] = ("measured in this run: torch._scaled_mm E4M3 8192^3 (burst)" if fp8_measured
                                   else roofline["peak_source"] + " x 2 (nominal dense fp8 : bf16 ratio)")
    if bound == "tensor" and "bf16_tflops_sustained" in peaks and peak == bf16_peak:
        roofline["frac_of_sustained"] = round(ach / float(peaks["bf16_tflops_sustained"]), 4)

    extras = {}
    if args.workload == WORKLOAD:
        extras["sampling_step"] = measure_euler_step(L, torch, device, hbm_peak)
        extras["hbm_sweeps"] = measure_hbm_sweeps(L, torch, device, hbm_peak)
        extras["single_block_parallel"] = measure_parallel_block(st, L, torch, bf16_peak)
        extras["linear_backward"] = measure_linear_bwd(L, torch, device, bf16_peak)
        extras["blockwise_fp8_linear"] = measure_blockwise_linear(L, torch, device)
        extras["mxfp8_linear"] = measure_mx_linear(L, torch, device)
        extras["double_block_backward"] = measure_block_bwd(st, L, torch, bf16_peak)
        extras["double_block_training"] = measure_block_train(st, L, torch, bf16_peak)
    if fp8:
        extras["fp8_peak"] = fp8_meas

    cpu, loss_check = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and hw is not None:
        if args.workload in (WORKLOAD, C3_WORKLOAD):
            # the whole step in the fp64 oracle, once: the CPU baseline, and the reference loss
            cpu, ref_loss = run_cpu_baseline_full(hw)
            gpu_loss = float(st.loss.item())
            loss_check = {"gpu": gpu_loss, "oracle_fp64": ref_loss,
                          "rel_err": abs(gpu_loss - ref_loss) / abs(ref_loss)}
        else:
            cpu = run_cpu_baseline(hw, args.cpu_seconds)

    if rank == 0:
        S = wl.seq
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 linears, bf16 attention and activations" if fp8 else "bf16",
            "data": "synthetic (seeded PCG64; N(0,0.02) weights, N(0,1) activations, text embeddings "
                    "and latents; no dataset or trained weights)",
            "config": {"workload": args.workload, **({"fp8_recipe": args.fp8_recipe} if fp8 else {}),
                       "global_batch": world * wl.batch, "seq_len": S,
                       "tokens": f"{wl.seq_img} image + {wl.seq_txt} text", "hidden": wl.hidden,
                       "heads": wl.heads, "head_dim": 128, "mlp_hidden": wl.mlp_hidden,
                       "parallelism": f"{world} independent replica(s), no exchange",
                       "l2": "flushed before every timed step (256 MB write outside the events)",
                       "launch": "plain calls" if args.no_graph else
                                 "CUDA-graph replay of the step (e2e: plain calls)",
                       "step": ("rope3d_freqs, double block, single block (E4M3 linears; "
                                + {"delayed": "delayed per-tensor scaling", "tensorwise": "current per-tensor scaling",
                                   "blockwise": "current per-tile scaling, 1 x 128 inputs and 128 x 128 weights",
                                   "mxfp8": "MXFP8: E4M3 with a power-of-two scale per 32 elements along K, "
                                            "products of the represented values on the bf16 tensor cores"}[
                                    args.fp8_recipe]
                                + "; weights cast at every call)") if fp8 else
                               ("rope3d_freqs, flow-matching noise, mmdit_flux_forward (conditioning, "
                                "every block's modulation in one launch, img_in, txt_in, "
                                f"{wl.n_double} double + {wl.n_single} single blocks, output head), "
                                "flow-matching loss") if model else
                               ("rope3d_freqs, img_in of z_t (noise fused into the patchify), "
                                + ("txt_in, " if wl.txt_from_ctx else "")
                                + ("double block, single block, " if "single" in wl.blocks else "double block, ")
                                + "output head with the flow-matching loss fused on"
                                + ("" if wl.batch == 1 else "; streams joined and split by strided "
                                   "copy-engine copies (mmdit_copy_rows)")),
                       "streams": ("two streams: every modulation of the step first, in one launch "
                                   "(mmdit_modulation_batched_fwd), then img_in on a second stream beside the "
                                   "RoPE tables and txt_in, joined before the double block")
                                  if type(st) is DeviceStep else
                                  "one stream; every modulation of the step runs first, in one "
                                  "launch (mmdit_modulation_batched_fwd)",
                       "flops_counted_per_step": st.flops_blocks,
                       "dense_flops_per_step_incl_embeds_and_head": st.flops_dense},
            "pct_of_bf16_peak": round(100 * value / world / bf16_peak, 2),
            **({"fp8_peak_tflops": fp8_peak, "fp8_peak_measured": fp8_measured,
                # (none under MXFP8, whose linears run on the bf16 tensor cores)
                "linears_pct_of_fp8_peak": round(100 * sum(r["achieved_tflops"] * r["avg_us"] for r in per_kernel
                                                           if r["bound"] == "tensor" and peak_of(r["kernel"]) == fp8_peak)
                                                 / max(1e-9, sum(r["avg_us"] for r in per_kernel if r["bound"] == "tensor"
                                                                 and peak_of(r["kernel"]) == fp8_peak)) / fp8_peak, 2)
                if args.fp8_recipe != "mxfp8" else None}
               if fp8 else {}),
            "tokens_per_s": round(world * wl.batch * S * args.steps / total_s, 1),
            "clocks": clocks,
            "e2e": {"value": round(whole_job_tflops(st.flops_blocks, args.steps, world, e2e_s), 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_s / args.steps * 1e3, 4),
                    "copies": ("each step's inputs on a copy stream inside the timed region (vec first: "
                               "the modulations wait for it alone, the embeddings for the rest); plain "
                               "calls, no graph; the result checked bit-equal to a plain step's")
                              if type(st) is DeviceStep else
                              ("each step's inputs on the step's stream before the step; plain calls, "
                               "no graph; the result checked bit-equal to a plain step's")},
            "gpu_launches": launches,
            "roofline": roofline,
            "per_kernel": per_kernel,
            "cpu_baseline": cpu,
            "loss_check": loss_check,
            "extras": extras,
            "peaks": {"bf16_tflops": bf16_peak, "hbm_gbs": hbm_peak, "source": peak_src},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
