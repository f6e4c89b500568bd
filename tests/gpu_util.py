"""Helpers shared by the GPU parity tests: device upload of seeded inputs, running the blocks
through the C ABI, and the parity bar (max |err| <= tol x RMS of the oracle output)."""
from __future__ import annotations

import numpy as np
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

TOL_BF16 = 2e-2   # max |err| <= 2e-2 x RMS(oracle output), the stated bar for bf16 (and tf32)
# Distance between the exact float64 block and any bf16-operand evaluation of it at the
# Flux-sized shapes: the bf16-autocast oracle itself sits 2.6e-2 (fp32 output) to 3.5e-2
# (bf16 output) x RMS from the float64 one, so GPU-vs-float64 is held to this looser bound.
TOL_VS_FP64 = 5e-2


def dev(a, dtype=torch.bfloat16) -> torch.Tensor:
    """Upload values that are already rounded to `dtype` (so the cast is exact)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(dtype)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(a) -> np.ndarray:
    """Half the spacing of bf16 values (8 significant bits) at magnitude |a|."""
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def max_err_over_rms(got, ref, out_bf16=False) -> tuple[float, float]:
    """max_i (|got_i - ref_i| - r_i) / RMS(ref), with r_i half a bf16 ulp when the output
    is stored in bf16 (the representation error of the output format) and 0 otherwise."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    if out_bf16:
        err = np.maximum(err - half_ulp_bf16(np.maximum(np.abs(got), np.abs(ref))), 0.0)
    return float(err.max()) / rms, rms


def assert_parity(got, ref, tol=TOL_BF16, what="", out_bf16=False):
    got = np.asarray(got, np.float64)
    assert got.shape == np.shape(ref), (what, got.shape, np.shape(ref))
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e, rms = max_err_over_rms(got, ref, out_bf16)
    extra = " beyond the bf16 output rounding" if out_bf16 else ""
    assert e <= tol, f"{what}: max|err|{extra} / RMS = {e:.3e} > {tol} (RMS {rms:.3e})"
    return e


def torch_dtype(act: str):
    return torch.float32 if act == "f32" else torch.bfloat16


def upload_weights(w: dict, act: str) -> dict:
    return {k: dev(v, torch_dtype(act)) for k, v in w.items()}


class BlockCase:
    """Seeded inputs and weights of one block call, on host (fp32 values) and device."""

    def __init__(self, B, S_i, S_t, D, H, F, act="bf16", seed=0, std=0.02, gain_jitter=0.1,
                 lat_hw=None, single=False, interleaved=True, gelu_tanh=False):
        self.B, self.S_i, self.S_t, self.D, self.H, self.F = B, S_i, S_t, D, H, F
        self.S = S_i + S_t
        self.act, self.single = act, single
        self.interleaved, self.gelu_tanh = interleaved, gelu_tanh
        cast = "f32" if act == "f32" else "bf16"
        inp = synth.block_inputs(B, S_i, S_t, D, cast, seed, lat_hw)
        rng = np.random.Generator(np.random.PCG64(seed + 1000))
        self.w_img = synth.stream_weights(rng, D, H, 128, F, cast, std, gain_jitter)
        self.w_txt = None if single else synth.stream_weights(rng, D, H, 128, F, cast, std, gain_jitter)
        self.x_img, self.x_txt, self.vec, self.ids = inp.x_img, inp.x_txt, inp.vec, inp.ids
        self.cos, self.sin = O.rope_cos_sin(self.ids)
        self.dims = L.make_dims(B, S_i, S_t, D, H, F, L.MMDIT_F32 if act == "f32" else L.MMDIT_BF16,
                                rope_interleaved=interleaved, gelu_tanh=gelu_tanh)

    def x_joint(self):
        return np.concatenate([self.x_img, self.x_txt], axis=1)

    def run_gpu(self):
        """Runs the block through the C ABI; returns (outputs..., workspace, rope tables)."""
        t = torch_dtype(self.act)
        ids = torch.from_numpy(self.ids).cuda()
        cos = torch.empty(self.B, self.S, 64, device="cuda")
        sin = torch.empty_like(cos)
        L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
        vec = dev(self.vec, t)
        wi = upload_weights(self.w_img, self.act)
        if self.single:
            x = dev(self.x_joint(), t)
            y = torch.empty_like(x)
            ws = L.mmdit_single_block_fwd(self.dims, wi, vec, cos, sin, x, y)
            torch.cuda.synchronize()
            assert L.mmdit_workspace_status(ws) == 0
            return (host(y),), ws, (cos, sin)
        wt = upload_weights(self.w_txt, self.act)
        xi, xt = dev(self.x_img, t), dev(self.x_txt, t)
        yi, yt = torch.empty_like(xi), torch.empty_like(xt)
        ws = L.mmdit_double_block_fwd(self.dims, wi, wt, vec, cos, sin, xi, xt, yi, yt)
        torch.cuda.synchronize()
        assert L.mmdit_workspace_status(ws) == 0
        return (host(yi), host(yt)), ws, (cos, sin)

    @property
    def mm_cast(self):
        """The oracle precision the bar is checked at: bf16 autocast for bf16 workloads."""
        return O.round_bf16 if self.act == "bf16" else None

    def oracle(self, mm_cast=None):
        if self.single:
            return (O.single_block(self.x_joint(), self.vec, self.cos, self.sin, self.w_img, self.H,
                                   self.interleaved, self.gelu_tanh, mm_cast=mm_cast),)
        return O.double_block(self.x_img, self.x_txt, self.vec, self.cos, self.sin, self.w_img,
                              self.w_txt, self.H, self.interleaved, self.gelu_tanh, mm_cast=mm_cast)

    def oracle_rows(self, rows_img, rows_txt=None, mm_cast=None):
        if self.single:
            return (O.single_block_rows(self.x_joint(), self.vec, self.cos, self.sin, self.w_img,
                                        self.H, rows_img, self.interleaved, self.gelu_tanh,
                                        mm_cast=mm_cast),)
        return O.double_block_rows(self.x_img, self.x_txt, self.vec, self.cos, self.sin, self.w_img,
                                   self.w_txt, self.H, rows_img, rows_txt, self.interleaved,
                                   self.gelu_tanh, mm_cast=mm_cast)


def workspace_view(ws: torch.Tensor, offset: int, shape, dtype) -> torch.Tensor:
    n = int(np.prod(shape))
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[offset:offset + nbytes].view(dtype).view(*shape)
