"""ctypes binding of libmmdit.so: argument marshalling only.

Every function here has the name of the C entry point it calls and forwards torch tensors as
raw device pointers together with torch's current CUDA stream.  No computation happens in
Python; when the library is missing, loading fails with an error (there is no fallback).
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build_ext

MMDIT_OK = 0
MMDIT_F32 = 0
MMDIT_BF16 = 1
STATUS_NAMES = {0: "MMDIT_OK", 1: "MMDIT_ERR_INVALID_ARG", 2: "MMDIT_ERR_UNSUPPORTED",
                3: "MMDIT_ERR_WORKSPACE", 4: "MMDIT_ERR_CUDA", 5: "MMDIT_ERR_NONFINITE",
                6: "MMDIT_ERR_DEVICE"}

# Names exported by the library, in include/mmdit.h order.
EXPORTED = [
    "mmdit_last_error", "mmdit_workspace_status", "mmdit_launch_count", "mmdit_launch_count_reset",
    "mmdit_profile_enable", "mmdit_profile_collect",
    "rope3d_freqs", "mmdit_modulation_fwd", "flow_match_workspace_size", "flow_match_noise_and_loss",
    "flow_match_noise_and_loss_noalloc", "flow_match_euler_step",
    "mmdit_linear_workspace_size", "mmdit_linear_fwd", "mmdit_img_in_workspace_size",
    "mmdit_img_in_fwd", "mmdit_img_in_noise_fwd", "mmdit_final_layer_workspace_size",
    "mmdit_final_layer_fwd", "mmdit_final_layer_loss_workspace_size", "mmdit_final_layer_loss_fwd",
    "mmdit_ln_modulate_fwd", "mmdit_copy_rows",
    "mmdit_attention_workspace_size", "mmdit_attention_fwd", "mmdit_fp8_attention_workspace_size",
    "mmdit_fp8_attention_fwd", "mmdit_double_block_workspace_size",
    "mmdit_double_block_fwd", "mmdit_single_block_workspace_size", "mmdit_single_block_fwd",
    "mmdit_block_workspace_offsets", "mmdit_fp8_quantize_e4m3", "mmdit_fp8_linear_workspace_size",
    "mmdit_fp8_linear_fwd", "mmdit_fp8_linear_bwd_workspace_size", "mmdit_fp8_linear_bwd",
    "mmdit_fp8_blockwise_linear_workspace_size", "mmdit_fp8_blockwise_linear_fwd",
    "mmdit_fp8_mxfp8_linear_workspace_size", "mmdit_fp8_mxfp8_linear_fwd",
    "mmdit_single_block_parallel_fwd", "mmdit_linear_bwd_workspace_size",
    "mmdit_linear_bwd", "mmdit_double_block_bwd_workspace_size", "mmdit_double_block_bwd",
    "mmdit_single_block_bwd_workspace_size", "mmdit_single_block_bwd", "mmdit_double_block_fwd_train",
    "mmdit_double_block_bwd_saved", "mmdit_single_block_fwd_train", "mmdit_single_block_bwd_saved",
    "mmdit_modulation_batched_fwd", "mmdit_conditioning_workspace_size",
    "mmdit_conditioning_fwd", "mmdit_flux_workspace_size", "mmdit_flux_forward",
]


class MMDitError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Dims(C.Structure):
    _fields_ = [("batch", C.c_int32), ("seq_img", C.c_int32), ("seq_txt", C.c_int32),
                ("hidden", C.c_int32), ("heads", C.c_int32), ("head_dim", C.c_int32),
                ("mlp_hidden", C.c_int32), ("ln_eps", C.c_float), ("rms_eps", C.c_float),
                ("rope_interleaved", C.c_int32), ("gelu_tanh", C.c_int32), ("act", C.c_int32),
                ("gemm", C.c_int32)]


STREAM_W_FIELDS = ["w_mod", "b_mod", "w_qkv", "b_qkv", "g_q", "g_k", "w_o", "b_o", "w_1", "b_1",
                   "w_2", "b_2"]


class StreamW(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in STREAM_W_FIELDS] + [("mod", C.c_void_p)]


class Fp8State(C.Structure):
    _fields_ = [("amax_history", C.c_void_p), ("scale", C.c_void_p), ("hist_len", C.c_int32),
                ("n_tensors", C.c_int32), ("pos", C.c_int32), ("amax_compute_algo", C.c_int32),
                ("margin", C.c_int32)]


AMAX_MOST_RECENT = 0
AMAX_MAX = 1


MMDIT_GEMM_NATIVE = 0
MMDIT_GEMM_FP8_E4M3 = 1
MMDIT_GEMM_FP8_TENSORWISE = 2
MMDIT_GEMM_FP8_BLOCKWISE = 3
MMDIT_GEMM_FP8_MXFP8 = 4
FP8_LINEARS = ("qkv", "o", "fc1", "fc2")


def fp8_tensor(slot: int, linear: str, operand: str) -> int:
    """Index of a tensor in the FP8 state: slot 0 image/single, 1 text; operand "x" or "w"."""
    return 8 * slot + 2 * FP8_LINEARS.index(linear) + (1 if operand == "w" else 0)


VP, SZ, I32, I64, F32 = C.c_void_p, C.c_size_t, C.c_int32, C.c_int64, C.c_float
PDIMS, PW, PFP8 = C.POINTER(Dims), C.POINTER(StreamW), C.POINTER(Fp8State)


class StreamGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in STREAM_W_FIELDS]


PGRADS = C.POINTER(StreamGrads)


class GemvJob(C.Structure):
    _fields_ = [("w", VP), ("b", VP), ("out", VP), ("rows", I32)]


class MlpEmbedderW(C.Structure):
    _fields_ = [("w1", VP), ("b1", VP), ("w2", VP), ("b2", VP)]


class CondW(C.Structure):
    _fields_ = [("time_in", MlpEmbedderW), ("vector_in", MlpEmbedderW), ("w_guidance", VP),
                ("b_guidance", VP)]


class FluxConfig(C.Structure):
    _fields_ = [("block", Dims), ("n_double", I32), ("n_single", I32), ("lat_h", I32), ("lat_w", I32),
                ("channels", I32), ("txt_dim", I32), ("time_dim", I32), ("vec_in_dim", I32),
                ("single_parallel", I32)]


class FluxW(C.Structure):
    _fields_ = [("w_img_in", VP), ("b_img_in", VP), ("w_txt_in", VP), ("b_txt_in", VP), ("cond", CondW),
                ("double_img", PW), ("double_txt", PW), ("single", PW), ("w_ada", VP), ("b_ada", VP),
                ("w_out", VP), ("b_out", VP)]


PCOND, PFLUXC, PFLUXW = C.POINTER(CondW), C.POINTER(FluxConfig), C.POINTER(FluxW)

_SIGS = {
    "mmdit_last_error": (C.c_char_p, []),
    "mmdit_workspace_status": (C.c_int, [VP, C.POINTER(C.c_uint32), VP]),
    "mmdit_launch_count": (C.c_uint64, []),
    "mmdit_launch_count_reset": (None, []),
    "mmdit_profile_enable": (None, [I32]),
    "mmdit_profile_collect": (I32, [VP, C.c_char_p, SZ, C.POINTER(F32), I32]),
    "rope3d_freqs": (C.c_int, [VP, I32, I32, C.POINTER(I32), F32, VP, VP, VP]),
    "mmdit_modulation_fwd": (C.c_int, [I32, I32, I32, I32, VP, VP, VP, VP, VP]),
    "flow_match_workspace_size": (SZ, [I32, I64]),
    "flow_match_noise_and_loss": (C.c_int, [I32, VP, VP, VP, I32, I64, VP, VP, VP, VP, SZ, VP]),
    "flow_match_noise_and_loss_noalloc": (C.c_int, [I32, VP, VP, VP, I32, I64, VP, VP, VP, VP]),
    "flow_match_euler_step": (C.c_int, [I32, I64, VP, VP, VP, F32, F32, VP, VP]),
    "mmdit_linear_workspace_size": (SZ, [I32, I32, I32, I32]),
    "mmdit_linear_fwd": (C.c_int, [I32, I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_img_in_workspace_size": (SZ, [I32, I32, I32, I32, I32]),
    "mmdit_img_in_fwd": (C.c_int, [I32, I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_img_in_noise_fwd": (C.c_int, [I32, I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP, SZ,
                                         VP]),
    "mmdit_final_layer_workspace_size": (SZ, [PDIMS, I32]),
    "mmdit_final_layer_loss_workspace_size": (SZ, [PDIMS, I32]),
    "mmdit_final_layer_loss_fwd": (C.c_int, [PDIMS, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP,
                                             VP, VP, SZ, VP]),
    "mmdit_final_layer_fwd": (C.c_int, [PDIMS, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_ln_modulate_fwd": (C.c_int, [I32, I32, I32, I32, I32, F32, VP, VP, VP, I64, VP, VP]),
    "mmdit_copy_rows": (C.c_int, [VP, I64, VP, I64, I64, I32, VP]),
    "mmdit_attention_workspace_size": (SZ, [I32, I32, I32]),
    "mmdit_attention_fwd": (C.c_int, [I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_fp8_attention_workspace_size": (SZ, [I32, I32, I32]),
    "mmdit_fp8_attention_fwd": (C.c_int, [I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_double_block_workspace_size": (SZ, [PDIMS]),
    "mmdit_double_block_fwd": (C.c_int, [PDIMS, PW, PW, VP, VP, VP, VP, VP, VP, VP, PFP8, VP, SZ, VP]),
    "mmdit_single_block_workspace_size": (SZ, [PDIMS]),
    "mmdit_single_block_fwd": (C.c_int, [PDIMS, PW, VP, VP, VP, VP, VP, PFP8, VP, SZ, VP]),
    "mmdit_block_workspace_offsets": (I32, [PDIMS, I32, C.POINTER(I64), I32]),
    "mmdit_fp8_quantize_e4m3": (C.c_int, [VP, I64, VP, VP, VP, VP]),
    "mmdit_fp8_linear_workspace_size": (SZ, []),
    "mmdit_fp8_linear_fwd": (C.c_int, [I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_fp8_linear_bwd_workspace_size": (SZ, [I32, I32, I32, I32]),
    "mmdit_fp8_linear_bwd": (C.c_int, [I32, I32, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ,
                                       VP]),
    "mmdit_single_block_parallel_fwd": (C.c_int, [PDIMS, PW, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_linear_bwd_workspace_size": (SZ, [I32, I32, I32, I32]),
    "mmdit_linear_bwd": (C.c_int, [I32, I32, I32, I32, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_double_block_bwd_workspace_size": (SZ, [PDIMS]),
    "mmdit_double_block_bwd": (C.c_int, [PDIMS, PW, PW, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, PGRADS, PGRADS,
                                         VP, SZ, VP]),
    "mmdit_single_block_bwd_workspace_size": (SZ, [PDIMS]),
    "mmdit_single_block_bwd": (C.c_int, [PDIMS, PW, VP, VP, VP, VP, VP, VP, VP, PGRADS, VP, SZ, VP]),
    "mmdit_fp8_blockwise_linear_workspace_size": (SZ, [I32, I32, I32]),
    "mmdit_fp8_blockwise_linear_fwd": (C.c_int, [I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_fp8_mxfp8_linear_workspace_size": (SZ, [I32, I32, I32]),
    "mmdit_fp8_mxfp8_linear_fwd": (C.c_int, [I32, I32, I32, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_double_block_fwd_train": (C.c_int, [PDIMS, PW, PW, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_double_block_bwd_saved": (C.c_int, [PDIMS, PW, PW, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, PGRADS, PGRADS,
                                               VP, SZ, VP]),
    "mmdit_single_block_fwd_train": (C.c_int, [PDIMS, PW, VP, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_single_block_bwd_saved": (C.c_int, [PDIMS, PW, VP, VP, VP, VP, VP, VP, VP, PGRADS, VP, SZ, VP]),
    "mmdit_modulation_batched_fwd": (C.c_int, [I32, I32, I32, VP, I32, C.POINTER(GemvJob), VP]),
    "mmdit_conditioning_workspace_size": (SZ, [I32, I32, I32, I32]),
    "mmdit_conditioning_fwd": (C.c_int, [I32, I32, I32, I32, I32, PCOND, VP, VP, VP, VP, VP, SZ, VP]),
    "mmdit_flux_workspace_size": (SZ, [PFLUXC]),
    "mmdit_flux_forward": (C.c_int, [PFLUXC, PFLUXW, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
}

_lib = None


def library_path() -> str:
    return build_ext.LIB


def load() -> C.CDLL:
    """Load libmmdit.so (built by ``build_ext.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with diffusion_transformer_flux_gb300."
                               "build_ext.build() (there is no CPU fallback)")
        lib = C.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def last_error() -> str:
    return load().mmdit_last_error().decode()


def _check(status: int):
    if status != MMDIT_OK:
        raise MMDitError(status, last_error())


def _ptr(t) -> int | None:
    """Device address of a CUDA tensor (ints pass through).  Every tensor argument of the library is
    device memory (host-side arguments are ctypes structs and arrays), so a tensor on another device
    is refused here rather than handed to a kernel."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.device.type != "cuda":
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}: the library reads and writes "
                         "device memory")
    return t.data_ptr()


def _stream(stream=None) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def act_of(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MMDIT_BF16
    if t.dtype == torch.float32:
        return MMDIT_F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def make_dims(batch, seq_img, seq_txt, hidden, heads, mlp_hidden, act, head_dim=128, ln_eps=1e-6,
              rms_eps=1e-6, rope_interleaved=True, gelu_tanh=False, gemm=0) -> Dims:
    return Dims(batch, seq_img, seq_txt, hidden, heads, head_dim, mlp_hidden, ln_eps, rms_eps,
                int(rope_interleaved), int(gelu_tanh), act, gemm)


def make_stream_w(w: dict) -> StreamW:
    """The C view of one stream's weights; an optional "mod" entry is a precomputed
    modulation [B, 6D] fp32 (see mmdit_modulation_fwd)."""
    return StreamW(*[_ptr(w[n]) for n in STREAM_W_FIELDS], _ptr(w.get("mod")))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace: a zeroed uint8 device tensor (256-byte aligned by torch)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- entry points
def mmdit_workspace_status(ws, stream=None) -> int:
    bits = C.c_uint32(0)
    st = load().mmdit_workspace_status(_ptr(ws), C.byref(bits), _stream(stream))
    if st not in (MMDIT_OK, 6):
        _check(st)
    return bits.value


def mmdit_launch_count() -> int:
    return load().mmdit_launch_count()


def mmdit_launch_count_reset():
    load().mmdit_launch_count_reset()


def mmdit_profile_enable(on: bool):
    load().mmdit_profile_enable(int(bool(on)))


def mmdit_profile_collect(stream=None, max_entries=1 << 16) -> list:
    """[(step name, milliseconds), ...] recorded since the last collect (synchronises)."""
    names = C.create_string_buffer(max_entries * 32)
    ms = (F32 * max_entries)()
    n = load().mmdit_profile_collect(_stream(stream), names, len(names), ms, max_entries)
    if n < 0:
        raise MMDitError(4, "profile collection failed")
    labels = names.raw.split(b"\0")[:n]
    return [(labels[i].decode(), float(ms[i])) for i in range(n)]


def rope3d_freqs(ids, axes_dim, theta, cos_out, sin_out, stream=None):
    B, S, _ = ids.shape
    axes = (I32 * 3)(*axes_dim)
    _check(load().rope3d_freqs(_ptr(ids), B, S, axes, float(theta), _ptr(cos_out), _ptr(sin_out),
                               _stream(stream)))


def mmdit_modulation_fwd(vec, w, b, out, stream=None):
    """out [B, rows] fp32 = SiLU(vec) w^T + b (the AdaLN modulation linear)."""
    B, dim = vec.shape
    rows = w.shape[0]
    _check(load().mmdit_modulation_fwd(act_of(vec), B, rows, dim, _ptr(vec), _ptr(w), _ptr(b), _ptr(out),
                                       _stream(stream)))


def flow_match_workspace_size(batch, n_per_sample) -> int:
    return load().flow_match_workspace_size(batch, n_per_sample)


def flow_match_noise_and_loss(z0, z1, t, z_t=None, pred=None, loss=None, ws=None, stream=None):
    B = z0.shape[0]
    n = z0.numel() // B
    if ws is None:
        ws = workspace(flow_match_workspace_size(B, n), z0.device)
    _check(load().flow_match_noise_and_loss(act_of(z0), _ptr(z0), _ptr(z1), _ptr(t), B, n, _ptr(z_t),
                                            _ptr(pred), _ptr(loss), _ptr(ws), ws.numel(),
                                            _stream(stream)))
    return ws


def flow_match_noise_and_loss_noalloc(z0, z1, t, z_t=None, pred=None, loss=None, stream=None):
    """flow_match_noise_and_loss without a workspace (see include/mmdit.h)."""
    B = z0.shape[0]
    n = z0.numel() // B
    _check(load().flow_match_noise_and_loss_noalloc(act_of(z0), _ptr(z0), _ptr(z1), _ptr(t), B, n,
                                                    _ptr(z_t), _ptr(pred), _ptr(loss),
                                                    _stream(stream)))


def flow_match_euler_step(z, v_cond, v_uncond, guidance, dt, z_out, stream=None):
    """z_out = z - dt (v_uncond + guidance (v_cond - v_uncond)); v_uncond may be None."""
    _check(load().flow_match_euler_step(act_of(z), z.numel(), _ptr(z), _ptr(v_cond), _ptr(v_uncond),
                                        float(guidance), float(dt), _ptr(z_out), _stream(stream)))


def mmdit_linear_workspace_size(act, M, N, K) -> int:
    return load().mmdit_linear_workspace_size(act, M, N, K)


def mmdit_linear_fwd(x, w, b, y, ws=None, stream=None):
    M, K = x.reshape(-1, x.shape[-1]).shape
    N = w.shape[0]
    if ws is None:
        ws = workspace(mmdit_linear_workspace_size(act_of(x), M, N, K), x.device)
    _check(load().mmdit_linear_fwd(act_of(x), M, N, K, _ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(ws),
                                   ws.numel(), _stream(stream)))
    return ws


def mmdit_img_in_workspace_size(act, batch, channels, lat_h, lat_w) -> int:
    return load().mmdit_img_in_workspace_size(act, batch, channels, lat_h, lat_w)


def mmdit_img_in_fwd(z, w, b, out, ws=None, stream=None):
    B, Cc, H, W = z.shape
    act = act_of(w)
    if ws is None:
        ws = workspace(mmdit_img_in_workspace_size(act, B, Cc, H, W), z.device)
    _check(load().mmdit_img_in_fwd(act, B, Cc, H, W, w.shape[0], _ptr(z), _ptr(w), _ptr(b), _ptr(out),
                                   _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def mmdit_img_in_noise_fwd(z0, z1, t, w, b, out, z_t=None, ws=None, stream=None):
    """img_in of the noised latents z_t = (1 - t) z0 + t z1, formed while patchifying."""
    B, Cc, H, W = z0.shape
    act = act_of(w)
    if ws is None:
        ws = workspace(mmdit_img_in_workspace_size(act, B, Cc, H, W), z0.device)
    _check(load().mmdit_img_in_noise_fwd(act, B, Cc, H, W, w.shape[0], _ptr(z0), _ptr(z1), _ptr(t), _ptr(w),
                                         _ptr(b), _ptr(out), _ptr(z_t), _ptr(ws), ws.numel(),
                                         _stream(stream)))
    return ws


def mmdit_final_layer_workspace_size(dims: Dims, channels: int) -> int:
    return load().mmdit_final_layer_workspace_size(C.byref(dims), channels)


def mmdit_final_layer_fwd(dims: Dims, lat_h, lat_w, x_img, vec, w_ada, b_ada, w_out, b_out, pred,
                          ws=None, stream=None):
    channels = w_out.shape[0]
    if ws is None:
        ws = workspace(mmdit_final_layer_workspace_size(dims, channels), x_img.device)
    _check(load().mmdit_final_layer_fwd(C.byref(dims), channels, lat_h, lat_w, _ptr(x_img), _ptr(vec),
                                        _ptr(w_ada), _ptr(b_ada), _ptr(w_out), _ptr(b_out), _ptr(pred),
                                        _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def mmdit_final_layer_loss_workspace_size(dims: Dims, channels: int) -> int:
    return load().mmdit_final_layer_loss_workspace_size(C.byref(dims), channels)


def mmdit_final_layer_loss_fwd(dims: Dims, lat_h, lat_w, x_img, vec, w_ada, b_ada, w_out, b_out, z0, z1,
                               loss, pred=None, mod=None, ws=None, stream=None):
    """The output head with the flow-matching loss fused onto its last kernel."""
    channels = w_out.shape[0]
    if ws is None:
        ws = workspace(mmdit_final_layer_loss_workspace_size(dims, channels), x_img.device)
    _check(load().mmdit_final_layer_loss_fwd(C.byref(dims), channels, lat_h, lat_w, _ptr(x_img), _ptr(vec),
                                             _ptr(w_ada), _ptr(b_ada), _ptr(w_out), _ptr(b_out), _ptr(z0),
                                             _ptr(z1), _ptr(pred), _ptr(loss), _ptr(mod), _ptr(ws), ws.numel(),
                                             _stream(stream)))
    return ws


def mmdit_ln_modulate_fwd(x, shift, scale, out, mod_bstride, eps=1e-6, stream=None):
    """out = LN(x) (1 + scale[b]) + shift[b]; x [B, R, D] (bf16/fp32, or fp32 with a bf16 out)."""
    B, R, D = x.shape
    act = act_of(out)
    x_f32 = int(x.dtype == torch.float32 and act == MMDIT_BF16)
    _check(load().mmdit_ln_modulate_fwd(act, x_f32, B, R, D, float(eps), _ptr(x), _ptr(shift), _ptr(scale),
                                        int(mod_bstride), _ptr(out), _stream(stream)))


def mmdit_copy_rows(dst, dst_stride, src, src_stride, row_bytes, n_rows, stream=None):
    """Copy n_rows rows of row_bytes bytes between strided device buffers (strides in bytes)."""
    _check(load().mmdit_copy_rows(_ptr(dst), int(dst_stride), _ptr(src), int(src_stride), int(row_bytes),
                                  int(n_rows), _stream(stream)))


def mmdit_attention_workspace_size(batch, heads, seq) -> int:
    return load().mmdit_attention_workspace_size(batch, heads, seq)


def mmdit_attention_fwd(q, k, v, out, ws=None, stream=None):
    B, H, S, d = q.shape
    if ws is None:
        ws = workspace(mmdit_attention_workspace_size(B, H, S), q.device)
    _check(load().mmdit_attention_fwd(act_of(out), B, H, S, d, _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                      _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def mmdit_double_block_workspace_size(dims: Dims) -> int:
    return load().mmdit_double_block_workspace_size(C.byref(dims))


def mmdit_single_block_workspace_size(dims: Dims) -> int:
    return load().mmdit_single_block_workspace_size(C.byref(dims))


def mmdit_block_workspace_offsets(dims: Dims, single: bool) -> list:
    out = (I64 * 17)()
    n = load().mmdit_block_workspace_offsets(C.byref(dims), int(single), out, 17)
    if n < 0:
        raise MMDitError(1, "bad dims")
    return list(out)[:n]


def make_fp8_state(amax_history, scale, pos: int = 0, algo: int = AMAX_MOST_RECENT,
                   margin: int = 0) -> Fp8State:
    """The C view of a delayed-scaling state: amax_history [n_tensors, hist_len] and scale
    [n_tensors], fp32 device tensors the caller owns."""
    n, h = amax_history.shape
    return Fp8State(_ptr(amax_history), _ptr(scale), h, n, pos, algo, margin)


def _fp8_arg(fp8):
    return None if fp8 is None else C.byref(fp8)


def mmdit_double_block_fwd(dims: Dims, w_img: dict, w_txt: dict, vec, rope_cos, rope_sin, x_img,
                           x_txt, y_img, y_txt, ws=None, stream=None, fp8: Fp8State | None = None):
    if ws is None:
        ws = workspace(mmdit_double_block_workspace_size(dims), vec.device)
    wi, wt = make_stream_w(w_img), make_stream_w(w_txt)
    _check(load().mmdit_double_block_fwd(C.byref(dims), C.byref(wi), C.byref(wt), _ptr(vec),
                                         _ptr(rope_cos), _ptr(rope_sin), _ptr(x_img), _ptr(x_txt),
                                         _ptr(y_img), _ptr(y_txt), _fp8_arg(fp8), _ptr(ws),
                                         ws.numel(), _stream(stream)))
    return ws


def mmdit_single_block_fwd(dims: Dims, w: dict, vec, rope_cos, rope_sin, x, y, ws=None, stream=None,
                           fp8: Fp8State | None = None):
    if ws is None:
        ws = workspace(mmdit_single_block_workspace_size(dims), vec.device)
    ww = make_stream_w(w)
    _check(load().mmdit_single_block_fwd(C.byref(dims), C.byref(ww), _ptr(vec), _ptr(rope_cos),
                                         _ptr(rope_sin), _ptr(x), _ptr(y), _fp8_arg(fp8), _ptr(ws),
                                         ws.numel(), _stream(stream)))
    return ws


def mmdit_fp8_quantize_e4m3(x, scale, amax, out, stream=None):
    """out (uint8 E4M3 codes) = E4M3(x * scale); amax = max(amax, max|x|); x bf16."""
    _check(load().mmdit_fp8_quantize_e4m3(_ptr(x), x.numel(), _ptr(scale), _ptr(amax), _ptr(out),
                                          _stream(stream)))


def mmdit_fp8_linear_fwd(x_q, w_q, scale_x, scale_w, b, y, ws=None, stream=None):
    """y (bf16) = (x_q w_q^T) / (scale_x scale_w) + b on E4M3 codes x_q [M, K], w_q [N, K]."""
    M, K = x_q.shape
    N = w_q.shape[0]
    if ws is None:
        ws = workspace(load().mmdit_fp8_linear_workspace_size(), x_q.device)
    _check(load().mmdit_fp8_linear_fwd(M, N, K, _ptr(x_q), _ptr(w_q), _ptr(scale_x), _ptr(scale_w),
                                       _ptr(b), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


# ----------------------------------------------------------------------------- whole model
def mmdit_modulation_batched_fwd(vec, jobs, stream=None):
    """jobs: [(w, b, out), ...]; out_j [B, rows_j] fp32 = SiLU(vec) w_j^T + b_j, one launch."""
    B, dim = vec.shape
    arr = (GemvJob * max(len(jobs), 1))(*[GemvJob(_ptr(w), _ptr(b), _ptr(o), w.shape[0]) for w, b, o in jobs])
    _check(load().mmdit_modulation_batched_fwd(act_of(vec), B, dim, _ptr(vec), len(jobs), arr,
                                               _stream(stream)))


def make_cond_w(w: dict) -> CondW:
    """w["time_in"], w["vector_in"]: (w1, b1, w2, b2) device tensors; w["guidance_in"]: (w, b) or absent."""
    g = w.get("guidance_in") or (None, None)
    return CondW(MlpEmbedderW(*[_ptr(x) for x in w["time_in"]]),
                 MlpEmbedderW(*[_ptr(x) for x in w["vector_in"]]), _ptr(g[0]), _ptr(g[1]))


def mmdit_conditioning_workspace_size(act, batch, hidden, time_dim=256) -> int:
    return load().mmdit_conditioning_workspace_size(act, batch, hidden, time_dim)


def mmdit_conditioning_fwd(t, y, w: dict, vec, guidance=None, time_dim=256, ws=None, stream=None):
    """vec [B, D] = time MLP(sinusoid(1000 t)) + vector MLP(y) (+ guidance term)."""
    B, vec_in_dim = y.shape
    D = vec.shape[1]
    act = act_of(vec)
    if ws is None:
        ws = workspace(mmdit_conditioning_workspace_size(act, B, D, time_dim), vec.device)
    cw = make_cond_w(w)
    _check(load().mmdit_conditioning_fwd(act, B, D, time_dim, vec_in_dim, C.byref(cw), _ptr(t), _ptr(y),
                                         _ptr(guidance), _ptr(vec), _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def make_flux_config(dims: Dims, n_double, n_single, lat_h, lat_w, channels=64, txt_dim=4096,
                     time_dim=256, vec_in_dim=768, single_parallel=False) -> FluxConfig:
    return FluxConfig(dims, n_double, n_single, lat_h, lat_w, channels, txt_dim, time_dim, vec_in_dim,
                      int(bool(single_parallel)))


def make_flux_w(w: dict) -> FluxW:
    """The C view of the model's device weights (the layout of ``synth.flux_weights``)."""
    di = (StreamW * max(len(w["double"]), 1))(*[make_stream_w(a) for a, _ in w["double"]])
    dt = (StreamW * max(len(w["double"]), 1))(*[make_stream_w(b) for _, b in w["double"]])
    sg = (StreamW * max(len(w["single"]), 1))(*[make_stream_w(x) for x in w["single"]])
    f = w["final"]
    fw = FluxW(_ptr(w["img_in"][0]), _ptr(w["img_in"][1]), _ptr(w["txt_in"][0]), _ptr(w["txt_in"][1]),
               make_cond_w(w), C.cast(di, PW), C.cast(dt, PW), C.cast(sg, PW), _ptr(f["w_ada"]),
               _ptr(f["b_ada"]), _ptr(f["w_out"]), _ptr(f["b_out"]))
    fw._keep = (di, dt, sg)  # the arrays the struct points to live as long as it does
    return fw


def mmdit_flux_workspace_size(cfg: FluxConfig) -> int:
    return load().mmdit_flux_workspace_size(C.byref(cfg))


def mmdit_flux_forward(cfg: FluxConfig, w, z_t, txt, t, y, rope_cos, rope_sin, pred, guidance=None,
                       ws=None, stream=None):
    """pred = the whole model at (z_t, txt, t, y); ``w`` is a dict of device weights or a FluxW."""
    fw = w if isinstance(w, FluxW) else make_flux_w(w)
    if ws is None:
        ws = workspace(mmdit_flux_workspace_size(cfg), z_t.device)
    _check(load().mmdit_flux_forward(C.byref(cfg), C.byref(fw), _ptr(z_t), _ptr(txt), _ptr(t), _ptr(y),
                                     _ptr(guidance), _ptr(rope_cos), _ptr(rope_sin), _ptr(pred), _ptr(ws),
                                     ws.numel(), _stream(stream)))
    return ws


def mmdit_single_block_parallel_fwd(dims: Dims, w: dict, vec, rope_cos, rope_sin, x, y, ws=None, stream=None):
    """The parallel-branch single block: w["w_mod"] is [3D, D] (shift, scale, gate)."""
    if ws is None:
        ws = workspace(mmdit_single_block_workspace_size(dims), x.device)
    sw = make_stream_w(w)
    _check(load().mmdit_single_block_parallel_fwd(C.byref(dims), C.byref(sw), _ptr(vec), _ptr(rope_cos),
                                                  _ptr(rope_sin), _ptr(x), _ptr(y), _ptr(ws), ws.numel(),
                                                  _stream(stream)))
    return ws


def mmdit_linear_bwd_workspace_size(act, M, N, K) -> int:
    return load().mmdit_linear_bwd_workspace_size(act, M, N, K)


def mmdit_linear_bwd(dy, x, w, dx=None, dw=None, db=None, ws=None, stream=None):
    """Backward of y = x W^T + b: dx = dy W, dW = dy^T x (fp32), db = sum of dy (fp32)."""
    M, N = dy.reshape(-1, dy.shape[-1]).shape
    K = w.shape[1]
    act = act_of(dy)
    if ws is None:
        ws = workspace(mmdit_linear_bwd_workspace_size(act, M, N, K), dy.device)
    _check(load().mmdit_linear_bwd(act, M, N, K, _ptr(dy), _ptr(x), _ptr(w), _ptr(dx), _ptr(dw), _ptr(db),
                                   _ptr(ws), ws.numel(), _stream(stream)))
    return ws


# ----------------------------------------------------------------------------- block backward
def make_stream_grads(g: dict | None):
    """The C view of one stream's fp32 weight gradients (missing names: not computed)."""
    if g is None:
        return None
    return StreamGrads(*[_ptr(g.get(n)) for n in STREAM_W_FIELDS])


def mmdit_double_block_bwd_workspace_size(dims: Dims) -> int:
    return load().mmdit_double_block_bwd_workspace_size(C.byref(dims))


def mmdit_single_block_bwd_workspace_size(dims: Dims) -> int:
    return load().mmdit_single_block_bwd_workspace_size(C.byref(dims))


def mmdit_double_block_bwd(dims: Dims, w_img: dict, w_txt: dict, vec, cos, sin, x_img, x_txt, dy_img, dy_txt,
                           dx_img, dx_txt, dvec=None, g_img=None, g_txt=None, ws=None, stream=None):
    """Gradients of the double block (see include/mmdit.h); g_img / g_txt are dicts of fp32 tensors
    named like the weights."""
    if ws is None:
        ws = workspace(mmdit_double_block_bwd_workspace_size(dims), x_img.device)
    wi, wt = make_stream_w(w_img), make_stream_w(w_txt)
    gi, gt = make_stream_grads(g_img), make_stream_grads(g_txt)
    _check(load().mmdit_double_block_bwd(C.byref(dims), C.byref(wi), C.byref(wt), _ptr(vec), _ptr(cos), _ptr(sin),
                                         _ptr(x_img), _ptr(x_txt), _ptr(dy_img), _ptr(dy_txt), _ptr(dx_img),
                                         _ptr(dx_txt), _ptr(dvec), C.byref(gi) if gi else None,
                                         C.byref(gt) if gt else None, _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def mmdit_single_block_bwd(dims: Dims, w: dict, vec, cos, sin, x, dy, dx, dvec=None, g=None, ws=None,
                           stream=None):
    """Gradients of the single block (see include/mmdit.h)."""
    if ws is None:
        ws = workspace(mmdit_single_block_bwd_workspace_size(dims), x.device)
    sw = make_stream_w(w)
    gg = make_stream_grads(g)
    _check(load().mmdit_single_block_bwd(C.byref(dims), C.byref(sw), _ptr(vec), _ptr(cos), _ptr(sin), _ptr(x),
                                         _ptr(dy), _ptr(dx), _ptr(dvec), C.byref(gg) if gg else None, _ptr(ws),
                                         ws.numel(), _stream(stream)))
    return ws


def mmdit_fp8_blockwise_linear_fwd(x, w, b, y, ws=None, stream=None):
    """y = x W^T + b under the blockwise FP8 recipe (see include/mmdit.h); x [M, K], w [N, K], y [M, N]
    bf16.  Returns the workspace, whose layout the header states (codes and scales after the call)."""
    M, K = x.shape[-2], x.shape[-1]
    N = w.shape[0]
    if ws is None:
        ws = workspace(mmdit_fp8_blockwise_linear_workspace_size(M, N, K), x.device)
    _check(load().mmdit_fp8_blockwise_linear_fwd(M, N, K, _ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(ws), ws.numel(),
                                                 _stream(stream)))
    return ws


def mmdit_fp8_blockwise_linear_workspace_size(M, N, K) -> int:
    return load().mmdit_fp8_blockwise_linear_workspace_size(M, N, K)


def mmdit_fp8_mxfp8_linear_fwd(x, w, b, y, ws=None, stream=None):
    """y = x W^T + b under the MXFP8 recipe (see include/mmdit.h); x [M, K], w [N, K], y [M, N] bf16.
    Returns the workspace, whose layout the header states (values, codes and scales after the call)."""
    M, K = x.shape[-2], x.shape[-1]
    N = w.shape[0]
    if ws is None:
        ws = workspace(mmdit_fp8_mxfp8_linear_workspace_size(M, N, K), x.device)
    _check(load().mmdit_fp8_mxfp8_linear_fwd(M, N, K, _ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(ws), ws.numel(),
                                             _stream(stream)))
    return ws


def mmdit_fp8_mxfp8_linear_workspace_size(M, N, K) -> int:
    return load().mmdit_fp8_mxfp8_linear_workspace_size(M, N, K)


def mmdit_double_block_fwd_train(dims: Dims, w_img: dict, w_txt: dict, vec, cos, sin, x_img, x_txt, y_img, y_txt,
                                 saved=None, stream=None):
    """The training pair's forward (see include/mmdit.h): the block outputs, and in `saved` (a
    backward-sized workspace, returned) what mmdit_double_block_bwd_saved reads."""
    if saved is None:
        saved = workspace(mmdit_double_block_bwd_workspace_size(dims), x_img.device)
    wi, wt = make_stream_w(w_img), make_stream_w(w_txt)
    _check(load().mmdit_double_block_fwd_train(C.byref(dims), C.byref(wi), C.byref(wt), _ptr(vec), _ptr(cos), _ptr(sin),
                                               _ptr(x_img), _ptr(x_txt), _ptr(y_img), _ptr(y_txt), _ptr(saved),
                                               saved.numel(), _stream(stream)))
    return saved


def mmdit_double_block_bwd_saved(dims: Dims, w_img: dict, w_txt: dict, vec, cos, sin, x_img, x_txt, dy_img, dy_txt,
                                 dx_img, dx_txt, saved, dvec=None, g_img=None, g_txt=None, stream=None):
    """The training pair's backward: gradients from the state mmdit_double_block_fwd_train left."""
    wi, wt = make_stream_w(w_img), make_stream_w(w_txt)
    gi, gt = make_stream_grads(g_img), make_stream_grads(g_txt)
    _check(load().mmdit_double_block_bwd_saved(C.byref(dims), C.byref(wi), C.byref(wt), _ptr(vec), _ptr(cos), _ptr(sin),
                                               _ptr(x_img), _ptr(x_txt), _ptr(dy_img), _ptr(dy_txt), _ptr(dx_img),
                                               _ptr(dx_txt), _ptr(dvec), C.byref(gi) if gi else None,
                                               C.byref(gt) if gt else None, _ptr(saved), saved.numel(),
                                               _stream(stream)))


def mmdit_single_block_fwd_train(dims: Dims, w: dict, vec, cos, sin, x, y, saved=None, stream=None):
    """The single block's training forward (see mmdit_double_block_fwd_train)."""
    if saved is None:
        saved = workspace(mmdit_single_block_bwd_workspace_size(dims), x.device)
    sw = make_stream_w(w)
    _check(load().mmdit_single_block_fwd_train(C.byref(dims), C.byref(sw), _ptr(vec), _ptr(cos), _ptr(sin), _ptr(x),
                                               _ptr(y), _ptr(saved), saved.numel(), _stream(stream)))
    return saved


def mmdit_single_block_bwd_saved(dims: Dims, w: dict, vec, cos, sin, x, dy, dx, saved, dvec=None, g=None,
                                 stream=None):
    """The single block's training backward (see mmdit_double_block_bwd_saved)."""
    sw = make_stream_w(w)
    gg = make_stream_grads(g)
    _check(load().mmdit_single_block_bwd_saved(C.byref(dims), C.byref(sw), _ptr(vec), _ptr(cos), _ptr(sin), _ptr(x),
                                               _ptr(dy), _ptr(dx), _ptr(dvec), C.byref(gg) if gg else None,
                                               _ptr(saved), saved.numel(), _stream(stream)))


def mmdit_fp8_linear_bwd(dy, x_q, w_q, scale_x, scale_w, scale_dy, amax_dy, dx, dw=None, db=None, x=None,
                         recipe="e4m3", fp8_wgrad=True, ws=None, stream=None):
    """Backward of the FP8 linear (see include/mmdit.h); recipe "e4m3" or "hybrid"."""
    M, N = dy.shape
    K = w_q.shape[1]
    if ws is None:
        ws = workspace(load().mmdit_fp8_linear_bwd_workspace_size(M, N, K, int(fp8_wgrad)), dy.device)
    _check(load().mmdit_fp8_linear_bwd(M, N, K, {"e4m3": 0, "hybrid": 1}[recipe], int(fp8_wgrad), _ptr(dy),
                                       _ptr(x_q), _ptr(w_q), _ptr(x), _ptr(scale_x), _ptr(scale_w),
                                       _ptr(scale_dy), _ptr(amax_dy), _ptr(dx), _ptr(dw), _ptr(db), _ptr(ws),
                                       ws.numel(), _stream(stream)))
    return ws


def mmdit_fp8_attention_fwd(q, k, v, scale_q, scale_k, scale_v, out, ws=None, stream=None):
    """Joint attention on E4M3 operands (see include/mmdit.h); scales are device fp32 scalars."""
    B, H, S, d = q.shape
    if ws is None:
        ws = workspace(load().mmdit_fp8_attention_workspace_size(B, H, S), q.device)
    _check(load().mmdit_fp8_attention_fwd(act_of(out), B, H, S, d, _ptr(q), _ptr(k), _ptr(v), _ptr(scale_q),
                                          _ptr(scale_k), _ptr(scale_v), _ptr(out), _ptr(ws), ws.numel(),
                                          _stream(stream)))
    return ws
