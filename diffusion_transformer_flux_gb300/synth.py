"""Seeded synthetic inputs for the Flux MMDiT block forward.

This module only draws random numbers and builds integer/position structure.
It holds none of the block's arithmetic, so that the fp64 oracle (under
``oracle/``) and the CUDA path can both be fed from it without sharing any
of the computation they are compared on.

Generator: numpy PCG64.  Seeds: ``1000 + i`` for the inputs of workload ``i``
and ``2000 + i`` for its weights.  Every linear weight and bias is N(0, 0.02);
activations, the conditioning vector ``vec`` and latents are N(0, 1).  The
timestep ``t`` is U(0, 1) or logit-normal(0, 1); the latter is drawn as
``n ~ N(0, 1)`` and passed through the logistic function, which is how the
logit-normal sampler of the "Flux model API reference" (§Training utilities
› LogitNormalSampler) defines it.

Values handed to a bf16 kernel are rounded to bf16 here (round to nearest,
ties to even) and given to BOTH sides as the same numbers: the oracle sees
them as float64, the GPU as the identical bf16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "bf16_round", "bf16_bits", "f32_from_bf16_bits",
    "stream_weights", "position_ids", "timesteps", "block_inputs",
    "latent_pair", "final_layer_weights", "embed_weights",
]


@dataclass(frozen=True)
class Workload:
    """Shapes of one synthetic Flux-shaped workload."""
    name: str
    dtype: str            # "f32" (tf32 MMA), "bf16", or "fp8" (E4M3 linears, bf16 rest)
    batch: int
    lat_h: int            # latent rows   (image tokens = lat_h * lat_w, patch size 1)
    lat_w: int
    seq_txt: int
    hidden: int
    heads: int
    head_dim: int
    mlp_hidden: int
    blocks: tuple         # ("double",) or ("double", "single")
    channels: int = 64    # latent channels
    ctx_dim: int = 4096   # text-encoder width feeding txt_in (only when txt_from_ctx)
    txt_from_ctx: bool = False   # text tokens come from [B, S_t, ctx_dim] through txt_in
    img_from_latents: bool = False  # image tokens come from latents through img_in
    loss: bool = False     # output head + flow-matching loss on the image stream
    t_dist: str = "uniform"  # "uniform" | "logit_normal"
    index: int = 0
    n_double: int = 0     # whole-model workloads ("model" blocks): double and single block counts
    n_single: int = 0
    vec_dim: int = 768    # pooled text vector feeding the conditioning embedder

    @property
    def seq_img(self) -> int:
        return self.lat_h * self.lat_w

    @property
    def seq(self) -> int:
        return self.seq_img + self.seq_txt


WORKLOADS = {
    "tiny_double_f32": Workload(
        "tiny_double_f32", "f32", 1, 16, 16, 32, 256, 2, 128, 1024, ("double",), index=0),
    "flux535m_bf16": Workload(
        "flux535m_bf16", "bf16", 1, 64, 64, 512, 3072, 24, 128, 12288, ("double", "single"),
        txt_from_ctx=True, img_from_latents=True, loss=True, t_dist="logit_normal", index=1),
    "flux12b_512px_bf16": Workload(
        "flux12b_512px_bf16", "bf16", 4, 32, 32, 512, 3072, 24, 128, 12288, ("double",),
        img_from_latents=True, loss=True, t_dist="uniform", index=2),
    "flux12b_1024px_bf16": Workload(
        "flux12b_1024px_bf16", "bf16", 2, 64, 64, 512, 3072, 24, 128, 12288, ("double", "single"),
        img_from_latents=True, loss=True, t_dist="logit_normal", index=3),
    "flux12b_2048px_fp8": Workload(
        "flux12b_2048px_fp8", "fp8", 1, 128, 128, 512, 3072, 24, 128, 12288, ("double", "single"),
        index=4),
    "flux12b_512px_model": Workload(
        "flux12b_512px_model", "bf16", 1, 32, 32, 512, 3072, 24, 128, 12288, ("model",),
        txt_from_ctx=True, img_from_latents=True, loss=True, t_dist="uniform", index=5,
        n_double=19, n_single=38),
}


# --------------------------------------------------------------------------- bf16 rounding
def bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the uint16 bit patterns.

    Works in uint32: for every non-NaN pattern u, u + 0x7FFF + 1 stays below 2^32."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += u
    r += np.uint32(0x7FFF)
    r >>= np.uint32(16)
    nan = np.isnan(f)
    if nan.any():
        r[nan] = 0x7FC0
    return r.astype(np.uint16)


def f32_from_bf16_bits(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_round(x) -> np.ndarray:
    """float32 array holding the bf16-rounded values of ``x``."""
    return f32_from_bf16_bits(bf16_bits(x))


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as the kernels will see them: bf16-rounded for bf16/fp8 workloads, else fp32."""
    x = np.asarray(x, dtype=np.float32)
    return bf16_round(x) if dtype in ("bf16", "fp8") else x


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


# --------------------------------------------------------------------------- weights
def stream_weights(rng, hidden, heads, head_dim, mlp_hidden, dtype="bf16",
                   std=0.02, gain_jitter=0.0):
    """One stream's weight set, ``[out, in]`` row-major, as float32 arrays.

    Keys: w_mod [6D,D], b_mod [6D], w_qkv [3D,D] (q|k|v blocks, head-major inside),
    b_qkv [3D], g_q [d], g_k [d], w_o [D,D], b_o [D], w_1 [F,D], b_1 [F], w_2 [D,F], b_2 [D].
    QK-RMSNorm gains are 1 (plus N(0, gain_jitter) if asked).
    """
    D, F, d = hidden, mlp_hidden, head_dim
    assert heads * head_dim == hidden
    w = {
        "w_mod": _normal(rng, (6 * D, D), std), "b_mod": _normal(rng, (6 * D,), std),
        "w_qkv": _normal(rng, (3 * D, D), std), "b_qkv": _normal(rng, (3 * D,), std),
        "w_o": _normal(rng, (D, D), std), "b_o": _normal(rng, (D,), std),
        "w_1": _normal(rng, (F, D), std), "b_1": _normal(rng, (F,), std),
        "w_2": _normal(rng, (D, F), std), "b_2": _normal(rng, (D,), std),
    }
    g_q = np.ones(d, np.float32)
    g_k = np.ones(d, np.float32)
    if gain_jitter:
        g_q = g_q + _normal(rng, (d,), gain_jitter)
        g_k = g_k + _normal(rng, (d,), gain_jitter)
    w["g_q"], w["g_k"] = g_q, g_k
    return {k: _cast(v, dtype) for k, v in w.items()}


def embed_weights(rng, in_dim, hidden, dtype="bf16", std=0.02):
    """Linear ``in_dim -> hidden`` (img_in / txt_in): w [D, in], b [D]."""
    return {"w": _cast(_normal(rng, (hidden, in_dim), std), dtype),
            "b": _cast(_normal(rng, (hidden,), std), dtype)}


def final_layer_weights(rng, hidden, channels, dtype="bf16", std=0.02):
    """Output head: conditioning linear w_ada [2D, D], b_ada [2D]; projection w_out [C, D], b_out [C]."""
    return {"w_ada": _cast(_normal(rng, (2 * hidden, hidden), std), dtype),
            "b_ada": _cast(_normal(rng, (2 * hidden,), std), dtype),
            "w_out": _cast(_normal(rng, (channels, hidden), std), dtype),
            "b_out": _cast(_normal(rng, (channels,), std), dtype)}


def mlp_embedder_weights(rng, in_dim, hidden, dtype="bf16", std=0.02):
    """Two-layer embedder (timestep or pooled-vector MLP): w1 [D, in], b1 [D], w2 [D, D], b2 [D]."""
    return (_cast(_normal(rng, (hidden, in_dim), std), dtype), _cast(_normal(rng, (hidden,), std), dtype),
            _cast(_normal(rng, (hidden, hidden), std), dtype), _cast(_normal(rng, (hidden,), std), dtype))


def flux_weights(rng, hidden, heads, mlp_hidden, n_double, n_single, txt_dim=4096, vec_dim=768,
                 time_dim=256, channels=64, guidance=False, dtype="bf16", std=0.02, single_parallel=False):
    """Random weights of the whole model: embedders, ``n_double`` double blocks (an image and a
    text stream each), ``n_single`` single blocks and the output head.  ``single_parallel``: the
    single blocks take the parallel-branch form's three modulation chunks (the first 3D rows of
    the same draw)."""
    d = hidden // heads
    w = {"img_in": tuple(embed_weights(rng, channels, hidden, dtype, std).values()),
         "txt_in": tuple(embed_weights(rng, txt_dim, hidden, dtype, std).values()),
         "time_in": mlp_embedder_weights(rng, time_dim, hidden, dtype, std),
         "vector_in": mlp_embedder_weights(rng, vec_dim, hidden, dtype, std)}
    if guidance:
        w["guidance_in"] = (_cast(_normal(rng, (hidden,), std), dtype), _cast(_normal(rng, (hidden,), std), dtype))
    w["double"] = [(stream_weights(rng, hidden, heads, d, mlp_hidden, dtype, std),
                    stream_weights(rng, hidden, heads, d, mlp_hidden, dtype, std)) for _ in range(n_double)]
    w["single"] = [stream_weights(rng, hidden, heads, d, mlp_hidden, dtype, std) for _ in range(n_single)]
    if single_parallel:
        for ws in w["single"]:
            ws["w_mod"], ws["b_mod"] = ws["w_mod"][:3 * hidden].copy(), ws["b_mod"][:3 * hidden].copy()
    w["final"] = final_layer_weights(rng, hidden, channels, dtype, std)
    return w


# --------------------------------------------------------------------------- structure
def position_ids(batch, lat_h, lat_w, seq_txt, img_first=True) -> np.ndarray:
    """Token ids ``[B, S, 3]`` (float32) in the joint order [image; text].

    Image token ``r * lat_w + c`` gets (0, r, c); text tokens get (0, 0, 0).
    """
    r, c = np.meshgrid(np.arange(lat_h), np.arange(lat_w), indexing="ij")
    img = np.stack([np.zeros(lat_h * lat_w), r.reshape(-1), c.reshape(-1)], axis=-1)
    txt = np.zeros((seq_txt, 3))
    ids = np.concatenate([img, txt] if img_first else [txt, img], axis=0).astype(np.float32)
    return np.broadcast_to(ids, (batch,) + ids.shape).copy()


def timesteps(rng, batch, dist="uniform") -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(0.0, 1.0, size=batch).astype(np.float32)
    if dist == "logit_normal":
        n = rng.standard_normal(size=batch)
        return (1.0 / (1.0 + np.exp(-n))).astype(np.float32)
    raise ValueError(dist)


def latent_pair(rng, batch, channels, lat_h, lat_w):
    """Clean latent z0 and noise z1, both N(0,1), ``[B, C, H, W]`` float32."""
    z0 = _normal(rng, (batch, channels, lat_h, lat_w))
    z1 = _normal(rng, (batch, channels, lat_h, lat_w))
    return z0, z1


@dataclass
class BlockInputs:
    x_img: np.ndarray
    x_txt: np.ndarray
    vec: np.ndarray
    ids: np.ndarray
    extra: dict = field(default_factory=dict)


def block_inputs(batch, seq_img, seq_txt, hidden, dtype, seed, lat_hw=None) -> BlockInputs:
    """Residual-stream activations N(0,1), ``vec`` N(0,1) and position ids for one block call."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x_img = _cast(_normal(rng, (batch, seq_img, hidden)), dtype)
    x_txt = _cast(_normal(rng, (batch, seq_txt, hidden)), dtype)
    vec = _cast(_normal(rng, (batch, hidden)), dtype)
    if lat_hw is None:
        # a near-square grid for the image ids; a ragged last row is fine
        w = int(np.ceil(np.sqrt(seq_img)))
        rr = np.arange(seq_img) // w
        cc = np.arange(seq_img) % w
        img = np.stack([np.zeros(seq_img), rr, cc], -1)
        ids = np.concatenate([img, np.zeros((seq_txt, 3))], 0).astype(np.float32)
        ids = np.broadcast_to(ids, (batch,) + ids.shape).copy()
    else:
        ids = position_ids(batch, lat_hw[0], lat_hw[1], seq_txt)
    return BlockInputs(x_img, x_txt, vec, ids)
