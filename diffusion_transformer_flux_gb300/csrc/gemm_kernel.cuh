// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM  C = A * W^T  with fused
// epilogues, for sm_103a.
//
// One CTA per SM walks a static list of 128 x BN output tiles.  Roles:
//   warp 0      TMA producer: streams 128-byte-wide K slices of A and W into a ring of shared-
//               memory stages (128-byte swizzle, the layout the tensor core reads directly);
//   warp 1      MMA issuer (one thread): tcgen05.mma into a double-buffered fp32 accumulator in
//               tensor memory (TMEM), so the epilogue of tile i overlaps the main loop of i+1;
//   warps 2..5  epilogue: tcgen05.ld of one accumulator row per thread, fused math, stores.
// Every wait is bounded (common.cuh); on a give-up the CTA drains what it started and exits.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace mmdit {

constexpr int kBM = 128;
constexpr int kGemmThreads = 192;

template <int KIND>
struct KindTraits;
template <>
struct KindTraits<kKindF16> {
  using T = __nv_bfloat16;
  static constexpr int kEltBytes = 2;
};
template <>
struct KindTraits<kKindTF32> {
  using T = float;
  static constexpr int kEltBytes = 4;
};

template <int BN>
struct GemmCfg {
  static constexpr int kStages = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kBarrierBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024;
};

// ----------------------------------------------------------------------------- vector I/O
__device__ __forceinline__ void load32(const __nv_bfloat16* p, float (&v)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = __ldg(q + i);
    v[8 * i + 0] = bf16_lo(u.x), v[8 * i + 1] = bf16_hi(u.x);
    v[8 * i + 2] = bf16_lo(u.y), v[8 * i + 3] = bf16_hi(u.y);
    v[8 * i + 4] = bf16_lo(u.z), v[8 * i + 5] = bf16_hi(u.z);
    v[8 * i + 6] = bf16_lo(u.w), v[8 * i + 7] = bf16_hi(u.w);
  }
}
__device__ __forceinline__ void load32(const float* p, float (&v)[32]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 u = __ldg(q + i);
    v[4 * i] = u.x, v[4 * i + 1] = u.y, v[4 * i + 2] = u.z, v[4 * i + 3] = u.w;
  }
}
__device__ __forceinline__ void store32(__nv_bfloat16* p, const float (&v)[32]) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    q[i] = u;
  }
}
__device__ __forceinline__ void store32(float* p, const float (&v)[32]) {
  float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ float gelu_f(float x, int tanh_form) {
  if (tanh_form) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * x * (1.f + tanhf(k0 * (x + 0.044715f * x * x * x)));
  }
  return 0.5f * x * (1.f + erff(x * 0.7071067811865476f));
}

// Loads 32 accumulator columns [col, col+32) of this thread's TMEM lane as floats.
__device__ __forceinline__ void tmem_load_f32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ----------------------------------------------------------------------------- epilogues
// Row-wise epilogue of one 128 x BN accumulator tile.  `m` is this thread's output row, `n0`
// the tile's first column.  All 32 lanes of the warp must call this (tcgen05.ld is collective).
template <typename T, int BN, int EPI>
__device__ __forceinline__ void gemm_epilogue(uint32_t taddr, int m, int n0, int M, int N,
                                              const EpiArgs& ep) {
  const bool row_ok = m < M;
  if constexpr (EPI == kEpiQkv) {
    // BN covers whole heads (128 columns each); q|k|v blocks are `hidden` columns wide.
    const int b = row_ok ? m / ep.rows_per_batch : 0;
    const int sj = (row_ok ? m % ep.rows_per_batch : 0) + ep.seq_offset;
#pragma unroll 1
    for (int hh = 0; hh < BN / 128; ++hh) {
      const int nh = n0 + hh * 128;
      if (nh >= N) break;
      const int which = nh / ep.hidden;
      const int head = (nh % ep.hidden) >> 7;
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float t[32];
        tmem_load_f32(taddr + hh * 128 + c * 32, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = t[i];
      }
      if (!row_ok) continue;
      if (ep.bias) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float bb[32];
          load32(reinterpret_cast<const T*>(ep.bias) + nh + c * 32, bb);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c * 32 + i] += bb[i];
        }
      }
      const size_t bh = static_cast<size_t>(b) * ep.heads + head;
      if (which < 2) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 128; ++i) ss = fmaf(v[i], v[i], ss);
        const float r = rsqrtf(ss * (1.f / 128.f) + ep.rms_eps);
        const T* g = reinterpret_cast<const T*>(which == 0 ? ep.g_q : ep.g_k);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float gg[32];
          load32(g + c * 32, gg);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c * 32 + i] *= r * gg[i];
        }
        const size_t rope_row = (static_cast<size_t>(b) * ep.seq_joint + sj) * 64;
        const float* cs = ep.rope_cos + rope_row;
        const float* sn = ep.rope_sin + rope_row;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float cc[32], ssn[32];
          load32(cs + c * 32, cc);
          load32(sn + c * 32, ssn);
          // pair j = c*32 + i rotates (v[2j], v[2j+1]) or, half-split, (v[j], v[j+64])
          if (ep.rope_interleaved) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int j = c * 32 + i;
              const float x0 = v[2 * j], x1 = v[2 * j + 1];
              v[2 * j] = x0 * cc[i] - x1 * ssn[i];
              v[2 * j + 1] = x0 * ssn[i] + x1 * cc[i];
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int j = c * 32 + i;
              const float x0 = v[j], x1 = v[j + 64];
              v[j] = x0 * cc[i] - x1 * ssn[i];
              v[j + 64] = x0 * ssn[i] + x1 * cc[i];
            }
          }
        }
        __nv_bfloat16* dst = (which == 0 ? ep.q : ep.k) + (bh * ep.seq_joint + sj) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float t[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = v[c * 32 + i];
          store32(dst + c * 32, t);
        }
      } else {
        __nv_bfloat16* dst = ep.vt + bh * 128 * static_cast<size_t>(ep.seq_pad) + sj;
#pragma unroll
        for (int j = 0; j < 128; ++j) dst[static_cast<size_t>(j) * ep.seq_pad] = __float2bfloat16_rn(v[j]);
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int n = n0 + c * 32;
      if (n >= N) break;  // uniform across the warp
      float v[32];
      tmem_load_f32(taddr + c * 32, v);
      if (!row_ok) continue;
      if (ep.bias) {
        float bb[32];
        load32(reinterpret_cast<const T*>(ep.bias) + n, bb);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bb[i];
      }
      if constexpr (EPI == kEpiGelu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i], ep.gelu_tanh);
      }
      if constexpr (EPI == kEpiGateResid) {
        const int b = m / ep.rows_per_batch;
        float g[32], x[32];
        load32(ep.gate + static_cast<size_t>(b) * ep.gate_bstride + n, g);
        load32(reinterpret_cast<const T*>(ep.resid) + static_cast<size_t>(m) * N + n, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaf(g[i], v[i], x[i]);
      }
      if constexpr (EPI == kEpiUnpatchify) {
        const int b = m / ep.rows_per_batch, s = m % ep.rows_per_batch;
        float* dst = reinterpret_cast<float*>(ep.out) +
                     (static_cast<size_t>(b) * N + n) * ep.rows_per_batch + s;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(i) * ep.rows_per_batch] = v[i];
      } else {
        store32(reinterpret_cast<T*>(ep.out) + static_cast<size_t>(m) * N + n, v);
      }
    }
  }
}

}  // namespace mmdit
