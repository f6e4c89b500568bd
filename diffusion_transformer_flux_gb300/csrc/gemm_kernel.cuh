// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM  C = A * W^T  with fused
// epilogues, for sm_103a.
//
// One CTA per SM walks a static list of 128 x BN output tiles.  Roles:
//   warp 0      TMA producer: streams 128-byte-wide K slices of A and W into a ring of shared-
//               memory stages (128-byte swizzle, the layout the tensor core reads directly);
//   warp 1      MMA issuer (one thread): tcgen05.mma into a double-buffered fp32 accumulator in
//               tensor memory (TMEM), so the epilogue of tile i overlaps the main loop of i+1;
//   warps 2..   epilogue: one or two warps per TMEM lane quarter (two split the tile's columns
//               for the GELU epilogue); tcgen05.ld of one accumulator row per thread, fused
//               math, stores.
// Every wait is bounded (common.cuh); on a give-up the CTA drains what it started and exits.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace mmdit {

constexpr int kBM = 128;
// Epilogue warp groups splitting the tile columns: two where the epilogue would otherwise
// outlast the next tile's main loop (GELU; the bias-only epilogue of short-K GEMMs such as the
// image embedding), one for the others.
template <int EPI>
struct EpiGroups {
  static constexpr int value =
      (EPI == kEpiGelu || EPI == kEpiGeluF8 || EPI == kEpiBias || EPI == kEpiDGelu || EPI == kEpiGateResid) ? 2 : 1;
};
template <int EPI>
constexpr int gemm_threads() {
  return 64 + 128 * EpiGroups<EPI>::value;
}

// Operand element size and the element type of the epilogue's bias, residual and output.
template <int KIND>
struct KindTraits;
template <>
struct KindTraits<kKindF16> {
  using TE = __nv_bfloat16;
  static constexpr int kEltBytes = 2;
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <>
struct KindTraits<kKindTF32> {
  using TE = float;
  static constexpr int kEltBytes = 4;
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <>
struct KindTraits<kKindF8> {  // E4M3 operands, bf16 activations around them
  using TE = __nv_bfloat16;
  static constexpr int kEltBytes = 1;
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_UINT8;
};

template <>
struct KindTraits<kKindF8E5M2> {  // E5M2 A (a gradient), E4M3 B, bf16 or fp32 output
  using TE = __nv_bfloat16;
  static constexpr int kEltBytes = 1;
  static constexpr CUtensorMapDataType kMapType = CU_TENSOR_MAP_DATA_TYPE_UINT8;
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

// GELU(x) = x * Phi(x) = 0.5 x (1 + erf(x / sqrt(2))), with erf from formula 7.1.26 of
// Abramowitz & Stegun, "Handbook of Mathematical Functions" (absolute error <= 1.5e-7 for
// z >= 0):  erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),  t = 1/(1 + p z).
// With q = (a1 t + ... + a5 t^5) exp(-z^2) at z = |x| / sqrt(2), 1 + erf(x / sqrt(2)) is 2 - q
// for x >= 0 and q for x < 0.  The reciprocal and the exponential use the hardware
// approximations (relative error near 2^-22), so GELU's relative error stays near 1e-7, far
// below the bf16 output's 2^-9.  Two MUFU operations and eight FMA-class ones per element.
constexpr float kAsP = 0.3275911f;
constexpr float kAsA1 = 0.254829592f, kAsA2 = -0.284496736f, kAsA3 = 1.421413741f;
constexpr float kAsA4 = -1.453152027f, kAsA5 = 1.061405429f;

__device__ __forceinline__ float gelu_erf(float x) {
  const float z = fabsf(x) * 0.7071067811865476f;  // |x| / sqrt(2)
  const float t = fast_rcp(fmaf(kAsP, z, 1.f));
  float poly = fmaf(t, kAsA5, kAsA4);
  poly = fmaf(t, poly, kAsA3);
  poly = fmaf(t, poly, kAsA2);
  poly = fmaf(t, poly, kAsA1);
  const float q = poly * t * fast_exp2(-z * z * 1.4426950408889634f);  // exp(-z^2)
  return 0.5f * x * (x >= 0.f ? 2.f - q : q);
}

__device__ __forceinline__ float gelu_f(float x, int tanh_form) {
  if (tanh_form) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * x * (1.f + tanhf(k0 * (x + 0.044715f * x * x * x)));
  }
  return gelu_erf(x);
}

// Loads 32 accumulator columns [col, col+32) of this thread's TMEM lane as floats.
__device__ __forceinline__ void tmem_load_f32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32_wait(taddr, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ----------------------------------------------------------------------------- epilogues
// Row-wise epilogue of one 128 x BN accumulator tile.  `m` is this thread's output row, `n0`
// the tile's first column.  All 32 lanes of the warp must call this (tcgen05.ld is collective).
// `group` selects which part of the tile's columns (or heads) this warp handles.
// With DEQ (E4M3 operands) the accumulator is multiplied by 1 / (scale_a * scale_w) first.
template <typename T, int BN, int EPI, bool DEQ>
__device__ __forceinline__ void gemm_epilogue(int group, uint32_t taddr, int m, int n0, int M, int N,
                                              const EpiArgs& ep) {
  const bool row_ok = m < M;
  const float dq = DEQ ? 1.f / (__ldg(ep.scale_a) * __ldg(ep.scale_w)) : 1.f;
  if constexpr (EPI == kEpiQkv) {
    // BN covers whole heads (128 columns each); q|k|v blocks are `hidden` columns wide.
    const int b = row_ok ? m / ep.rows_per_batch : 0;
    const int sj = (row_ok ? m % ep.rows_per_batch : 0) + ep.seq_offset;
#pragma unroll 1
    for (int hh = group; hh < BN / 128; hh += EpiGroups<EPI>::value) {
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
      if constexpr (DEQ) {
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] *= dq;
      }
      if (ep.bias) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float bb[32];
          load32(reinterpret_cast<const T*>(ep.bias) + nh + c * 32, bb);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c * 32 + i] += bb[i];
        }
      }
      if (ep.pre) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float t[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] = v[c * 32 + i];
          store32(reinterpret_cast<T*>(ep.pre) + static_cast<size_t>(m) * N + nh + c * 32, t);
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
        // V is a bf16 value of the attention (autocast precision); it is stored in fp16, which
        // holds every such value exactly, because the PV product runs on fp16 operands
        __half* dst = ep.vt + bh * 128 * static_cast<size_t>(ep.seq_pad) + sj;
#pragma unroll
        for (int j = 0; j < 128; ++j)
          dst[static_cast<size_t>(j) * ep.seq_pad] = __float2half_rn(__bfloat162float(__float2bfloat16_rn(v[j])));
      }
    }
  } else {
    constexpr int kChunks = BN / 32;
    constexpr int kPer = (kChunks + EpiGroups<EPI>::value - 1) / EpiGroups<EPI>::value;
    float amax = 0.f;  // kEpiGeluF8: largest |GELU(.)| this thread wrote
    for (int c = group * kPer; c < (group + 1) * kPer && c < kChunks; ++c) {
      const int n = n0 + c * 32;
      if (n >= N) break;  // uniform across the warp
      float v[32];
      tmem_load_f32(taddr + c * 32, v);
      if (!row_ok) continue;
      if constexpr (DEQ) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= dq;
      }
      if constexpr (EPI == kEpiPartial) {
        store32(reinterpret_cast<float*>(ep.out) + static_cast<size_t>(m) * N + n, v);
        continue;
      }
      if (ep.bias) {
        float bb[32];
        load32(reinterpret_cast<const T*>(ep.bias) + n, bb);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bb[i];
      }
      if constexpr (EPI == kEpiGelu || EPI == kEpiGateResid) {
        if (ep.pre) store32(reinterpret_cast<T*>(ep.pre) + static_cast<size_t>(m) * N + n, v);
      }
      if constexpr (EPI == kEpiDGelu) {
        float u[32];
        load32(reinterpret_cast<const T*>(ep.aux) + static_cast<size_t>(m) * N + n, u);
        if (ep.gelu_tanh) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gelu_grad_f(u[i], 1);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gelu_grad_f(u[i], 0);
        }
      }
      if constexpr (EPI == kEpiGelu || EPI == kEpiGeluF8) {
        // the variant is chosen once per chunk so the 32 evaluations interleave
        if (ep.gelu_tanh) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i], 1);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i], 0);
        }
      }
      if constexpr (EPI == kEpiGateResid) {
        const int b = m / ep.rows_per_batch;
        float g[32], x[32];
        load32(ep.gate + static_cast<size_t>(b) * ep.gate_bstride + n, g);
        if (ep.resid_f32)
          load32(reinterpret_cast<const float*>(ep.resid) + static_cast<size_t>(m) * N + n, x);
        else
          load32(reinterpret_cast<const T*>(ep.resid) + static_cast<size_t>(m) * N + n, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaf(g[i], v[i], x[i]);
      }
      if constexpr (EPI == kEpiGeluF8) {
        const float qs = __ldg(ep.out_scale);
        uint2 u[4];
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = e4m3x8(v + 8 * i, qs);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(ep.out) + static_cast<size_t>(m) * N + n);
        dst[0] = make_uint4(u[0].x, u[0].y, u[1].x, u[1].y);
        dst[1] = make_uint4(u[2].x, u[2].y, u[3].x, u[3].y);
      } else if constexpr (EPI == kEpiUnpatchify) {
        const int b = m / ep.rows_per_batch, s = m % ep.rows_per_batch;
        float* dst = reinterpret_cast<float*>(ep.out) +
                     (static_cast<size_t>(b) * N + n) * ep.rows_per_batch + s;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(i) * ep.rows_per_batch] = v[i];
      } else if (ep.out_f32) {
        store32(reinterpret_cast<float*>(ep.out) + static_cast<size_t>(m) * N + n, v);
      } else {
        store32(reinterpret_cast<T*>(ep.out) + static_cast<size_t>(m) * N + n, v);
      }
    }
    if constexpr (EPI == kEpiGeluF8) {
      amax = warp_max(amax);
      if ((threadIdx.x & 31) == 0 && amax > 0.f) atomic_max_nonneg(ep.out_amax, amax);
    }
  }
}


// ----------------------------------------------------------------------------- kernel
template <int KIND, int BN, int EPI>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_b0,
                   const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_b1,
                   int M0, int M1, int N, int K, int splits, const __grid_constant__ EpiArgs ep0,
                   const __grid_constant__ EpiArgs ep1, uint32_t* status) {
  using Cfg = GemmCfg<BN>;
  using TE = typename KindTraits<KIND>::TE;
  constexpr int kBK = 128 / KindTraits<KIND>::kEltBytes;     // elements per 128-byte K slice
  constexpr int kUmmaK = 32 / KindTraits<KIND>::kEltBytes;   // K of one tcgen05.mma
  constexpr int kKSteps = kBK / kUmmaK;
  constexpr uint32_t kIdesc = make_idesc<KIND>(kBM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* tfull = empty + Cfg::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (K + kBK - 1) / kBK;
  // Two problems of equal N and K share the launch (e.g. the image and text streams); the tile
  // list holds problem 0's tiles, M fastest, then problem 1's.
  const int num_n = (N + BN - 1) / BN;
  const int num_m0 = (M0 + kBM - 1) / kBM, num_m1 = (M1 + kBM - 1) / kBM;
  const int tiles0 = num_m0 * num_n;
  const int tiles = tiles0 + num_m1 * num_n;
  // split-K: work item w covers tile w % tiles over the split's range of K slices
  const int num_tiles = tiles * splits;
  const int kb_per_split = (num_kb + splits - 1) / splits;
  auto decode = [&](int item, int& prob, int& mb, int& nb) {
    const int tile = item % tiles;
    prob = tile >= tiles0;
    const int t = prob ? tile - tiles0 : tile;
    const int nm = prob ? num_m1 : num_m0;
    mb = t % nm, nb = t / nm;
  };
  auto k_range = [&](int item, int& kb0, int& kb1) {
    const int split = item / tiles;
    kb0 = split * kb_per_split;
    kb1 = kb0 + kb_per_split < num_kb ? kb0 + kb_per_split : num_kb;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], 1);
    for (int a = 0; a < 2; ++a) mbar_init(&tfull[a], 1), mbar_init(&tempty[a], 32 * 4 * EpiGroups<EPI>::value);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the set-up above overlapped the previous kernel; its results are visible now
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tm_a0);
      tma_prefetch_desc(&tm_b0);
      if (M1 > 0) tma_prefetch_desc(&tm_a1), tma_prefetch_desc(&tm_b1);
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[Cfg::kStages];
      for (int s = 0; s < Cfg::kStages; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int prob, mb, nb;
        decode(tile, prob, mb, nb);
        const CUtensorMap* ma = prob ? &tm_a1 : &tm_a0;
        const CUtensorMap* mw = prob ? &tm_b1 : &tm_b0;
        int kb0, kb1;
        k_range(tile, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, status, kErrGemmWait)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
          tma_load_2d(sa, ma, &full[stage], kb * kBK, mb * kBM);
          tma_load_2d(sa + Cfg::kABytes, mw, &full[stage], kb * kBK, nb * BN);
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == Cfg::kStages) stage = 0, phase ^= 1;
        }
      }
      if (*abort_flag) {
        // Give the copies already issued a bounded chance to land before the CTA exits.
        int never = 0;
        for (int s = 0; s < Cfg::kStages; ++s)
          if (last_parity[s] >= 0)
            mbar_wait(&full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, status, kErrGemmWait)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        int kb0, kb1;
        k_range(tile, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, status, kErrGemmWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kKSteps; ++k)
            tc_mma<KIND>(d_tmem, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32),
                         kIdesc, (kb != kb0 || k != 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == Cfg::kStages) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (*abort_flag) {
        // Wait (bounded) for every MMA issued so far before TMEM is released.
        int never = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &never, status, 0);
      }
    }
  } else {
    // ---------------- epilogue warps 2..; warp w reads TMEM lanes 32*(w%4) .. +31 and takes
    // the part of the columns given by its group (warps 2..5: group 0, 6..9: group 1)
    const int quarter = warp & 3;
    const int group = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int prob, mb, nb;
      decode(tile, prob, mb, nb);
      bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, status, kErrGemmWait);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      // a private copy, so the epilogue's arguments live in registers rather than being
      // re-read from parameter space around every store
      EpiArgs ep = prob ? ep1 : ep0;
      if constexpr (EPI == kEpiPartial)
        ep.out = reinterpret_cast<float*>(ep.out) +
                 static_cast<size_t>(tile / tiles) * static_cast<size_t>(prob ? M1 : M0) * N;
      gemm_epilogue<TE, BN, EPI, (KIND == kKindF8 || KIND == kKindF8E5M2)>(group, taddr, mb * kBM + row, nb * BN,
                                                  prob ? M1 : M0, N, ep);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ----------------------------------------------------------------------------- host side
template <int KIND, int BN, int EPI>
cudaError_t run_gemm(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  using Cfg = GemmCfg<BN>;
  constexpr int kElt = KindTraits<KIND>::kEltBytes;
  constexpr int kBK = 128 / kElt;
  const CUtensorMapDataType dt = KindTraits<KIND>::kMapType;
  const bool two = p.M1 > 0;
  if (two && p.K1 > 0 && p.K1 != p.K) return cudaErrorInvalidValue;  // one K for both problems here
  CUtensorMap ta0, tb0, ta1, tb1;
  const uint64_t stride[1] = {static_cast<uint64_t>(p.K) * kElt};
  const uint32_t box_a[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
  const uint32_t box_b[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(BN)};
  const uint64_t da0[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
  const uint64_t db[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
  const uint64_t da1[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(two ? p.M1 : p.M)};
  if (!encode_tmap(&ta0, dt, 2, p.A, da0, stride, box_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tb0, dt, 2, p.W, db, stride, box_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&ta1, dt, 2, two ? p.A1 : p.A, da1, stride, box_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tb1, dt, 2, two ? p.W1 : p.W, db, stride, box_b, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = gemm_tc_kernel<KIND, BN, EPI>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int num_n = (p.N + BN - 1) / BN;
  const int splits = EPI == kEpiPartial ? (p.splits > 1 ? p.splits : 1) : 1;
  const int tiles = ((p.M + kBM - 1) / kBM + (two ? (p.M1 + kBM - 1) / kBM : 0)) * num_n * splits;
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  {
    const cudaError_t e_ = launch_pdl(kern, dim3(grid), dim3(gemm_threads<EPI>()), Cfg::kSmemBytes, stream, ta0,
                                        tb0, ta1, tb1, p.M, two ? p.M1 : 0, p.N, p.K, splits, p.ep,
                                        two ? p.ep1 : p.ep, status);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

template <int KIND, int BN, int EPI, int MAJ = 0>
cudaError_t run_gemm_pair(const GemmProblem& p, uint32_t* status, cudaStream_t stream);

// GEMMs that take the CTA-pair kernel (gemm_pair.cuh): the block linears' epilogues and plain
// bias outputs (embeddings, the backward's GEMMs), N a multiple of 256, and enough rows for the
// 256-row tiles to pay.
inline bool use_pair(const GemmProblem& p) {
  // (a plain-bias GEMM with a short K, such as img_in's 64, is one k-step: the pair's set-up
  // does not pay there)
  const bool epi_ok = p.epi == kEpiQkv || p.epi == kEpiGateResid || p.epi == kEpiGelu || p.epi == kEpiGeluF8 ||
                      (p.epi == kEpiBias && p.K >= 512);
  const bool qkv_ok = p.epi != kEpiQkv || p.ep.hidden % 256 == 0;
  return epi_ok && qkv_ok && p.N % 256 == 0 && p.M + p.M1 >= 512;
}

// Picks the tile width for N and the epilogue, then launches.
template <int KIND>
cudaError_t dispatch_gemm(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  if (p.a_mn || p.b_mn) {
    // transposed operands: the pair kernel's plain-bias products only
    if constexpr (KIND == kKindF16) {
      if ((p.epi != kEpiBias && p.epi != kEpiDGelu) || p.N % 256 != 0 || p.splits != 1)
        return cudaErrorInvalidValue;
      if (p.epi == kEpiDGelu && p.M1 > 0 && !p.ep1.aux) return cudaErrorInvalidValue;
      if (p.epi == kEpiDGelu) {
        if (p.a_mn || !p.ep.aux) return cudaErrorInvalidValue;
        return run_gemm_pair<KIND, 256, kEpiDGelu, 2>(p, status, stream);
      }
      if (p.a_mn && p.b_mn) return run_gemm_pair<KIND, 256, kEpiBias, 3>(p, status, stream);
      if (p.b_mn) return run_gemm_pair<KIND, 256, kEpiBias, 2>(p, status, stream);
      return run_gemm_pair<KIND, 256, kEpiBias, 1>(p, status, stream);
    }
    return cudaErrorInvalidValue;
  }
  if constexpr (KIND == kKindF16) {
    if (use_pair(p)) {
      switch (p.epi) {
        case kEpiQkv: return run_gemm_pair<KIND, 256, kEpiQkv>(p, status, stream);
        case kEpiGateResid: return run_gemm_pair<KIND, 256, kEpiGateResid>(p, status, stream);
        case kEpiGelu: return run_gemm_pair<KIND, 256, kEpiGelu>(p, status, stream);
        case kEpiBias: return run_gemm_pair<KIND, 256, kEpiBias>(p, status, stream);
        default: break;
      }
    }
  }
#define MMDIT_GEMM_EPI(BN)                                                          \
  switch (p.epi) {                                                                  \
    case kEpiBias: return run_gemm<KIND, BN, kEpiBias>(p, status, stream);          \
    case kEpiGelu: return run_gemm<KIND, BN, kEpiGelu>(p, status, stream);          \
    case kEpiGateResid: return run_gemm<KIND, BN, kEpiGateResid>(p, status, stream); \
    case kEpiUnpatchify: return run_gemm<KIND, BN, kEpiUnpatchify>(p, status, stream); \
    case kEpiPartial: return run_gemm<KIND, BN, kEpiPartial>(p, status, stream);       \
    default: return cudaErrorInvalidValue;                                          \
  }
  if (p.epi == kEpiQkv) {
    if (p.N % 256 == 0 && p.ep.hidden % 256 == 0) return run_gemm<KIND, 256, kEpiQkv>(p, status, stream);
    return run_gemm<KIND, 128, kEpiQkv>(p, status, stream);
  }
  if (p.N % 256 == 0) { MMDIT_GEMM_EPI(256) }
  if (p.N % 128 == 0) { MMDIT_GEMM_EPI(128) }
  if (p.N % 64 == 0) { MMDIT_GEMM_EPI(64) }
  MMDIT_GEMM_EPI(32)
#undef MMDIT_GEMM_EPI
}

}  // namespace mmdit
