// elementwise.cu -- the memory-bound steps of the block: 3D RoPE tables, the AdaLN modulation
// GEMV, LayerNorm + modulate, latent patchify, V transpose, and the rectified-flow noise/loss.
// All use 128-bit loads and stores along the contiguous axis.
#include <math.h>

#include <type_traits>

#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "rowwise.cuh"

namespace mmdit {
namespace {

// ----------------------------------------------------------------------------- 3D RoPE tables
struct RopeTable {
  float inv_freq[128];  // theta^(-2i/d_a) of pair j
  int axis[128];        // axis of pair j
  int pairs;
};

__global__ void rope3d_kernel(const float* __restrict__ ids, int64_t n_tok, RopeTable tab,
                              float* __restrict__ cos_out, float* __restrict__ sin_out) {
  // the per-pair table in shared memory: lanes read different pairs, which kernel-parameter
  // reads would serialise
  __shared__ float inv_freq[128];
  __shared__ int axis[128];
  for (int j = threadIdx.x; j < tab.pairs; j += blockDim.x) inv_freq[j] = tab.inv_freq[j], axis[j] = tab.axis[j];
  __syncthreads();
  pdl_wait();  // the previous kernel's results are visible from here on
  const int64_t total = n_tok * tab.pairs;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = i / tab.pairs;
    const int j = static_cast<int>(i - tok * tab.pairs);
    const double ang = static_cast<double>(ids[tok * 3 + axis[j]]) * inv_freq[j];
    float s, c;
    sincosf(static_cast<float>(ang), &s, &c);
    cos_out[i] = c;
    sin_out[i] = s;
  }
}

// ----------------------------------------------------------------------------- modulation GEMV
// m[b, r] = sum_k SiLU(vec[b, k]) w[r, k] + bias[r], one warp per weight row, batch <= 8 per
// launch.  Up to two weight sets (the image and text streams of a double block) share a launch.
// Each warp issues all of a row's 16-byte loads (NC per lane) before using any of them.
constexpr int kModMaxBatch = 8;
constexpr int kModThreads = 128;

struct ModJob {
  const void* w;
  const void* bias;
  void* out;  // [batch, rows]: fp32, or the activation type under kGemvOutAct
  int rows;
};

// Up to kModMaxJobs weight matrices that read the same input share a launch; their rows form
// one index space, job i owning rows [start[i], start[i + 1]).
constexpr int kModMaxJobs = 80;
struct ModJobs {
  ModJob j[kModMaxJobs];
  int start[kModMaxJobs + 1];
  int n;
};

template <typename T, int NC, int NB>
__global__ void __launch_bounds__(kModThreads) modulation_kernel(const void* __restrict__ vec,
                                                                 const __grid_constant__ ModJobs jobs,
                                                                 int dim, int silu, int mode,
                                                                 int vec_f32) {
  pdl_wait();  // the previous kernel's results are visible from here on
  constexpr int batch = NB;  // batch rows handled by this launch (compile time: no idle lanes)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int total = jobs.start[jobs.n];
  const int stride = gridDim.x * warps;
  auto job_of = [&](int g) {  // the job owning row g (binary search over the row starts)
    int lo = 0, hi = jobs.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g >= jobs.start[mid])
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  };
  // Rows are software-pipelined: the loads of a warp's next row are issued before its current
  // row is reduced, so every warp keeps one row (NC 16-byte loads per lane) in flight.
  auto load_row = [&](int g, int ji, Raw8<T> (&raw)[NC]) {
    const ModJob& job = jobs.j[ji];
    const T* wr = reinterpret_cast<const T*>(job.w) + static_cast<size_t>(g - jobs.start[ji]) * dim;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int k = c * 256 + lane * 8;
      if (k < dim) raw[c].load(wr + k);
    }
  };
  // the first row's weights are requested before the block prepares SiLU(vec)
  Raw8<T> ra[NC], rb[NC];
  int g = blockIdx.x * warps + warp;
  int ja = 0, jb = 0;
  if (g < total) {
    ja = job_of(g);
    load_row(g, ja, ra);
  }
  // [batch, dim] SiLU(vec) (or vec itself when silu == 0): fp32, or in bf16 mode the bf16
  // operand it is there (stored as bf16, so each 16-byte weight load pairs with one 16-byte
  // shared-memory load)
  extern __shared__ float svec[];
  __nv_bfloat16* svec_bf = reinterpret_cast<__nv_bfloat16*>(svec);
  for (int i = threadIdx.x; i < batch * dim; i += blockDim.x) {
    // vec is of the weights' type, or fp32 (an fp32 hidden layer feeding a bf16 linear)
    const float v = vec_f32 ? static_cast<const float*>(vec)[i] : to_f32(static_cast<const T*>(vec)[i]);
    const float sv = silu ? v / (1.f + expf(-v)) : v;
    if constexpr (sizeof(T) == 2)
      svec_bf[i] = __float2bfloat16_rn(sv);
    else
      svec[i] = sv;
  }
  __syncthreads();
  auto reduce_row = [&](int g, int ji, const Raw8<T> (&raw)[NC]) {
    const ModJob& job = jobs.j[ji];
    const int r = g - jobs.start[ji];
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int k = c * 256 + lane * 8;
      if (k < dim) {
        float wv[8];
        raw[c].to_f32(wv);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float sv[8];
          if constexpr (sizeof(T) == 2) {
            const uint4 u = *reinterpret_cast<const uint4*>(svec_bf + b * dim + k);
            sv[0] = bf16_lo(u.x), sv[1] = bf16_hi(u.x), sv[2] = bf16_lo(u.y), sv[3] = bf16_hi(u.y);
            sv[4] = bf16_lo(u.z), sv[5] = bf16_hi(u.z), sv[6] = bf16_lo(u.w), sv[7] = bf16_hi(u.w);
          } else {
            const float4 s0 = *reinterpret_cast<const float4*>(svec + b * dim + k);
            const float4 s1 = *reinterpret_cast<const float4*>(svec + b * dim + k + 4);
            sv[0] = s0.x, sv[1] = s0.y, sv[2] = s0.z, sv[3] = s0.w;
            sv[4] = s1.x, sv[5] = s1.y, sv[6] = s1.z, sv[7] = s1.w;
          }
          acc[b] += wv[0] * sv[0] + wv[1] * sv[1] + wv[2] * sv[2] + wv[3] * sv[3] + wv[4] * sv[4] +
                    wv[5] * sv[5] + wv[6] * sv[6] + wv[7] * sv[7];
        }
      }
    }
    const float bb = job.bias ? to_f32(reinterpret_cast<const T*>(job.bias)[r]) : 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sum = warp_sum(acc[b]) + bb;
      if (lane == 0) {
        const size_t o = static_cast<size_t>(b) * job.rows + r;
        if (mode == kGemvOutAct) {
          if constexpr (sizeof(T) == 2)
            reinterpret_cast<__nv_bfloat16*>(job.out)[o] = __float2bfloat16_rn(sum);
          else
            reinterpret_cast<float*>(job.out)[o] = sum;
        } else if (mode == kGemvOutF32Add) {
          reinterpret_cast<float*>(job.out)[o] += sum;
        } else {
          reinterpret_cast<float*>(job.out)[o] = sum;
        }
      }
    }
  };
  while (g < total) {
    const int g1 = g + stride;
    if (g1 < total) {
      jb = job_of(g1);
      load_row(g1, jb, rb);
    }
    reduce_row(g, ja, ra);
    const int g2 = g1 + stride;
    if (g2 < total) {
      ja = job_of(g2);
      load_row(g2, ja, ra);
    }
    if (g1 < total) reduce_row(g1, jb, rb);
    g = g2;
  }
}

// ----------------------------------------------------------------------------- LN + modulate
// One 128-thread block per row: each thread holds NCT chunks of 8 consecutive elements (one
// load round trip), the mean and the biased variance are exact two-pass block reductions over
// the register-resident row, then out = (x - mean) * rsqrt(var + eps) * (1 + scale[b]) + shift[b].
// Up to two row sets (the image and text streams) share a launch.
constexpr int kLnThreads = 128;
constexpr int kLnMaxChunks = 8;  // rows of up to 128 * 8 * 8 = 8192 elements

struct LnJob {
  const void* x;
  const float* shift;
  const float* scale;
  int64_t mod_bstride;
  void* out;
  int rows;
  int rpb;
  const float* q_scale;  // E4M3 output only
  float* q_amax;
};

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read by the previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];
  return t;
}

template <typename TI, typename T, int NCT>
__global__ void __launch_bounds__(kLnThreads) ln_modulate_kernel(LnJob j0, LnJob j1, int dim, float eps) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float red[kLnThreads / 32];
  const int g = blockIdx.x;
  const bool second = g >= j0.rows;
  const LnJob& job = second ? j1 : j0;
  const int r = second ? g - j0.rows : g;
  const TI* xr = static_cast<const TI*>(job.x) + static_cast<size_t>(r) * dim;
  Raw8<TI> raw[NCT];
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    const int k = (c * kLnThreads + threadIdx.x) * 8;
    if (k < dim) raw[c].load(xr + k);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    if ((c * kLnThreads + threadIdx.x) * 8 < dim) {
      float v[8];
      raw[c].to_f32(v);
#pragma unroll
      for (int e = 0; e < 8; ++e) s += v[e];
    }
  }
  const float mean = block_sum(s, red) / dim;
  float q = 0.f;
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    if ((c * kLnThreads + threadIdx.x) * 8 < dim) {
      float v[8];
      raw[c].to_f32(v);
#pragma unroll
      for (int e = 0; e < 8; ++e) q = fmaf(v[e] - mean, v[e] - mean, q);
    }
  }
  const float rstd = rsqrtf(block_sum(q, red) / dim + eps);
  const int b = r / job.rpb;
  const float* sh = job.shift + b * job.mod_bstride;
  const float* sc = job.scale + b * job.mod_bstride;
  T* orow = static_cast<T*>(job.out) + static_cast<size_t>(r) * dim;
  // E4M3 output (T = uint8_t): codes of the result times the tensor's scale, and its amax
  constexpr bool kE4m3 = std::is_same<T, uint8_t>::value;
  const float qs = kE4m3 ? __ldg(job.q_scale) : 1.f;
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    const int k = (c * kLnThreads + threadIdx.x) * 8;
    if (k < dim) {
      float v[8], a[8], m[8];
      raw[c].to_f32(v);
      load8(sh + k, a);
      load8(sc + k, m);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = fmaf((v[e] - mean) * rstd, 1.f + m[e], a[e]);
      if constexpr (kE4m3) {
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        *reinterpret_cast<uint2*>(orow + k) = e4m3x8(v, qs);
      } else {
        store8(orow + k, v);
      }
    }
  }
  if constexpr (kE4m3) {
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0 && amax > 0.f) atomic_max_nonneg(job.q_amax, amax);
  }
}

// ----------------------------------------------------------------------------- transposes
// z [B, C, HW] fp32 -> out [B, HW, C].  With z1 non-null the latents are the rectified-flow
// interpolation z = (1 - t[b]) z0 + t[b] z1 of z0 = `z` and z1, formed as they are read (the same
// arithmetic as flow_kernel, so the values are bit-equal) and, with z_t non-null, also written to
// z_t [B, C, HW] fp32.
template <typename T>
__global__ void patchify_kernel(const float* __restrict__ z, int channels, int hw, T* __restrict__ out,
                                const float* __restrict__ z1, const float* __restrict__ t,
                                float* __restrict__ z_t) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float tile[32][33];
  const int b = blockIdx.z;
  const int s0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const size_t boff = static_cast<size_t>(b) * channels * hw;
  const float* zb = z + boff;
  const float tt = z1 ? t[b] : 0.f;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, s = s0 + threadIdx.x;
    float v = 0.f;
    if (c < channels && s < hw) {
      const size_t o = static_cast<size_t>(c) * hw + s;
      v = zb[o];
      if (z1) {
        v = fmaf(tt, z1[boff + o], (1.f - tt) * v);
        if (z_t) z_t[boff + o] = v;
      }
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  T* ob = out + static_cast<size_t>(b) * hw * channels;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int s = s0 + i, c = c0 + threadIdx.x;
    if (s < hw && c < channels) {
      if constexpr (sizeof(T) == 2)
        ob[static_cast<size_t>(s) * channels + c] = __float2bfloat16_rn(tile[threadIdx.x][i]);
      else
        ob[static_cast<size_t>(s) * channels + c] = tile[threadIdx.x][i];
    }
  }
}

// v [BH, S, 128] bf16 -> vt [BH, 128, S_pad] fp16
__global__ void transpose_v_kernel(const __nv_bfloat16* __restrict__ v, int seq, int seq_pad,
                                   __half* __restrict__ vt) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ __nv_bfloat16 tile[32][34];
  const size_t bh = blockIdx.z;
  const int s0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int s = s0 + i;
    tile[i][threadIdx.x] = s < seq ? v[(bh * seq + s) * 128 + j0 + threadIdx.x] : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int s = s0 + threadIdx.x;
    if (s < seq) vt[(bh * 128 + j0 + i) * seq_pad + s] = __float2half_rn(__bfloat162float(tile[threadIdx.x][i]));
  }
}

// ----------------------------------------------------------------------------- split-K finish
// out[m, n] = sum_s partial[s][m][n] + bias[n], summed in split order (deterministic); 8
// consecutive columns per thread.  unpatchify_rows > 0 writes pred[b, n, r] (fp32) instead.
template <typename T>
__global__ void splitk_reduce_kernel(const float* __restrict__ partials, int splits, int M, int N,
                                     const T* __restrict__ bias, void* __restrict__ out,
                                     int unpatchify_rows) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int64_t total = static_cast<int64_t>(M) * N / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 8;
    const int m = static_cast<int>(e / N), n = static_cast<int>(e % N);
    float v[8];
    load8(partials + e, v);
    for (int sp = 1; sp < splits; ++sp) {
      float w[8];
      load8(partials + static_cast<size_t>(sp) * M * N + e, w);
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] += w[q];
    }
    if (bias) {
      float b[8];
      load8(bias + n, b);
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] += b[q];
    }
    if (unpatchify_rows > 0) {
      const int bb = m / unpatchify_rows, r = m % unpatchify_rows;
      float* dst = static_cast<float*>(out) + (static_cast<size_t>(bb) * N + n) * unpatchify_rows + r;
#pragma unroll
      for (int q = 0; q < 8; ++q) dst[static_cast<size_t>(q) * unpatchify_rows] = v[q];
    } else {
      store8(static_cast<T*>(out) + e, v);
    }
  }
}

// ----------------------------------------------------------------------------- output head + loss
// The output stage of the output head with the rectified-flow loss fused on: per tile of
// kHeadRows tokens x kHeadCols channels,
//   v[m, n] = sum_s partial[s][m][n] + bias[n]       (split order: deterministic)
//   pred[b, n, r] = v (unpatchified, m = b * hw + r)   (if pred is non-null)
//   acc += (v - (z1[b, n, r] - z0[b, n, r]))^2         (if z0 is non-null)
// The partials are read along n and pred, z0, z1 along r, both coalesced, through a shared-memory
// transpose.  Each block writes one partial sum of squares; the last block to finish (a ticket
// counter that it resets to 0) adds them in block order and writes loss = sum / (M * N).
constexpr int kHeadRows = 32, kHeadCols = 64, kHeadThreads = 256;

__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
  // a fixed-shape tree: lane shuffles, then warp 0 over the warps' sums (same order every call)
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float w = 0.f;
  if (threadIdx.x < 32) {
    w = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
    w = warp_sum(w);
  }
  __syncthreads();
  return w;  // valid in thread 0
}

template <typename T>
__global__ void __launch_bounds__(kHeadThreads) head_finish_kernel(
    const float* __restrict__ partials, int splits, int M, int N, const T* __restrict__ bias, int hw,
    float* __restrict__ pred, const float* __restrict__ z0, const float* __restrict__ z1,
    float* __restrict__ loss_partials, unsigned int* __restrict__ ticket, float* __restrict__ loss,
    double inv_total) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float tile[kHeadCols][kHeadRows + 1];
  __shared__ float red[kHeadThreads / 32];
  __shared__ bool last;
  const int col_tiles = (N + kHeadCols - 1) / kHeadCols;
  const int n_tiles = ((M + kHeadRows - 1) / kHeadRows) * col_tiles;
  float acc = 0.f;
  for (int tile_i = blockIdx.x; tile_i < n_tiles; tile_i += gridDim.x) {
    const int m0 = (tile_i / col_tiles) * kHeadRows, n0 = (tile_i % col_tiles) * kHeadCols;
    {
      // 8 consecutive columns of one row per thread
      const int rl = threadIdx.x / (kHeadCols / 8), cl = (threadIdx.x % (kHeadCols / 8)) * 8;
      const int m = m0 + rl, n = n0 + cl;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.f;
      if (m < M && n < N) {  // N is a multiple of 32 and n of 8: the 8 columns are all in range
        const size_t e = static_cast<size_t>(m) * N + n;
        load8(partials + e, v);
        for (int sp = 1; sp < splits; ++sp) {
          float w[8];
          load8(partials + static_cast<size_t>(sp) * M * N + e, w);
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] += w[q];
        }
        if (bias) {
          float bb[8];
          load8(bias + n, bb);
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] += bb[q];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) tile[cl + q][rl] = v[q];
    }
    __syncthreads();
    {
      // one token per lane, kHeadThreads / kHeadRows channels per pass
      const int rl = threadIdx.x % kHeadRows;
      const int m = m0 + rl;
      if (m < M) {
        const int b = m / hw, r = m % hw;
        for (int cl = threadIdx.x / kHeadRows; cl < kHeadCols; cl += kHeadThreads / kHeadRows) {
          const int n = n0 + cl;
          if (n >= N) break;
          const float v = tile[cl][rl];
          const size_t o = (static_cast<size_t>(b) * N + n) * hw + r;
          if (pred) pred[o] = v;
          if (z0) {
            const float d = v - (z1[o] - z0[o]);
            acc = fmaf(d, d, acc);
          }
        }
      }
    }
    __syncthreads();
  }
  if (!z0) return;
  const float part = block_sum_fixed(acc, red);
  if (threadIdx.x == 0) {
    loss_partials[blockIdx.x] = part;
    __threadfence();  // the partial is visible device-wide before the ticket is taken
    last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  float v = 0.f;
  for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) v += __ldcg(loss_partials + i);
  const float total = block_sum_fixed(v, red);
  if (threadIdx.x == 0) {
    *loss = static_cast<float>(static_cast<double>(total) * inv_total);
    *ticket = 0u;  // ready for the next call on this workspace
  }
}

// ----------------------------------------------------------------------------- rectified flow
constexpr int kFlowThreads = 256;
static_assert(kFlowElemsPerPartial == kFlowThreads * 8 * 4, "four rounds of 8 elements per thread");

template <typename T>
__global__ void __launch_bounds__(kFlowThreads) flow_kernel(const T* __restrict__ z0, const T* __restrict__ z1,
                                                            const float* __restrict__ t, int64_t n_per,
                                                            int64_t n_total, T* __restrict__ z_t,
                                                            const T* __restrict__ pred,
                                                            float* __restrict__ partials) {
  pdl_wait();  // the previous kernel's results are visible from here on
  float acc = 0.f;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 8; i < n_total;
       i += step) {
    float a[8], c[8];
    load8(z0 + i, a);
    load8(z1 + i, c);
    if (z_t) {
      const float tt = t[i / n_per];
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = fmaf(tt, c[e], (1.f - tt) * a[e]);
      store8(z_t + i, o);
    }
    if (pred) {
      float p[8];
      load8(pred + i, p);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = p[e] - (c[e] - a[e]);
        acc = fmaf(d, d, acc);
      }
    }
  }
  if (!partials) return;
  __shared__ float red[kFlowThreads / 32];
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < kFlowThreads / 32 ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) partials[blockIdx.x] = v;
  }
}

// Sums the partials in a fixed order and writes sum / n_total.
__global__ void __launch_bounds__(kFlowThreads) flow_finish_kernel(const float* __restrict__ partials,
                                                                   int n, double inv_total,
                                                                   float* __restrict__ loss) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float red[kFlowThreads / 32];
  float v = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) v += partials[i];
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kFlowThreads / 32 ? red[threadIdx.x] : 0.f;
    w = warp_sum(w);
    if (threadIdx.x == 0) *loss = static_cast<float>(static_cast<double>(w) * inv_total);
  }
}

// ----------------------------------------------------------------------------- sampling step
// One Euler step with classifier-free guidance, 8 elements per thread and round:
// v = vu + w (vc - vu) (v = vc without vu), out = z - dt v.  out may alias z (each element is
// read and written by the same thread).
template <typename T>
__global__ void __launch_bounds__(256) euler_cfg_kernel(const T* z, const T* __restrict__ vc,
                                                        const T* __restrict__ vu, float w, float dt,
                                                        int64_t n, T* out) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n; i += step) {
    float a[8], c[8];
    load8(z + i, a);
    load8(vc + i, c);
    if (vu) {
      float u[8];
      load8(vu + i, u);
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = fmaf(w, c[e] - u[e], u[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = fmaf(-dt, c[e], a[e]);
    store8(out + i, a);
  }
}


}  // namespace

// ----------------------------------------------------------------------------- conditioning
// Sinusoidal timestep features [B, 2 half] ("Flux architecture deep dive", §Model components ›
// 1. Input embeddings › Conditioning): cos(tau f_k) in column k, sin(tau f_k) in column
// half + k, tau = time_factor * t[b].  The frequencies come from the host in double; the angle
// and its sine and cosine are taken in double (the angle reaches 1000 rad), then rounded once.
constexpr int kTimeMaxHalf = 256;
struct TimeFreqs {
  double f[kTimeMaxHalf];
};

template <typename T>
__global__ void timestep_features_kernel(const float* __restrict__ t, int batch, int half,
                                         double time_factor, const __grid_constant__ TimeFreqs fr,
                                         T* __restrict__ out) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= batch * half) return;
  const int b = i / half, k = i - b * half;
  const double ang = time_factor * static_cast<double>(__ldg(t + b)) * fr.f[k];
  double sn, cs;
  sincos(ang, &sn, &cs);
  T* row = out + static_cast<size_t>(b) * 2 * half;
  row[k] = static_cast<T>(static_cast<float>(cs));
  row[half + k] = static_cast<T>(static_cast<float>(sn));
}

// vec[b, k] = v32[b, k] + g[b] w_g[k] + b_g[k] (the guidance term only when g is given), in
// the activation type.
template <typename T>
__global__ void vec_finish_kernel(const float* __restrict__ v32, const float* __restrict__ g,
                                  const T* __restrict__ wg, const T* __restrict__ bg, int batch,
                                  int dim, T* __restrict__ vec) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= batch * dim) return;
  float v = v32[i];
  if (g) {
    const int b = i / dim, k = i - b * dim;
    v += __ldg(g + b) * to_f32(wg[k]) + to_f32(bg[k]);
  }
  vec[i] = static_cast<T>(v);
}

// ----------------------------------------------------------------------------- linear backward
// out [C, ld_out] = in [R, C] transposed, with columns R .. ld_out - 1 of out set to zero (32 x 32
// tiles through shared memory; 32 x 8 threads).  The backward GEMMs read the transposes as
// K-major operands.
template <typename T>
__global__ void transpose_pad_kernel(const T* __restrict__ in, int R, int C, int ld_out, T* __restrict__ out) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < R && c < C) ? to_f32(in[static_cast<size_t>(r) * C + c]) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < ld_out) out[static_cast<size_t>(c) * ld_out + r] = static_cast<T>(tile[threadIdx.x][i]);
  }
}

// Column sums of in [R, C] in a fixed order: chunk y of the rows into part[y, c], then the
// chunks added in a fixed two-level order.  With C % 8 == 0 a thread sums 8 adjacent columns
// from 16-byte (bf16) or 32-byte (fp32) loads, four rows in flight; otherwise one column.
template <typename T, bool VEC>
__global__ void colsum_partial_kernel(const T* __restrict__ in, int R, int C, float* __restrict__ part) {
  pdl_wait();  // the previous kernel's results are visible from here on
  constexpr int W = VEC ? 8 : 1;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * W;
  if (c >= C) return;
  const int per = (R + gridDim.y - 1) / gridDim.y;
  const int r0 = blockIdx.y * per;
  const int r1 = r0 + per < R ? r0 + per : R;
  float acc[W];
#pragma unroll
  for (int e = 0; e < W; ++e) acc[e] = 0.f;
  if constexpr (VEC) {
    int r = r0;
    for (; r + 4 <= r1; r += 4) {
      float v[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) load8(in + static_cast<size_t>(r + u) * C + c, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += v[u][e];
    }
    for (; r < r1; ++r) {
      float v[8];
      load8(in + static_cast<size_t>(r) * C + c, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += v[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) part[static_cast<size_t>(blockIdx.y) * C + c + e] = acc[e];
  } else {
    for (int r = r0; r < r1; ++r) acc[0] += to_f32(in[static_cast<size_t>(r) * C + c]);
    part[static_cast<size_t>(blockIdx.y) * C + c] = acc[0];
  }
}

// Block (32, 32) over 32 columns: thread (x, y) adds chunks y, y + 32, ... of its column in order,
// thread row 0 then adds the 32 group sums in order.
__global__ void __launch_bounds__(1024) colsum_finish_kernel(const float* __restrict__ part, int chunks, int C,
                                                             float* __restrict__ out) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float grp[32][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  float acc = 0.f;
  if (c < C)
    for (int i = threadIdx.y; i < chunks; i += 32) acc += part[static_cast<size_t>(i) * C + c];
  grp[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y != 0 || c >= C) return;
  float t = 0.f;
#pragma unroll 8
  for (int g = 0; g < 32; ++g) t += grp[g][threadIdx.x];
  out[c] = t;
}

// ----------------------------------------------------------------------------- launchers
cudaError_t launch_rope3d(const float* ids, int batch, int seq, const int axes[3], float theta,
                          float* cos_out, float* sin_out, cudaStream_t stream) {
  RopeTable tab{};
  int j = 0;
  for (int a = 0; a < 3; ++a)
    for (int i = 0; i < axes[a] / 2; ++i, ++j) {
      tab.inv_freq[j] = static_cast<float>(pow(static_cast<double>(theta), -2.0 * i / axes[a]));
      tab.axis[j] = a;
    }
  tab.pairs = j;
  const int64_t n_tok = static_cast<int64_t>(batch) * seq;
  if (n_tok == 0 || j == 0) return cudaSuccess;
  const int grid = blocks_for(n_tok * j, 256, num_sms() * 8);
  {
    const cudaError_t e_ = launch_pdl(rope3d_kernel, dim3(grid), dim3(256), 0, stream, ids, n_tok, tab, cos_out, sin_out);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

template <typename T, int NC, int NB>
cudaError_t launch_mod(const void* vec, const ModJobs& jobs, int dim, int silu, int mode, int vec_f32,
                       size_t smem, cudaStream_t stream) {
  auto kern = modulation_kernel<T, NC, NB>;
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kModThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const int rows = jobs.start[jobs.n];
  const int grid = blocks_for(rows, kModThreads / 32, num_sms() * per_sm);
  {
    const cudaError_t e_ = launch_pdl(kern, dim3(grid), dim3(kModThreads), smem, stream,
                                      vec, jobs, dim, silu, mode, vec_f32);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

template <typename T, int NC>
cudaError_t launch_mod_nb(const void* vec, const ModJobs& jobs, int nb, int dim, int silu, int mode,
                          int vec_f32, size_t smem, cudaStream_t stream) {
  switch (nb) {
    case 1: return launch_mod<T, NC, 1>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 2: return launch_mod<T, NC, 2>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 3: return launch_mod<T, NC, 3>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 4: return launch_mod<T, NC, 4>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 5: return launch_mod<T, NC, 5>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 6: return launch_mod<T, NC, 6>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    case 7: return launch_mod<T, NC, 7>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
    default: return launch_mod<T, NC, 8>(vec, jobs, dim, silu, mode, vec_f32, smem, stream);
  }
}

cudaError_t launch_gemv(int act, const void* vec, const ModulationJob* jobs, int njobs, int batch,
                        int dim, int silu, int mode, cudaStream_t stream, int vec_f32) {
  const size_t elt = act == 1 ? 2 : 4;
  const size_t vec_elt = vec_f32 ? 4 : elt;
  const size_t out_elt = mode == kGemvOutAct ? elt : 4;
  const int chunks = (dim + 255) / 256;
  for (int j0 = 0; j0 < njobs; j0 += kModMaxJobs) {
    const int nj = njobs - j0 < kModMaxJobs ? njobs - j0 : kModMaxJobs;
    for (int b0 = 0; b0 < batch; b0 += kModMaxBatch) {
      const int nb = batch - b0 < kModMaxBatch ? batch - b0 : kModMaxBatch;
      const size_t smem = static_cast<size_t>(nb) * dim * sizeof(float);
      ModJobs mj{};
      int rows = 0;
      mj.n = 0;
      for (int i = 0; i < nj; ++i) {
        const ModulationJob& jb = jobs[j0 + i];
        if (jb.rows <= 0) continue;
        mj.j[mj.n] = {jb.w, jb.bias, static_cast<uint8_t*>(jb.out) + static_cast<size_t>(b0) * jb.rows * out_elt,
                      jb.rows};
        mj.start[mj.n] = rows;
        rows += jb.rows;
        ++mj.n;
      }
      mj.start[mj.n] = rows;
      if (rows == 0) continue;
      const void* vb = static_cast<const uint8_t*>(vec) + static_cast<size_t>(b0) * dim * vec_elt;
      cudaError_t e;
      if (act == 1) {
        if (chunks <= 4) e = launch_mod_nb<__nv_bfloat16, 4>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
        else if (chunks <= 8) e = launch_mod_nb<__nv_bfloat16, 8>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
        else if (chunks <= 12) e = launch_mod_nb<__nv_bfloat16, 12>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
        else e = launch_mod_nb<__nv_bfloat16, 24>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
      } else {
        if (chunks <= 4) e = launch_mod_nb<float, 4>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
        else if (chunks <= 8) e = launch_mod_nb<float, 8>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
        else e = launch_mod_nb<float, 16>(vb, mj, nb, dim, silu, mode, vec_f32, smem, stream);
      }
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_modulation2(int act, const void* vec, const ModulationJob* jobs, int njobs,
                               int batch, int dim, cudaStream_t stream) {
  return launch_gemv(act, vec, jobs, njobs, batch, dim, 1, kGemvOutF32, stream);
}

cudaError_t launch_modulation(int act, const void* vec, const void* w, const void* bias, int batch,
                              int rows, int dim, float* m, cudaStream_t stream) {
  ModulationJob job{w, bias, m, rows};
  return launch_modulation2(act, vec, &job, 1, batch, dim, stream);
}

cudaError_t launch_ln_modulate2(int act, int x_f32, const LnModJob* jobs, int njobs, int dim,
                                float eps, cudaStream_t stream, int out_e4m3) {
  LnJob j[2] = {{nullptr, nullptr, nullptr, 0, nullptr, 0, 1, nullptr, nullptr},
                {nullptr, nullptr, nullptr, 0, nullptr, 0, 1, nullptr, nullptr}};
  int rows = 0;
  for (int i = 0; i < njobs && i < 2; ++i) {
    j[i] = {jobs[i].x, jobs[i].shift, jobs[i].scale, jobs[i].mod_bstride, jobs[i].out, jobs[i].rows,
            jobs[i].rows_per_batch, jobs[i].q_scale, jobs[i].q_amax};
    rows += jobs[i].rows;
  }
  if (out_e4m3 && act != 1) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  const int chunks = (dim + kLnThreads * 8 - 1) / (kLnThreads * 8);
  if (chunks > kLnMaxChunks) return cudaErrorInvalidValue;
  cudaError_t launch_err = cudaSuccess;
  auto go = [&](auto nct_tag) {
    constexpr int NCT = decltype(nct_tag)::value;
    if (out_e4m3 && x_f32)
      launch_err = launch_pdl(ln_modulate_kernel<float, uint8_t, NCT>, dim3(rows), dim3(kLnThreads), 0, stream, j[0], j[1], dim, eps);
    else if (out_e4m3)
      launch_err = launch_pdl(ln_modulate_kernel<__nv_bfloat16, uint8_t, NCT>, dim3(rows), dim3(kLnThreads), 0, stream, j[0], j[1], dim, eps);
    else if (act == 1 && x_f32)
      launch_err = launch_pdl(ln_modulate_kernel<float, __nv_bfloat16, NCT>, dim3(rows), dim3(kLnThreads), 0, stream, j[0], j[1], dim, eps);
    else if (act == 1)
      launch_err = launch_pdl(ln_modulate_kernel<__nv_bfloat16, __nv_bfloat16, NCT>, dim3(rows), dim3(kLnThreads), 0, stream, j[0], j[1], dim, eps);
    else
      launch_err = launch_pdl(ln_modulate_kernel<float, float, NCT>, dim3(rows), dim3(kLnThreads), 0, stream, j[0], j[1], dim, eps);
  };
  if (chunks <= 1)
    go(std::integral_constant<int, 1>());
  else if (chunks <= 2)
    go(std::integral_constant<int, 2>());
  else if (chunks <= 3)
    go(std::integral_constant<int, 3>());
  else if (chunks <= 4)
    go(std::integral_constant<int, 4>());
  else
    go(std::integral_constant<int, kLnMaxChunks>());
  if (launch_err != cudaSuccess) return launch_err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_ln_modulate(int act, int x_f32, const void* x, const float* shift, const float* scale,
                               int64_t mod_bstride, int rows, int rows_per_batch, int dim, float eps,
                               void* out, cudaStream_t stream) {
  const LnModJob job{x, shift, scale, mod_bstride, out, rows, rows_per_batch};
  return launch_ln_modulate2(act, x_f32, &job, 1, dim, eps, stream);
}

cudaError_t launch_patchify(int act, const float* z, int batch, int channels, int hw, void* out,
                            cudaStream_t stream, const float* z1, const float* t, float* z_t) {
  const dim3 grid((hw + 31) / 32, (channels + 31) / 32, batch), block(32, 8);
  if (act == 1) {
    const cudaError_t e_ = launch_pdl(patchify_kernel<__nv_bfloat16>, dim3(grid), dim3(block), 0, stream, z, channels, hw,
                                      static_cast<__nv_bfloat16*>(out), z1, t, z_t);
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(patchify_kernel<float>, dim3(grid), dim3(block), 0, stream, z, channels, hw,
                                      static_cast<float*>(out), z1, t, z_t);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_transpose_v(const __nv_bfloat16* v, int bh, int seq, int seq_pad, __half* vt,
                               cudaStream_t stream) {
  const dim3 grid((seq + 31) / 32, 4, bh), block(32, 8);
  {
    const cudaError_t e_ = launch_pdl(transpose_v_kernel, dim3(grid), dim3(block), 0, stream, v, seq, seq_pad, vt);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(int act, const float* partials, int splits, int M, int N,
                                 const void* bias, void* out, int unpatchify_rows,
                                 cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N / 8;
  if (total == 0) return cudaSuccess;
  const int grid = blocks_for(total, 256, num_sms() * 8);
  if (act == 1) {
    const cudaError_t e_ = launch_pdl(splitk_reduce_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream,
        partials, splits, M, N, static_cast<const __nv_bfloat16*>(bias), out, unpatchify_rows);
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(splitk_reduce_kernel<float>, dim3(grid), dim3(256), 0, stream, partials, splits, M, N,
                                                          static_cast<const float*>(bias), out,
                                                          unpatchify_rows);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

int head_finish_blocks(int M, int N) {
  const int64_t tiles = static_cast<int64_t>((M + kHeadRows - 1) / kHeadRows) * ((N + kHeadCols - 1) / kHeadCols);
  return blocks_for(tiles, 1, num_sms() * 4);
}

cudaError_t launch_head_finish(int act, const float* partials, int splits, int M, int N, const void* bias,
                               int hw, float* pred, const float* z0, const float* z1,
                               float* loss_partials, unsigned int* ticket, float* loss,
                               cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int grid = head_finish_blocks(M, N);
  const double inv_total = 1.0 / (static_cast<double>(M) * N);
  cudaError_t e;
  if (act == 1)
    e = launch_pdl(head_finish_kernel<__nv_bfloat16>, dim3(grid), dim3(kHeadThreads), 0, stream, partials,
                   splits, M, N, static_cast<const __nv_bfloat16*>(bias), hw, pred, z0, z1, loss_partials,
                   ticket, loss, inv_total);
  else
    e = launch_pdl(head_finish_kernel<float>, dim3(grid), dim3(kHeadThreads), 0, stream, partials, splits, M,
                   N, static_cast<const float*>(bias), hw, pred, z0, z1, loss_partials, ticket, loss,
                   inv_total);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

int flow_partial_blocks(int64_t n_total) {
  return blocks_for(n_total, static_cast<int>(kFlowElemsPerPartial), kFlowMaxPartials);
}

cudaError_t launch_flow_match(int dtype, const void* z0, const void* z1, const float* t, int batch,
                              int64_t n_per_sample, void* z_t, const void* pred, float* loss,
                              float* partials, int n_partials, cudaStream_t stream) {
  const int64_t n_total = static_cast<int64_t>(batch) * n_per_sample;
  if (n_total == 0) return cudaSuccess;
  const bool want_loss = pred != nullptr && loss != nullptr;
  const int grid = n_partials;
  if (dtype == 1) {
    const cudaError_t e_ = launch_pdl(flow_kernel<__nv_bfloat16>, dim3(grid), dim3(kFlowThreads), 0, stream,
        static_cast<const __nv_bfloat16*>(z0), static_cast<const __nv_bfloat16*>(z1), t,
        n_per_sample, n_total, static_cast<__nv_bfloat16*>(z_t),
        want_loss ? static_cast<const __nv_bfloat16*>(pred) : nullptr, want_loss ? partials : nullptr);
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(flow_kernel<float>, dim3(grid), dim3(kFlowThreads), 0, stream,
        static_cast<const float*>(z0), static_cast<const float*>(z1), t, n_per_sample, n_total,
        static_cast<float*>(z_t), want_loss ? static_cast<const float*>(pred) : nullptr,
        want_loss ? partials : nullptr);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !want_loss) return e;
  {
    const cudaError_t e_ = launch_pdl(flow_finish_kernel, dim3(1), dim3(kFlowThreads), 0, stream, partials, grid, 1.0 / static_cast<double>(n_total),
                                                     loss);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_euler_cfg(int dtype, int64_t n, const void* z, const void* v_cond,
                             const void* v_uncond, float guidance, float dt, void* z_out,
                             cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int grid = blocks_for((n + 7) / 8, 256, num_sms() * 8);
  if (dtype == 1) {
    const cudaError_t e_ = launch_pdl(euler_cfg_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream,
                                      static_cast<const __nv_bfloat16*>(z), static_cast<const __nv_bfloat16*>(v_cond),
                                      static_cast<const __nv_bfloat16*>(v_uncond), guidance, dt, n,
                                      static_cast<__nv_bfloat16*>(z_out));
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(euler_cfg_kernel<float>, dim3(grid), dim3(256), 0, stream,
                                      static_cast<const float*>(z), static_cast<const float*>(v_cond),
                                      static_cast<const float*>(v_uncond), guidance, dt, n,
                                      static_cast<float*>(z_out));
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_timestep_features(int act, const float* t, int batch, int dim,
                                     double time_factor, double max_period, void* out,
                                     cudaStream_t stream) {
  const int half = dim / 2;
  if (dim % 2 != 0 || half < 1 || half > kTimeMaxHalf) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  TimeFreqs fr{};
  for (int k = 0; k < half; ++k) fr.f[k] = std::pow(max_period, -static_cast<double>(k) / half);
  const int grid = (batch * half + 255) / 256;
  if (act == 1) {
    const cudaError_t e_ = launch_pdl(timestep_features_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0,
                                      stream, t, batch, half, time_factor, fr,
                                      static_cast<__nv_bfloat16*>(out));
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(timestep_features_kernel<float>, dim3(grid), dim3(256), 0, stream,
                                      t, batch, half, time_factor, fr, static_cast<float*>(out));
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_vec_finish(int act, const float* v32, const float* g, const void* wg,
                              const void* bg, int batch, int dim, void* vec, cudaStream_t stream) {
  if (batch <= 0 || dim <= 0) return cudaSuccess;
  const int grid = (batch * dim + 255) / 256;
  if (act == 1) {
    const cudaError_t e_ = launch_pdl(vec_finish_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, v32,
                                      g, static_cast<const __nv_bfloat16*>(wg),
                                      static_cast<const __nv_bfloat16*>(bg), batch, dim,
                                      static_cast<__nv_bfloat16*>(vec));
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(vec_finish_kernel<float>, dim3(grid), dim3(256), 0, stream, v32, g,
                                      static_cast<const float*>(wg), static_cast<const float*>(bg), batch,
                                      dim, static_cast<float*>(vec));
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_transpose_pad(int act, const void* in, int R, int C, int ld_out, void* out,
                                 cudaStream_t stream) {
  if (R <= 0 && ld_out <= 0) return cudaSuccess;
  if (C <= 0 || ld_out < R) return cudaErrorInvalidValue;
  const dim3 grid((C + 31) / 32, (ld_out + 31) / 32), block(32, 8);
  if (act == 1) {
    const cudaError_t e_ = launch_pdl(transpose_pad_kernel<__nv_bfloat16>, grid, block, 0, stream,
                                      static_cast<const __nv_bfloat16*>(in), R, C, ld_out,
                                      static_cast<__nv_bfloat16*>(out));
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(transpose_pad_kernel<float>, grid, block, 0, stream,
                                      static_cast<const float*>(in), R, C, ld_out, static_cast<float*>(out));
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_colsum(int act, const void* in, int R, int C, float* part, int chunks, float* out,
                          cudaStream_t stream) {
  if (C <= 0) return cudaSuccess;
  if (chunks < 1) return cudaErrorInvalidValue;
  const size_t elt = act == 1 ? 2 : 4;
  const bool vec = C % 8 == 0 && reinterpret_cast<uintptr_t>(in) % (8 * elt) == 0;
  const dim3 grid(vec ? (C / 8 + 127) / 128 : (C + 127) / 128, chunks);
  cudaError_t e_;
  if (act == 1)
    e_ = vec ? launch_pdl(colsum_partial_kernel<__nv_bfloat16, true>, grid, dim3(128), 0, stream,
                          static_cast<const __nv_bfloat16*>(in), R, C, part)
             : launch_pdl(colsum_partial_kernel<__nv_bfloat16, false>, grid, dim3(128), 0, stream,
                          static_cast<const __nv_bfloat16*>(in), R, C, part);
  else
    e_ = vec ? launch_pdl(colsum_partial_kernel<float, true>, grid, dim3(128), 0, stream,
                          static_cast<const float*>(in), R, C, part)
             : launch_pdl(colsum_partial_kernel<float, false>, grid, dim3(128), 0, stream,
                          static_cast<const float*>(in), R, C, part);
  if (e_ != cudaSuccess) return e_;
  count_launch();
  e_ = launch_pdl(colsum_finish_kernel, dim3((C + 31) / 32), dim3(32, 32), 0, stream, part, chunks, C, out);
  if (e_ != cudaSuccess) return e_;
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
