// backward.cu -- the row-wise (memory-bound) steps of the block backward: the gradients of
// LayerNorm-modulate, the gated residuals, the GELU, QK-RMSNorm + RoPE and the AdaLN modulation,
// the attention backward's pre-pass (D = rowsum(dO * O), dO head-major, the gradient scale), and
// the fixed-order column sums that finish every reduction over rows.
//
// The pages train these blocks ("Flux architecture deep dive", §Training data flow; "Flux model
// API reference", §Training workflow example) and print no backward: each kernel is the chain
// rule of the forward step it names.  Every reduction over rows is written as per-block partial
// sums and finished in a fixed order (deterministic, no atomics), except amax(dO), whose atomic
// maximum is exact and order-independent.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "rowwise.cuh"

namespace mmdit {
namespace {

constexpr int kRowThreads = 128;   // LayerNorm backward: one block per row group, 8 elements per thread
constexpr int kRowMaxChunks = 8;   // rows of up to 128 * 8 * 8 = 8192 elements
constexpr int kBwdRowsPerBlock = 32;   // rows of one batch element per block (column sums)
constexpr int kLnBwdRowsPerBlock = 8;  // LayerNorm backward: rows per block (more blocks in flight)
constexpr int kColsumGroups = 32;      // column-sum finish: partial rows summed by 32 thread rows

// The attention backward's gradient scale from amax(dO): 2^(8 - ceil(log2 amax)), 1 for 0 (headroom for dS = p (dP - D) / sqrt(d) in fp16).
__device__ __forceinline__ float grad_scale_of(const float* amax) {
  if (!amax) return 1.f;
  const float a = *amax;
  if (!(a > 0.f) || !isfinite(a)) return 1.f;
  int e;
  frexpf(a, &e);              // a = f 2^e, f in [0.5, 1): ceil(log2 a) <= e
  return ldexpf(1.f, 8 - e);
}

// ----------------------------------------------------------------------------- LayerNorm-modulate
// h = LN(x) (1 + scale) + shift.  Given dh: g = dh (1 + scale),
//   dx += r (g - mean(g) - xhat mean(g xhat)),  dscale = sum_rows dh xhat,  dshift = sum_rows dh.
struct LnBwdJob {
  const void* x;        // [rows, dim], TX
  const void* dh;       // [rows, dim], TG
  const float* scale;   // batch b at scale + b * mod_bstride
  int64_t mod_bstride;
  float* dx;            // [rows, dim] fp32, accumulated into
  float* part;          // [gridDim.x, 2, dim]: dscale, dshift sums of the block's rows
  int rows;
  int rpb;              // rows per batch element
};

__device__ __forceinline__ void block_sum2(float& a, float& b, float* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read by the previous reduction
  if (lane == 0) red[warp] = a, red[kRowThreads / 32 + warp] = b;
  __syncthreads();
  float s = 0.f, t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) s += red[w], t += red[kRowThreads / 32 + w];
  a = s;
  b = t;
}

template <typename TX, typename TG, int NCT>
__global__ void __launch_bounds__(kRowThreads) ln_modulate_bwd_kernel(LnBwdJob job, int dim, float eps) {
  pdl_wait();
  __shared__ float red[2 * (kRowThreads / 32)];
  const int bpb = (job.rpb + kLnBwdRowsPerBlock - 1) / kLnBwdRowsPerBlock;
  const int b = blockIdx.x / bpb;
  const int r0 = b * job.rpb + (blockIdx.x - b * bpb) * kLnBwdRowsPerBlock;
  const int r_end = (b + 1) * job.rpb;
  const int r1 = r0 + kLnBwdRowsPerBlock < r_end ? r0 + kLnBwdRowsPerBlock : r_end;
  const float* sc = job.scale + b * job.mod_bstride;
  float dsc[NCT][8], dsh[NCT][8], opc[NCT][8];
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    const int k = (c * kRowThreads + threadIdx.x) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) dsc[c][e] = 0.f, dsh[c][e] = 0.f, opc[c][e] = 1.f;
    if (k < dim) {
      float m[8];
      load8(sc + k, m);
#pragma unroll
      for (int e = 0; e < 8; ++e) opc[c][e] = 1.f + m[e];
    }
  }
  // x and dh of the next row are loaded while this row is reduced
  Raw8<TX> rx[NCT];
  Raw8<TG> rg[NCT];
  auto load_row = [&](int r, Raw8<TX>(&ox)[NCT], Raw8<TG>(&og)[NCT]) {
    const TX* xr = static_cast<const TX*>(job.x) + static_cast<size_t>(r) * dim;
    const TG* gr = static_cast<const TG*>(job.dh) + static_cast<size_t>(r) * dim;
#pragma unroll
    for (int c = 0; c < NCT; ++c) {
      const int k = (c * kRowThreads + threadIdx.x) * 8;
      if (k < dim) ox[c].load(xr + k), og[c].load(gr + k);
    }
  };
  // (rows of more than four chunks per thread load in place: a second set of registers would spill)
  constexpr bool kPrefetch = NCT <= 4;
  if (kPrefetch && r0 < r1) load_row(r0, rx, rg);
  for (int r = r0; r < r1; ++r) {
    Raw8<TX> nx[kPrefetch ? NCT : 1];
    Raw8<TG> ng[kPrefetch ? NCT : 1];
    if constexpr (kPrefetch) {
      if (r + 1 < r1) load_row(r + 1, nx, ng);
    } else {
      load_row(r, rx, rg);
    }
    // mean and variance of x, two passes over the registers as the forward does
    float s = 0.f, unused = 0.f;
#pragma unroll
    for (int c = 0; c < NCT; ++c)
      if ((c * kRowThreads + threadIdx.x) * 8 < dim) {
        float v[8];
        rx[c].to_f32(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += v[e];
      }
    block_sum2(s, unused, red);
    const float mean = s / dim;
    float q = 0.f;
    unused = 0.f;
#pragma unroll
    for (int c = 0; c < NCT; ++c)
      if ((c * kRowThreads + threadIdx.x) * 8 < dim) {
        float v[8];
        rx[c].to_f32(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) q = fmaf(v[e] - mean, v[e] - mean, q);
      }
    block_sum2(q, unused, red);
    const float rstd = rsqrtf(q / dim + eps);
    // g = dh (1 + scale); the two means the input gradient needs
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int c = 0; c < NCT; ++c)
      if ((c * kRowThreads + threadIdx.x) * 8 < dim) {
        float v[8], d[8];
        rx[c].to_f32(v);
        rg[c].to_f32(d);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = (v[e] - mean) * rstd;
          const float g = d[e] * opc[c][e];
          dsc[c][e] = fmaf(d[e], xh, dsc[c][e]);
          dsh[c][e] += d[e];
          sg += g;
          sgx = fmaf(g, xh, sgx);
        }
      }
    block_sum2(sg, sgx, red);
    const float mg = sg / dim, mgx = sgx / dim;
    float* dxr = job.dx + static_cast<size_t>(r) * dim;
#pragma unroll
    for (int c = 0; c < NCT; ++c) {
      const int k = (c * kRowThreads + threadIdx.x) * 8;
      if (k < dim) {
        float v[8], d[8], acc[8];
        rx[c].to_f32(v);
        rg[c].to_f32(d);
        load8(dxr + k, acc);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = (v[e] - mean) * rstd;
          acc[e] = fmaf(rstd, d[e] * opc[c][e] - mg - xh * mgx, acc[e]);
        }
        store8(dxr + k, acc);
      }
    }
    if constexpr (kPrefetch) {
#pragma unroll
      for (int c = 0; c < NCT; ++c) rx[c] = nx[c], rg[c] = ng[c];
    }
  }
  float* p = job.part + static_cast<size_t>(blockIdx.x) * 2 * dim;
#pragma unroll
  for (int c = 0; c < NCT; ++c) {
    const int k = (c * kRowThreads + threadIdx.x) * 8;
    if (k < dim) store8(p + k, dsc[c]), store8(p + dim + k, dsh[c]);
  }
}

// Fixed-order sums of per-block partials [B * bpb, nvec, dim] over each batch element's blocks:
// out_v[b * out_bstride + k] (=, or += when accumulate) sum_i part[b * bpb + i][v][k].
struct ColsumOut {
  float* out[4];
  int64_t out_bstride;
  int nvec;
  int accumulate;
};

// Block (32, kColsumGroups): thread (x, y) sums partials y, y + 32, ... of column 32 blockIdx.x + x
// in order; thread row 0 then adds the 32 group sums in order (a fixed-order two-level sum).
__global__ void __launch_bounds__(32 * kColsumGroups) batch_colsum_finish_kernel(const float* __restrict__ part,
                                                                                 int bpb, int dim, ColsumOut o) {
  pdl_wait();
  __shared__ float grp[kColsumGroups][33];
  const int k = blockIdx.x * 32 + threadIdx.x;
  const int b = blockIdx.y;
  for (int v = 0; v < o.nvec; ++v) {
    if (!o.out[v]) continue;  // a gradient the caller did not ask for
    float acc = 0.f;
    if (k < dim) {
      const float* col = part + static_cast<size_t>(b) * bpb * o.nvec * dim + static_cast<size_t>(v) * dim + k;
#pragma unroll 4
      for (int i = threadIdx.y; i < bpb; i += kColsumGroups) acc += col[static_cast<size_t>(i) * o.nvec * dim];
    }
    grp[threadIdx.y][threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.y == 0 && k < dim) {
      float t = 0.f;
#pragma unroll 8
      for (int g = 0; g < kColsumGroups; ++g) t += grp[g][threadIdx.x];
      float* dst = o.out[v] + b * o.out_bstride + k;
      *dst = o.accumulate ? *dst + t : t;
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------- gated residual
// y = x + gate f.  Given dy (fp32, the running gradient of the residual stream, which is also
// dx): df = dy gate (type TO, the operand of the linear backward), dgate = sum_rows dy f.
// Grid: x = column groups of 8 * blockDim.x, y = B * bpb row blocks.
template <typename TF, typename TO>
__global__ void gated_residual_bwd_kernel(const float* __restrict__ dy, const TF* __restrict__ f,
                                          const float* __restrict__ gate, int64_t gate_bstride,
                                          int rpb, int dim, TO* __restrict__ df, float* __restrict__ part) {
  pdl_wait();
  const int k = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  const int bpb = (rpb + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock;
  const int b = blockIdx.y / bpb;
  const int r0 = b * rpb + (blockIdx.y - b * bpb) * kBwdRowsPerBlock;
  const int r_end = (b + 1) * rpb;
  const int r1 = r0 + kBwdRowsPerBlock < r_end ? r0 + kBwdRowsPerBlock : r_end;
  if (k >= dim) return;
  float gt[8], acc[8];
  load8(gate + b * gate_bstride + k, gt);
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int r = r0; r < r1; ++r) {
    float d[8], fv[8], o[8];
    load8(dy + static_cast<size_t>(r) * dim + k, d);
    load8(f + static_cast<size_t>(r) * dim + k, fv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[e] = fmaf(d[e], fv[e], acc[e]);
      o[e] = d[e] * gt[e];
    }
    store8(df + static_cast<size_t>(r) * dim + k, o);
  }
  store8(part + static_cast<size_t>(blockIdx.y) * dim + k, acc);
}

// ----------------------------------------------------------------------------- GELU
// du_pre = du * GELU'(u_pre): Phi(u) + u phi(u) (erf form) or the tanh form's derivative.
template <typename T>
__global__ void gelu_bwd_kernel(const T* __restrict__ du, const T* __restrict__ u_pre, int64_t n,
                                int tanh_form, T* __restrict__ out) {
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
    float d[8], u[8], o[8];
    load8(du + i, d);
    load8(u_pre + i, u);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = d[e] * gelu_grad_f(u[e], tanh_form);
    store8(out + i, o);
  }
}

// ----------------------------------------------------------------------------- QK-RMSNorm + RoPE
// For one stream: q_pre, k_pre are columns [0, D) and [D, 2D) of qkv_pre [B, S_s, 3D] (the QKV
// GEMM's output with bias, before the norm).  The attention backward gives dQ, dK, dV
// [B, H, S_joint, 128] (TG) at joint rows seq_offset + s.  Per (b, s, h), one warp, lane l
// holding elements 4l .. 4l+3 of the head:
//   dyn  = RoPE^T(dQ)                        (rotation by the negative angle)
//   xn   = q_pre r,  r = (mean(q_pre^2) + eps)^(-1/2)
//   dg  += dyn xn,   dq_pre = r (g dyn - xn mean(g dyn xn))
// and the same for k; dv is copied.  Results go to dqkv [B, S_s, 3D] (TO) at q | k | v columns.
// part [gridDim.x, 2, 128]: the block's dg_q, dg_k sums (warps in fixed order).

template <typename TA, typename TG>
__device__ __forceinline__ void qk_one(const TA* pre, const TG* dsrc, const float* c, const float* s, float g[4],
                                       int lane, int interleaved, float eps, float inv_gs, float out[4],
                                       float dg[4]) {
  float x[4], d[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = to_f32(pre[4 * lane + e]), d[e] = to_f32(dsrc[4 * lane + e]) * inv_gs;
  // inverse rotation of the gradient
  float dn[4];
  if (interleaved) {
    // pairs (4l, 4l+1) and (4l+2, 4l+3): angle indices 2l and 2l+1
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float cc = c[2 * lane + p], ss = s[2 * lane + p];
      const float a = d[2 * p], bb = d[2 * p + 1];
      dn[2 * p] = a * cc + bb * ss;
      dn[2 * p + 1] = -a * ss + bb * cc;
    }
  } else {
    // pairs (j, j + 64): lanes 0..15 hold the first halves, lanes 16..31 the partners
    float pd[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pd[e] = __shfl_xor_sync(0xffffffffu, d[e], 16);
    const int j0 = 4 * (lane & 15);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float cc = c[j0 + e], ss = s[j0 + e];
      if (lane < 16)
        dn[e] = d[e] * cc + pd[e] * ss;    // first of the pair: a' = a c - b s  ->  da = da' c + db' s
      else
        dn[e] = -pd[e] * ss + d[e] * cc;   // second: b' = a s + b c  ->  db = -da' s + db' c
    }
  }
  float ss2 = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) ss2 = fmaf(x[e], x[e], ss2);
  ss2 = warp_sum(ss2);
  const float r = rsqrtf(ss2 / 128.f + eps);
  float t = 0.f;
  float xn[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    xn[e] = x[e] * r;
    dg[e] = fmaf(dn[e], xn[e], dg[e]);
    t = fmaf(g[e] * dn[e], xn[e], t);
  }
  t = warp_sum(t) / 128.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) out[e] = r * (g[e] * dn[e] - xn[e] * t);
}

template <typename TA, typename TG, typename TO>
__global__ void __launch_bounds__(256) qk_norm_rope_bwd_kernel(QkBwdArgs a) {
  pdl_wait();
  __shared__ float red[8][2][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = a.hidden;
  float gq[4], gk[4], dgq[4] = {0.f, 0.f, 0.f, 0.f}, dgk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    gq[e] = to_f32(static_cast<const TA*>(a.g_q)[4 * lane + e]),
    gk[e] = to_f32(static_cast<const TA*>(a.g_k)[4 * lane + e]);
  const float inv_gs = 1.f / grad_scale_of(a.amax);   // a power of two: exact
  const int64_t total = static_cast<int64_t>(a.batch) * a.seq_s * a.heads;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + warp; w < total; w += static_cast<int64_t>(gridDim.x) * 8) {
    const int h = static_cast<int>(w % a.heads);
    const int64_t bs = w / a.heads;           // b * seq_s + s
    const int b = static_cast<int>(bs / a.seq_s);
    const int s = static_cast<int>(bs - static_cast<int64_t>(b) * a.seq_s);
    const int sj = a.seq_offset + s;
    const TA* pre = static_cast<const TA*>(a.qkv_pre) + bs * 3 * D + h * 128;
    const size_t hrow = ((static_cast<size_t>(b) * a.heads + h) * a.seq_joint + sj) * 128;
    const float* c = a.cos + (static_cast<size_t>(b) * a.seq_joint + sj) * 64;
    const float* sn = a.sin + (static_cast<size_t>(b) * a.seq_joint + sj) * 64;
    TO* o = static_cast<TO*>(a.dqkv) + bs * 3 * D + h * 128;
    float out[4];
    qk_one(pre, static_cast<const TG*>(a.dq) + hrow, c, sn, gq, lane, a.interleaved, a.eps, inv_gs, out, dgq);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[4 * lane + e] = static_cast<TO>(out[e]);
    qk_one(pre + D, static_cast<const TG*>(a.dk) + hrow, c, sn, gk, lane, a.interleaved, a.eps, inv_gs, out, dgk);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[D + 4 * lane + e] = static_cast<TO>(out[e]);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[2 * D + 4 * lane + e] = static_cast<TO>(to_f32(static_cast<const TG*>(a.dv)[hrow + 4 * lane + e]) * inv_gs);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) red[warp][0][4 * lane + e] = dgq[e], red[warp][1][4 * lane + e] = dgk[e];
  __syncthreads();
  const int v = threadIdx.x >> 7, j = threadIdx.x & 127;   // 256 threads: (q | k) x 128
  float acc = 0.f;
#pragma unroll
  for (int w8 = 0; w8 < 8; ++w8) acc += red[w8][v][j];
  a.part[(static_cast<size_t>(blockIdx.x) * 2 + v) * 128 + j] = acc;
}

// ----------------------------------------------------------------------------- attention pre-pass
// The gradient scale: dO is multiplied by g = 2^(8 - ceil(log2 amax(dO))) (1 for amax 0) so that
// the fp16 operands of the attention backward hold it in their normal range; the consumers of
// dQ, dK, dV divide by g.  amax is raised with atomic_max_nonneg (exact, order-independent).
__global__ void amax_kernel_bf16(const __nv_bfloat16* __restrict__ x, int64_t n, float* __restrict__ amax) {
  pdl_wait();
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
    float v[8];
    load8(x + i, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0 && m > 0.f) atomic_max_nonneg(amax, m);
}


// D[b, h, s] = sum_j dO[b, s, h*128 + j] O[b, s, h*128 + j] g, and g dO copied head-major to
// dOh [B, H, S_joint, 128] bf16 for the attention backward.  The stream's rows are joint rows
// seq_offset .. seq_offset + seq_s - 1.  One warp per (b, s, h).  D is stored with row stride
// seq_pad ([B, H, seq_pad]).
template <typename T>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                           int batch, int seq_s, int seq_joint, int seq_pad,
                                                           int seq_offset, int heads, const float* __restrict__ amax,
                                                           float* __restrict__ Dsum, __half* __restrict__ doh) {
  pdl_wait();
  const float g = grad_scale_of(amax);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t total = static_cast<int64_t>(batch) * seq_s * heads;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + warp; w < total; w += static_cast<int64_t>(gridDim.x) * 8) {
    const int h = static_cast<int>(w % heads);
    const int64_t bs = w / heads;
    const int b = static_cast<int>(bs / seq_s);
    const int s = static_cast<int>(bs - static_cast<int64_t>(b) * seq_s);
    const size_t src = static_cast<size_t>(bs) * heads * 128 + h * 128 + 4 * lane;
    float acc = 0.f;
    float d4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      d4[e] = to_f32(dout[src + e]) * g;   // a power of two: exact
      acc = fmaf(d4[e], to_f32(o[src + e]), acc);
    }
    acc = warp_sum(acc);
    const size_t bh = static_cast<size_t>(b) * heads + h;
    if (lane == 0) Dsum[bh * seq_pad + seq_offset + s] = acc;
    uint2 pk;  // the scaled dO in fp16 (the attention backward's operand)
    pk.x = pack_half2(d4[0], d4[1]);
    pk.y = pack_half2(d4[2], d4[3]);
    *reinterpret_cast<uint2*>(doh + (bh * seq_joint + seq_offset + s) * 128 + 4 * lane) = pk;
  }
}

// V [BH, S, 128] fp16 from V^T [BH, 128, S_pad] fp16.
__global__ void untranspose_vt_kernel(const __half* __restrict__ vt, int seq, int seq_pad, __half* __restrict__ v) {
  pdl_wait();
  __shared__ float tile[32][33];
  const size_t bh = blockIdx.z;
  const int s0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int s = s0 + threadIdx.x;
    tile[i][threadIdx.x] = s < seq ? __half2float(vt[(bh * 128 + j0 + i) * seq_pad + s]) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int s = s0 + i;
    if (s < seq) v[(bh * seq + s) * 128 + j0 + threadIdx.x] = __float2half_rn(tile[threadIdx.x][i]);
  }
}

// q16 = q, k16 = k (bf16 -> fp16), 8 elements per thread.
__global__ void qk_to_f16_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int64_t n,
                                 __half* __restrict__ q16, __half* __restrict__ k16) {
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < 2 * n; i += stride) {
    const bool second = i >= n;
    const int64_t j = second ? i - n : i;
    float v[8];
    load8((second ? k : q) + j, v);
    uint4 o;
    o.x = pack_half2(v[0], v[1]), o.y = pack_half2(v[2], v[3]), o.z = pack_half2(v[4], v[5]), o.w = pack_half2(v[6], v[7]);
    *reinterpret_cast<uint4*>((second ? k16 : q16) + j) = o;
  }
}

// ----------------------------------------------------------------------------- modulation
// m = SiLU(vec) W^T + b.  dW[n, k] = sum_b dm[b, n] sv[b, k] (fp32, written once), db[n] =
// sum_b dm[b, n]; sv = SiLU(vec) as the forward used it (rounded to bf16 in bf16 mode).
// One warp per row n, 4 consecutive columns per lane per step (a warp covers 128 consecutive
// columns: conflict-free shared reads, 512-byte stores); sv in shared memory [batch, dim].
template <typename T>
__global__ void __launch_bounds__(256) modulation_wgrad_kernel(const T* __restrict__ vec, const float* __restrict__ dm,
                                                               int batch, int rows, int dim,
                                                               float* __restrict__ dw, float* __restrict__ db) {
  pdl_wait();
  extern __shared__ float sv[];
  for (int i = threadIdx.x; i < batch * dim; i += blockDim.x) {
    const float v = to_f32(vec[i]);
    float x = v / (1.f + expf(-v));
    if constexpr (sizeof(T) == 2) x = __bfloat162float(__float2bfloat16_rn(x));
    sv[i] = x;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int n = blockIdx.x * 8 + warp; n < rows; n += gridDim.x * 8) {
    float dmb[8];
#pragma unroll
    for (int bb = 0; bb < 8; ++bb) dmb[bb] = bb < batch ? dm[static_cast<size_t>(bb) * rows + n] : 0.f;
    if (lane == 0 && db) {
      float s = 0.f;
      for (int bb = 0; bb < batch; ++bb) s += dmb[bb];
      db[n] = s;
    }
    for (int k = lane * 4; dw && k < dim; k += 32 * 4) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int bb = 0; bb < batch; ++bb) {
        const float4 v = *reinterpret_cast<const float4*>(sv + bb * dim + k);
        o.x = fmaf(dmb[bb], v.x, o.x), o.y = fmaf(dmb[bb], v.y, o.y);
        o.z = fmaf(dmb[bb], v.z, o.z), o.w = fmaf(dmb[bb], v.w, o.w);
      }
      *reinterpret_cast<float4*>(dw + static_cast<size_t>(n) * dim + k) = o;
    }
  }
}

// dvec[b, k] = SiLU'(vec[b, k]) sum_n dm[b, n] W[n, k]: W read row by row in 16-byte loads;
// grid x = column groups of 8 * blockDim.x, y = row chunks; part [gridDim.y, batch, dim].
template <typename T>
__global__ void __launch_bounds__(128) modulation_dvec_partial_kernel(const T* __restrict__ w, const float* __restrict__ dm,
                                                                      int batch, int rows, int dim,
                                                                      float* __restrict__ part) {
  pdl_wait();
  const int k = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  const int per = (rows + gridDim.y - 1) / gridDim.y;
  const int n0 = blockIdx.y * per;
  const int n1 = n0 + per < rows ? n0 + per : rows;
  if (k >= dim) return;
  float acc[8][8];
#pragma unroll
  for (int bb = 0; bb < 8; ++bb)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[bb][e] = 0.f;
  // rows in ascending order; four rows' loads are issued before their products
  auto rows_from = [&](int n, int count) {
    float wv[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (u < count) load8(w + static_cast<size_t>(n + u) * dim + k, wv[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u >= count) break;
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) {
        if (bb < batch) {
          const float d = __ldg(dm + static_cast<size_t>(bb) * rows + n + u);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[bb][e] = fmaf(d, wv[u][e], acc[bb][e]);
        }
      }
    }
  };
  int n = n0;
  for (; n + 4 <= n1; n += 4) rows_from(n, 4);
  if (n < n1) rows_from(n, n1 - n);
#pragma unroll
  for (int bb = 0; bb < 8; ++bb)
    if (bb < batch) store8(part + (static_cast<size_t>(blockIdx.y) * batch + bb) * dim + k, acc[bb]);
}

// Block (32, kColsumGroups) over 32 columns: the chunk partials in the same two-level fixed order
// as batch_colsum_finish_kernel, then the SiLU derivative.
template <typename T>
__global__ void __launch_bounds__(32 * kColsumGroups) modulation_dvec_finish_kernel(
    const float* __restrict__ part, const T* __restrict__ vec, int chunks, int batch, int dim, int accumulate,
    float* __restrict__ dvec) {
  pdl_wait();
  __shared__ float grp[kColsumGroups][33];
  const int k = blockIdx.x * 32 + threadIdx.x;
  const int bb = blockIdx.y;
  float g = 0.f;
  if (k < dim)
    for (int i = threadIdx.y; i < chunks; i += kColsumGroups) g += part[(static_cast<size_t>(i) * batch + bb) * dim + k];
  grp[threadIdx.y][threadIdx.x] = g;
  __syncthreads();
  if (threadIdx.y != 0 || k >= dim) return;
  float acc = 0.f;
#pragma unroll 8
  for (int i = 0; i < kColsumGroups; ++i) acc += grp[i][threadIdx.x];
  const float v = to_f32(vec[static_cast<size_t>(bb) * dim + k]);
  const float sg = 1.f / (1.f + expf(-v));
  const float d = acc * sg * (1.f + v * (1.f - sg));
  float* dst = dvec + static_cast<size_t>(bb) * dim + k;
  *dst = accumulate ? *dst + d : d;
}

// ----------------------------------------------------------------------------- conversions
// out[i] = in[i] (TI -> TO), 8 elements per thread; n a multiple of 8.
template <typename TI, typename TO>
__global__ void convert_kernel(const TI* __restrict__ in, int64_t n, TO* __restrict__ out) {
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
    float v[8];
    load8(in + i, v);
    store8(out + i, v);
  }
}

}  // namespace

// Bytes of the partial-sum buffer the LayerNorm-modulate backward needs.
size_t ln_modulate_bwd_part_bytes(int batch, int rows_per_batch, int dim) {
  const int bpb = (rows_per_batch + kLnBwdRowsPerBlock - 1) / kLnBwdRowsPerBlock;
  return static_cast<size_t>(batch) * bpb * 2 * dim * sizeof(float);
}

// dx (fp32, accumulated) and the per-batch dscale, dshift (written into dmod at the given
// chunk pointers, batch stride mod_bstride) of h = LN(x)(1 + scale) + shift.
cudaError_t launch_ln_modulate_bwd(int act, int x_f32, const void* x, const void* dh, const float* scale,
                                   int64_t mod_bstride, int batch, int rows_per_batch, int dim, float eps,
                                   float* dx, float* dscale, float* dshift, int accumulate, float* part,
                                   cudaStream_t stream) {
  if (batch == 0 || rows_per_batch == 0) return cudaSuccess;
  const int chunks = (dim + kRowThreads * 8 - 1) / (kRowThreads * 8);
  if (chunks > kRowMaxChunks || dim % 8 != 0) return cudaErrorInvalidValue;
  const int bpb = (rows_per_batch + kLnBwdRowsPerBlock - 1) / kLnBwdRowsPerBlock;
  const LnBwdJob job{x, dh, scale, mod_bstride, dx, part, batch * rows_per_batch, rows_per_batch};
  const dim3 grid(batch * bpb);
  cudaError_t err = cudaSuccess;
  auto go = [&](auto nct) {
    constexpr int NCT = decltype(nct)::value;
    if (act == 1 && x_f32)
      err = launch_pdl(ln_modulate_bwd_kernel<float, __nv_bfloat16, NCT>, grid, dim3(kRowThreads), 0, stream, job, dim, eps);
    else if (act == 1)
      err = launch_pdl(ln_modulate_bwd_kernel<__nv_bfloat16, __nv_bfloat16, NCT>, grid, dim3(kRowThreads), 0, stream, job, dim, eps);
    else
      err = launch_pdl(ln_modulate_bwd_kernel<float, float, NCT>, grid, dim3(kRowThreads), 0, stream, job, dim, eps);
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
    go(std::integral_constant<int, kRowMaxChunks>());
  if (err != cudaSuccess) return err;
  count_launch();
  ColsumOut o{};
  o.out[0] = dscale;
  o.out[1] = dshift;
  o.out_bstride = mod_bstride;
  o.nvec = 2;
  o.accumulate = accumulate;
  err = launch_pdl(batch_colsum_finish_kernel, dim3((dim + 31) / 32, batch), dim3(32, kColsumGroups), 0, stream, part,
                   bpb, dim, o);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

size_t gated_residual_bwd_part_bytes(int batch, int rows_per_batch, int dim) {
  const int bpb = (rows_per_batch + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock;
  return static_cast<size_t>(batch) * bpb * dim * sizeof(float);
}

// df = dy gate (activation type) and dgate (per batch, into dgate + b * gate_bstride).
cudaError_t launch_gated_residual_bwd(int act, const float* dy, const void* f, const float* gate,
                                      int64_t gate_bstride, int batch, int rows_per_batch, int dim,
                                      void* df, float* dgate, float* part, cudaStream_t stream) {
  if (batch == 0 || rows_per_batch == 0) return cudaSuccess;
  if (dim % 8 != 0) return cudaErrorInvalidValue;
  const int bpb = (rows_per_batch + kBwdRowsPerBlock - 1) / kBwdRowsPerBlock;
  const dim3 grid((dim / 8 + 127) / 128, batch * bpb);
  cudaError_t err;
  if (act == 1)
    err = launch_pdl(gated_residual_bwd_kernel<__nv_bfloat16, __nv_bfloat16>, grid, dim3(128), 0, stream, dy,
                     static_cast<const __nv_bfloat16*>(f), gate, gate_bstride, rows_per_batch, dim,
                     static_cast<__nv_bfloat16*>(df), part);
  else
    err = launch_pdl(gated_residual_bwd_kernel<float, float>, grid, dim3(128), 0, stream, dy,
                     static_cast<const float*>(f), gate, gate_bstride, rows_per_batch, dim,
                     static_cast<float*>(df), part);
  if (err != cudaSuccess) return err;
  count_launch();
  ColsumOut o{};
  o.out[0] = dgate;
  o.out_bstride = gate_bstride;
  o.nvec = 1;
  o.accumulate = 0;
  err = launch_pdl(batch_colsum_finish_kernel, dim3((dim + 31) / 32, batch), dim3(32, kColsumGroups), 0, stream, part,
                   bpb, dim, o);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_gelu_bwd(int act, const void* du, const void* u_pre, int64_t n, int tanh_form, void* out,
                            cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const int grid = blocks_for(n / 8, 256, num_sms() * 8);
  cudaError_t err;
  if (act == 1)
    err = launch_pdl(gelu_bwd_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const __nv_bfloat16*>(du), static_cast<const __nv_bfloat16*>(u_pre), n, tanh_form,
                     static_cast<__nv_bfloat16*>(out));
  else
    err = launch_pdl(gelu_bwd_kernel<float>, dim3(grid), dim3(256), 0, stream, static_cast<const float*>(du),
                     static_cast<const float*>(u_pre), n, tanh_form, static_cast<float*>(out));
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

// dq, dk, dv fp32 [B, H, S_joint, 128] (the attention backward's outputs); dqkv and the norm
// gains in the activation type; dg_q, dg_k fp32 [128] written (fixed order over the blocks).
int qk_norm_rope_bwd_blocks() { return num_sms() * 4; }

cudaError_t launch_qk_norm_rope_bwd(int act, const QkBwdArgs& a, float* dg_q, float* dg_k, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.seq_s * a.heads;
  if (rows == 0) return cudaSuccess;
  const int grid = qk_norm_rope_bwd_blocks();
  cudaError_t err;
  // (the finish kernel skips a null dg_q or dg_k)
  if (act == 1)
    err = launch_pdl(qk_norm_rope_bwd_kernel<__nv_bfloat16, float, __nv_bfloat16>, dim3(grid), dim3(256), 0, stream, a);
  else
    err = launch_pdl(qk_norm_rope_bwd_kernel<float, float, float>, dim3(grid), dim3(256), 0, stream, a);
  if (err != cudaSuccess) return err;
  count_launch();
  ColsumOut o{};
  o.out[0] = dg_q;
  o.out[1] = dg_k;
  o.out_bstride = 0;
  o.nvec = 2;
  o.accumulate = 0;
  // the block partials are [grid, 2, 128]: one "batch" of `grid` blocks
  err = launch_pdl(batch_colsum_finish_kernel, dim3(128 / 32, 1), dim3(32, kColsumGroups), 0, stream, a.part, grid,
                   128, o);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

// amax(dO) over both streams' attention-output gradients (amax zeroed here), then per stream
// the pre-pass.  dO of stream s is [B, seq_s, H*128] of the activation type (bf16 here).
cudaError_t launch_grad_amax(const __nv_bfloat16* x, int64_t n, float* amax, bool zero_first, cudaStream_t stream) {
  if (zero_first) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    pdl_begin_call();  // the next kernel follows a memset: an ordinary launch
  }
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const int grid = blocks_for(n / 8, 256, num_sms() * 4);
  cudaError_t err = launch_pdl(amax_kernel_bf16, dim3(grid), dim3(256), 0, stream, x, n, amax);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_attn_bwd_pre(const __nv_bfloat16* o, const __nv_bfloat16* dout, int batch, int seq_s,
                                int seq_joint, int seq_pad, int seq_offset, int heads, const float* amax,
                                float* Dsum, __half* doh, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(batch) * seq_s * heads;
  if (rows == 0) return cudaSuccess;
  const int grid = blocks_for(rows, 8, num_sms() * 8);
  cudaError_t err = launch_pdl(attn_bwd_pre_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, o, dout,
                               batch, seq_s, seq_joint, seq_pad, seq_offset, heads, amax, Dsum, doh);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_untranspose_vt(const __half* vt, int bh, int seq, int seq_pad, __half* v, cudaStream_t stream) {
  const dim3 grid((seq + 31) / 32, 4, bh), block(32, 8);
  cudaError_t err = launch_pdl(untranspose_vt_kernel, grid, block, 0, stream, vt, seq, seq_pad, v);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_qk_to_f16(const __nv_bfloat16* q, const __nv_bfloat16* k, int64_t n, __half* q16, __half* k16,
                             cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const int grid = blocks_for(2 * n / 8, 256, num_sms() * 8);
  cudaError_t err = launch_pdl(qk_to_f16_kernel, dim3(grid), dim3(256), 0, stream, q, k, n, q16, k16);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

// Modulation backward: dW [rows, dim] fp32, db [rows] fp32 (may be null), dvec [batch, dim]
// fp32 (= or +=).  batch <= 8.  part: dvec_part_chunks() * batch * dim floats.
int modulation_dvec_chunks(int rows) { return rows < 128 ? (rows > 0 ? rows : 1) : 128; }

cudaError_t launch_modulation_bwd(int act, const void* vec, const void* w, const float* dm, int batch, int rows,
                                  int dim, float* dw, float* db, float* dvec, int accumulate, float* part,
                                  cudaStream_t stream) {
  if (batch == 0 || rows == 0) return cudaSuccess;
  if (batch > 8 || dim % 8 != 0) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(batch) * dim * sizeof(float);
  cudaError_t err;
  if (dw || db) {
    const int grid = blocks_for(rows, 8, num_sms() * 4);
    if (act == 1) {
      err = cudaFuncSetAttribute(modulation_wgrad_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err == cudaSuccess)
        err = launch_pdl(modulation_wgrad_kernel<__nv_bfloat16>, dim3(grid), dim3(256), smem, stream,
                         static_cast<const __nv_bfloat16*>(vec), dm, batch, rows, dim, dw, db);
    } else {
      err = cudaFuncSetAttribute(modulation_wgrad_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err == cudaSuccess)
        err = launch_pdl(modulation_wgrad_kernel<float>, dim3(grid), dim3(256), smem, stream,
                         static_cast<const float*>(vec), dm, batch, rows, dim, dw, db);
    }
    if (err != cudaSuccess) return err;
    count_launch();
  }
  if (dvec) {
    const int chunks = modulation_dvec_chunks(rows);
    const dim3 grid((dim / 8 + 127) / 128, chunks);
    if (act == 1)
      err = launch_pdl(modulation_dvec_partial_kernel<__nv_bfloat16>, grid, dim3(128), 0, stream,
                       static_cast<const __nv_bfloat16*>(w), dm, batch, rows, dim, part);
    else
      err = launch_pdl(modulation_dvec_partial_kernel<float>, grid, dim3(128), 0, stream,
                       static_cast<const float*>(w), dm, batch, rows, dim, part);
    if (err != cudaSuccess) return err;
    count_launch();
    const dim3 g2((dim + 31) / 32, batch), b2(32, kColsumGroups);
    if (act == 1)
      err = launch_pdl(modulation_dvec_finish_kernel<__nv_bfloat16>, g2, b2, 0, stream, part,
                       static_cast<const __nv_bfloat16*>(vec), chunks, batch, dim, accumulate, dvec);
    else
      err = launch_pdl(modulation_dvec_finish_kernel<float>, g2, b2, 0, stream, part,
                       static_cast<const float*>(vec), chunks, batch, dim, accumulate, dvec);
    if (err != cudaSuccess) return err;
    count_launch();
  }
  return cudaSuccess;
}

// dst = src converted between the activation type and fp32 (to_f32 = 1: act -> fp32).
cudaError_t launch_convert(int act, int to_f32, const void* src, int64_t n, void* dst, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const int grid = blocks_for(n / 8, 256, num_sms() * 8);
  cudaError_t err;
  if (act == 1 && to_f32)
    err = launch_pdl(convert_kernel<__nv_bfloat16, float>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const __nv_bfloat16*>(src), n, static_cast<float*>(dst));
  else if (act == 1)
    err = launch_pdl(convert_kernel<float, __nv_bfloat16>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const float*>(src), n, static_cast<__nv_bfloat16*>(dst));
  else
    err = launch_pdl(convert_kernel<float, float>, dim3(grid), dim3(256), 0, stream,
                     static_cast<const float*>(src), n, static_cast<float*>(dst));
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

}  // namespace mmdit
