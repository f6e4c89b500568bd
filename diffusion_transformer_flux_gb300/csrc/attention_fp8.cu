// attention_fp8.cu -- joint attention with E4M3 operands on tcgen05 tensor cores: the opt-in
// fp8_dot_product_attention of "FP8 training for Flux models" (§Configuration, FP8 model
// configuration; off by default, where the blocks keep attention in bf16).
//
// Per (batch, head), with per-tensor scales s_q, s_k, s_v (device scalars, e.g. delayed scaling's
// 448 / amax) and the probabilities' scale s_p = 448:
//   S  = E4M3(q s_q) E4M3(k s_k)^T / (s_q s_k sqrt(d))
//   Pt = exp(S - rowmax(S))                      (largest entry of each row exactly 1)
//   O  = E4M3(Pt s_p) E4M3(v s_v) / (s_p s_v) / rowsum(Pt)
// Both products are E4M3 x E4M3 (kind::f8f6f4, fp32 accumulation); the softmax is fp32 and the row
// sum is taken over the unquantised Pt.  The row maximum is the flash-style running maximum, moved
// whenever a tile raises it (so Pt <= 1 and its cast never saturates); O is rescaled in TMEM when
// that happens.  A tile's Pt is therefore cast relative to the maximum seen so far, which for
// rows whose maximum arrives late differs from the whole row's by a factor the cast rounds
// differently: those rows agree with the definition above to E4M3 rounding, not bit for bit.
//
// Layout as the bf16 kernel (attention.cu): one CTA owns two tiles of 128 query rows of one head
// and streams keys in tiles of 128 through a two-stage ring; warp 0 loads with TMA, warp 1 issues
// the MMAs (S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...), warps 4..7 and 8..11 run the
// softmax of tile A and B, one query row per thread.  Every operand tile is 128 rows x 128 bytes
// (one 128-byte swizzle block); P goes through shared memory as E4M3 codes (the A operand of the
// PV product).  A tile's P buffer is rewritten only after S of the next key tile is ready, which
// the MMA pipe completes after the previous PV product that read it.
// TMEM columns: S of A [0,128), S of B [128,256), O of A [256,384), O of B [384,512).
// Inputs are cast by the launcher: Q, K [B, H, S, 128] and V^T [B, H, 128, S_pad] as E4M3 codes.
#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kF8Threads = 384;
constexpr int kF8QTile = 128;
constexpr int kF8KvTile = 128;
constexpr int kF8Stages = 2;
constexpr int kTile8 = 128 * 128;  // 128 rows x 128 E4M3 codes
// Q_A Q_B | K x 2 | V x 2 | P_A P_B: 128 KB
constexpr int kF8SmemData = 8 * kTile8;
constexpr int kF8Smem = kF8SmemData + 256 + 1024;
constexpr uint32_t kF8TmemCols = 512;
constexpr uint32_t kIdesc8 = make_idesc<kKindF8>(128, 128);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 448.f;  // s_p: the scale of a tensor whose amax is 1

struct F8Barriers {
  uint64_t q_full;
  uint64_t k_full[kF8Stages];
  uint64_t v_full[kF8Stages];
  uint64_t kv_empty[kF8Stages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ uint8_t* f8_q(uint8_t* smem, int x) { return smem + x * kTile8; }
__device__ __forceinline__ uint8_t* f8_k(uint8_t* smem, int st) { return smem + (2 + st) * kTile8; }
__device__ __forceinline__ uint8_t* f8_v(uint8_t* smem, int st) { return smem + (4 + st) * kTile8; }
__device__ __forceinline__ uint8_t* f8_p(uint8_t* smem, int x) { return smem + (6 + x) * kTile8; }

// Softmax, P cast and output of query tile X (warps 4+4X .. 7+4X), one query row per thread.
template <typename OutT>
__device__ __forceinline__ void f8_softmax_role(F8Barriers* sb, uint8_t* smem, int X, uint32_t tmem, int q0,
                                                int bh, int heads, int seq, int split, int n_kv, OutT* out0,
                                                OutT* out1, float qk_scale_log2, float inv_pv, uint32_t* status) {
  volatile int* abort_flag = &sb->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_cols = tmem + static_cast<uint32_t>(X * 128) + lane_off;
  const uint32_t o_cols = tmem + 256u + static_cast<uint32_t>(X * 128) + lane_off;
  uint8_t* p_row = f8_p(smem, X) + row * 128;  // this row's 128-byte line of the P tile
  float m_run = -INFINITY, l_run = 0.f;
  for (int j = 0; j < n_kv; ++j) {
    const bool w = mbar_wait(&sb->s_full[X], static_cast<uint32_t>(j) & 1u, abort_flag, status, kErrAttnWait);
    if (!__all_sync(0xffffffffu, w)) return;
    tc_fence_after();
    const int kv0 = j * kF8KvTile;
    uint32_t r[4][32];
    tmem_ld32(s_cols, r[0]);
    tmem_ld32(s_cols + 32, r[1]);
    tmem_ld64_wait(s_cols + 64, r[2], r[3]);
    tmem_ld_deps64(r[0], r[1]);
    if (kv0 + kF8KvTile > seq) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (kv0 + 32 * c + i >= seq) r[c][i] = __float_as_uint(-INFINITY);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int i = 0; i < 32; i += 2) mx = fmax3(mx, __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
    mx *= qk_scale_log2;
    float alpha = 1.f;
    bool rescale = false;
    if (j == 0) {
      m_run = mx;
    } else if (mx > m_run) {
      alpha = fast_exp2(m_run - mx);
      m_run = mx;
      rescale = true;
    }
    // Pt = exp2(s c - m) in [0, 1]; the row sum over the fp32 values; E4M3 codes of Pt * 448
    // into this row's line of the P tile, chunk k of 16 keys at 16 (k ^ (row & 7)) (the 128-byte
    // swizzle the MMA descriptor reads)
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          p[i] = fast_exp2(fmaf(__uint_as_float(r[c][16 * h + i]), qk_scale_log2, -m_run));
          sum += p[i];
        }
        const uint2 lo = e4m3x8(p, kPScale), hi = e4m3x8(p + 8, kPScale);
        const int chunk = 2 * c + h;
        *reinterpret_cast<uint4*>(p_row + ((chunk ^ (row & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[16];
        tmem_ld16_wait(o_cols + c * 16, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st16(o_cols + c * 16, o);
      }
      tmem_st_wait();
    }
    l_run = l_run * alpha + sum;
    fence_proxy_async_smem();  // the P codes are read by the tensor core (async proxy)
    tc_fence_before();
    mbar_arrive(&sb->p_full[X]);
  }
  const bool w = mbar_wait(&sb->o_full, 0, abort_flag, status, kErrAttnWait);
  if (!__all_sync(0xffffffffu, w)) return;
  tc_fence_after();
  const int s_row = q0 + X * kF8QTile + row;
  const float f = inv_pv / l_run;  // 1 / (s_p s_v) for the codes, 1 / rowsum for the softmax
  OutT* dst = nullptr;
  if (s_row < seq) {
    const int b = bh / heads, hh = bh % heads;
    if (s_row < split)
      dst = out0 + ((static_cast<size_t>(b) * split + s_row) * heads + hh) * 128;
    else
      dst = out1 + ((static_cast<size_t>(b) * (seq - split) + (s_row - split)) * heads + hh) * 128;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld32_wait(o_cols + c * 32, o);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * f;
    if (dst) store32(dst + c * 32, v);
  }
}

template <typename OutT>
__global__ void __launch_bounds__(kF8Threads, 1)
    attention_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_vt, int heads, int seq, int split, OutT* out0,
                         OutT* out1, const float* __restrict__ scale_q, const float* __restrict__ scale_k,
                         const float* __restrict__ scale_v, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  F8Barriers* sb = reinterpret_cast<F8Barriers*>(smem + kF8SmemData);
  volatile int* abort_flag = &sb->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * 2 * kF8QTile;
  const int bh = blockIdx.y;
  const int n_kv = (seq + kF8KvTile - 1) / kF8KvTile;

  if (threadIdx.x == 0) {
    mbar_init(&sb->q_full, 1);
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&sb->k_full[s], 1);
      mbar_init(&sb->v_full[s], 1);
      mbar_init(&sb->kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sb->s_full[x], 1);
      mbar_init(&sb->p_full[x], 128);
    }
    mbar_init(&sb->o_full, 1);
    mbar_init(&sb->drain, 1);
    sb->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sb->tmem_slot, kF8TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tmem_slot;
  pdl_wait();  // the set-up above overlapped the previous kernel; its results are visible now

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: one 128 x 128-byte box per operand tile
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      mbar_arrive_expect_tx(&sb->q_full, 2 * kTile8);
      for (int x = 0; x < 2; ++x) tma_load_3d(f8_q(smem, x), &tm_q, &sb->q_full, 0, q0 + x * kF8QTile, bh);
      int last_parity[kF8Stages] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kF8Stages;
        const uint32_t ph = static_cast<uint32_t>(j / kF8Stages) & 1u;
        if (!mbar_wait(&sb->kv_empty[st], ph ^ 1u, abort_flag, status, kErrAttnWait)) break;
        const int kv0 = j * kF8KvTile;
        mbar_arrive_expect_tx(&sb->k_full[st], kTile8);
        tma_load_3d(f8_k(smem, st), &tm_k, &sb->k_full[st], 0, kv0, bh);
        mbar_arrive_expect_tx(&sb->v_full[st], kTile8);
        tma_load_3d(f8_v(smem, st), &tm_vt, &sb->v_full[st], kv0, 0, bh);
        last_parity[st] = static_cast<int>(ph);
      }
      if (*abort_flag) {
        // give the copies already issued a bounded chance to land before the CTA exits
        int never = 0;
        mbar_wait(&sb->q_full, 0, &never, status, 0);
        for (int s = 0; s < kF8Stages; ++s)
          if (last_parity[s] >= 0) {
            mbar_wait(&sb->k_full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
            mbar_wait(&sb->v_full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (the bf16 kernel's order; 4 MMAs of K = 32 codes per product)
      const uint64_t dq[2] = {sdesc_kmajor_sw128(smem_addr(f8_q(smem, 0))), sdesc_kmajor_sw128(smem_addr(f8_q(smem, 1)))};
      const uint64_t dk[2] = {sdesc_kmajor_sw128(smem_addr(f8_k(smem, 0))), sdesc_kmajor_sw128(smem_addr(f8_k(smem, 1)))};
      const uint64_t dv[2] = {sdesc_kmajor_sw128(smem_addr(f8_v(smem, 0))), sdesc_kmajor_sw128(smem_addr(f8_v(smem, 1)))};
      const uint64_t dp[2] = {sdesc_kmajor_sw128(smem_addr(f8_p(smem, 0))), sdesc_kmajor_sw128(smem_addr(f8_p(smem, 1)))};
      // K-step k: 32 codes (32 bytes) into the 128-byte swizzled rows
      auto koff = [](int k) -> uint64_t { return static_cast<uint64_t>((k * 32) >> 4); };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait(bar, parity, abort_flag, status, kErrAttnWait);
      };
      auto mma_s = [&](int x, int j) {
        const uint64_t k_desc = (j % kF8Stages) ? dk[1] : dk[0];
        const uint32_t d_s = tmem + static_cast<uint32_t>(x * 128);
#pragma unroll
        for (int k = 0; k < 4; ++k) tc_mma<kKindF8>(d_s, dq[x] + koff(k), k_desc + koff(k), kIdesc8, k > 0 ? 1u : 0u);
        tc_commit(&sb->s_full[x]);
      };
      auto mma_pv = [&](int x, int j) {
        const uint64_t v_desc = (j % kF8Stages) ? dv[1] : dv[0];
        const uint32_t d_o = tmem + 256u + static_cast<uint32_t>(x * 128);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma<kKindF8>(d_o, dp[x] + koff(k), v_desc + koff(k), kIdesc8, (j > 0 || k > 0) ? 1u : 0u);
      };
      auto k_ready = [&](int j) { return wait(&sb->k_full[j % kF8Stages], static_cast<uint32_t>(j / kF8Stages) & 1u); };
      auto v_ready = [&](int j) { return wait(&sb->v_full[j % kF8Stages], static_cast<uint32_t>(j / kF8Stages) & 1u); };
      auto p_ready = [&](int x, int j) {
        if (!wait(&sb->p_full[x], static_cast<uint32_t>(j) & 1u)) return false;
        tc_fence_after();
        return true;
      };
      bool ok = wait(&sb->q_full, 0) && k_ready(0);
      if (ok) {
        mma_s(0, 0);
        mma_s(1, 0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const bool more = j + 1 < n_kv;
        if (!(v_ready(j) && p_ready(0, j))) break;
        mma_pv(0, j);
        if (more) {
          if (!k_ready(j + 1)) break;
          mma_s(0, j + 1);
        }
        if (!p_ready(1, j)) break;
        mma_pv(1, j);
        tc_commit(&sb->kv_empty[j % kF8Stages]);
        if (more) mma_s(1, j + 1);
        if (j + 1 == n_kv) tc_commit(&sb->o_full);
      }
      if (*abort_flag) {
        int never = 0;
        tc_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, &never, status, 0);
      }
    }
  } else if (warp >= 4) {
    const float sq = __ldg(scale_q), sk = __ldg(scale_k), sv = __ldg(scale_v);
    const float qk_scale_log2 = kLog2e * 0.08838834764831845f / (sq * sk);  // log2(e) / (sqrt(128) s_q s_k)
    f8_softmax_role<OutT>(sb, smem, (warp - 4) >> 2, tmem, q0, bh, heads, seq, split, n_kv, out0, out1,
                          qk_scale_log2, 1.f / (kPScale * sv), status);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kF8TmemCols);
  }
}

// v [BH, S, 128] bf16 -> vt [BH, 128, S_pad] E4M3 codes of v * scale (zero codes past S).
__global__ void cast_transpose_v8_kernel(const __nv_bfloat16* __restrict__ v, int seq, int seq_pad,
                                         const float* __restrict__ scale, uint8_t* __restrict__ vt) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ float tile[32][33];
  const size_t bh = blockIdx.z;
  const int s0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  const float s = __ldg(scale);
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int t = s0 + i;
    tile[i][threadIdx.x] = t < seq ? __bfloat162float(v[(bh * seq + t) * 128 + j0 + threadIdx.x]) * s : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int t = s0 + threadIdx.x;
    if (t < seq_pad) vt[(bh * 128 + j0 + i) * seq_pad + t] = static_cast<uint8_t>(e4m3x2(tile[threadIdx.x][i], 0.f) & 0xFF);
  }
}

}  // namespace

cudaError_t launch_attention_fp8(const AttnFp8Problem& p, uint32_t* status, cudaStream_t stream) {
  const uint64_t bh = static_cast<uint64_t>(p.batch) * p.heads;
  if (bh == 0 || p.seq == 0) return cudaSuccess;
  if (p.seq_pad % 16 != 0 || p.seq_pad < p.seq) return cudaErrorInvalidValue;  // 16-byte rows of V^T codes
  // the casts: Q, K in place of layout, V transposed
  {
    QuantJob q[2] = {{p.q, p.q8, static_cast<int64_t>(bh) * p.seq * 128, p.scale_q, p.amax + 0},
                     {p.k, p.k8, static_cast<int64_t>(bh) * p.seq * 128, p.scale_k, p.amax + 1}};
    cudaError_t e = launch_quantize_e4m3(q, 2, stream);
    if (e != cudaSuccess) return e;
    const dim3 grid((p.seq_pad + 31) / 32, 4, static_cast<unsigned>(bh)), block(32, 8);
    e = launch_pdl(cast_transpose_v8_kernel, grid, block, 0, stream, p.v, p.seq, p.seq_pad, p.scale_v, p.vt8);
    if (e != cudaSuccess) return e;
    count_launch();
  }
  CUtensorMap tq, tk, tv;
  const uint64_t dqk[3] = {128, static_cast<uint64_t>(p.seq), bh};
  const uint64_t sqk[2] = {128, static_cast<uint64_t>(p.seq) * 128};
  const uint64_t dv[3] = {static_cast<uint64_t>(p.seq), 128, bh};
  const uint64_t sv[2] = {static_cast<uint64_t>(p.seq_pad), static_cast<uint64_t>(p.seq_pad) * 128};
  const uint32_t box[3] = {128, 128, 1};
  if (!encode_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.q8, dqk, sqk, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.k8, dqk, sqk, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.vt8, dv, sv, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const dim3 grid((p.seq + 2 * kF8QTile - 1) / (2 * kF8QTile), static_cast<unsigned>(bh));
  int dev = 0;
  cudaGetDevice(&dev);
  static int configured = -1;
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(attention_fp8_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attention_fp8_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  cudaError_t e;
  if (p.act == 1)
    e = launch_pdl(attention_fp8_kernel<__nv_bfloat16>, grid, dim3(kF8Threads), kF8Smem, stream, tq, tk, tv, p.heads,
                   p.seq, p.split, static_cast<__nv_bfloat16*>(p.out0), static_cast<__nv_bfloat16*>(p.out1),
                   p.scale_q, p.scale_k, p.scale_v, status);
  else
    e = launch_pdl(attention_fp8_kernel<float>, grid, dim3(kF8Threads), kF8Smem, stream, tq, tk, tv, p.heads, p.seq,
                   p.split, static_cast<float*>(p.out0), static_cast<float*>(p.out1), p.scale_q, p.scale_k,
                   p.scale_v, status);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
