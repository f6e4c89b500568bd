// attention.cu -- joint softmax attention on tcgen05 tensor cores (flash-style online softmax).
//
// Computes, per (batch, head), O = softmax(Q K^T / sqrt(128)) V over every key (no mask), the
// attention of "Flux architecture deep dive", §Implementation details (Attention implementation,
// Joint Attention Trick): one call over the concatenated [image; text] sequence.
//
// One CTA owns two tiles of 128 query rows (A and B) of one head and streams the keys in tiles
// of 128.  Twelve warps:
//   warp 0       TMA producer: both Q tiles once, then K and V^T tiles into a two-stage ring
//                (K and V of a stage have separate arrival barriers, so S can start before V
//                lands);
//   warp 1       MMA issuer, in the order S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//                so that the tensor core works on one query tile while the other's softmax runs
//                (a strict alternation: two independent issuers drift into lock-step);
//   warps 4..7   softmax of tile A, warps 8..11 softmax of tile B: one query row per thread (its
//                TMEM lane).  The row's 128 scores come out of TMEM in one round trip; a tree of
//                three-input maxima gives the row maximum; P = exp2(S * log2(e)/sqrt(d) - m) is
//                written back as packed fp16 over the score columns, where the PV product (fp16
//                P and V) reads it as its A operand straight from TMEM.  The running maximum is
//                only moved (and O rescaled in TMEM) when a row's maximum grows by more than
//                2^8; the final division by the row sum makes the result exact either way.
// TMEM columns: S/P of A [0,128), S/P of B [128,256), O of A [256,384), O of B [384,512).
// V arrives transposed ([B, H, 128, S_pad], fp16 holding the bf16 values) so the PV product
// reads a K-major operand.
#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kAttnThreads = 384;
constexpr int kQTile = 128;
constexpr int kKvTile = 128;
constexpr int kStages = 2;
constexpr int kHalfTile = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle column block)
constexpr int kTileBytes = 2 * kHalfTile;  // 128 rows x 128 bf16 = 32 KB
// Q_A Q_B | K x kStages | V x kStages: 192 KB
constexpr int kSmemData = (2 + 2 * kStages) * kTileBytes;
constexpr int kAttnSmem = kSmemData + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = make_idesc<kKindF16>(128, 128);      // S = Q K^T, bf16 operands
constexpr uint32_t kIdescPV = make_idesc_fp16(128, 128);          // O += P V, fp16 operands
constexpr float kScaleLog2 = 0.12751743074380043f;  // log2(e) / sqrt(128)
constexpr float kRescaleThreshold = 8.0f;           // in log2 units

struct AttnBarriers {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ uint8_t* q_tile(uint8_t* smem, int x) { return smem + x * kTileBytes; }
__device__ __forceinline__ uint8_t* k_tile(uint8_t* smem, int st) {
  return smem + (2 + st) * kTileBytes;
}
__device__ __forceinline__ uint8_t* v_tile(uint8_t* smem, int st) {
  return smem + (2 + kStages + st) * kTileBytes;
}

// Softmax, correction and output of query tile X (warps 4+4X .. 7+4X).
template <typename OutT>
__device__ __forceinline__ void softmax_role(AttnBarriers* sb, int X, uint32_t tmem, int q0, int bh,
                                             int heads, int seq, int split, int n_kv, OutT* out0,
                                             OutT* out1, float* lse, int lse_stride, uint32_t* status) {
  volatile int* abort_flag = &sb->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_cols = tmem + static_cast<uint32_t>(X * 128) + lane_off;
  const uint32_t o_cols = tmem + 256u + static_cast<uint32_t>(X * 128) + lane_off;
  float m_run = -INFINITY, l_run = 0.f;
  for (int j = 0; j < n_kv; ++j) {
    const bool w = mbar_wait(&sb->s_full[X], static_cast<uint32_t>(j) & 1u, abort_flag, status,
                             kErrAttnWait);
    if (!__all_sync(0xffffffffu, w)) return;
    tc_fence_after();
    const int kv0 = j * kKvTile;
    const bool tail = kv0 + kKvTile > seq;
    // the 128 scores of this row: one TMEM round trip (four loads, one wait)
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32(s_cols, r0);
    tmem_ld32(s_cols + 32, r1);
    tmem_ld64_wait(s_cols + 64, r2, r3);
    tmem_ld_deps64(r0, r1);
    if (tail) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (kv0 + i >= seq) r0[i] = __float_as_uint(-INFINITY);
        if (kv0 + 32 + i >= seq) r1[i] = __float_as_uint(-INFINITY);
        if (kv0 + 64 + i >= seq) r2[i] = __float_as_uint(-INFINITY);
        if (kv0 + 96 + i >= seq) r3[i] = __float_as_uint(-INFINITY);
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      mx0 = fmax3(mx0, fmax3(__uint_as_float(r0[i]), __uint_as_float(r1[i]), __uint_as_float(r2[i])),
                  __uint_as_float(r3[i]));
      mx1 = fmax3(mx1, fmax3(__uint_as_float(r0[i + 1]), __uint_as_float(r1[i + 1]),
                             __uint_as_float(r2[i + 1])),
                  __uint_as_float(r3[i + 1]));
    }
    const float mx = fmaxf(mx0, mx1) * kScaleLog2;
    float alpha = 1.f;
    bool rescale = false;
    if (j == 0) {
      m_run = mx;
    } else if (mx > m_run + kRescaleThreshold) {
      alpha = fast_exp2(m_run - mx);
      m_run = mx;
      rescale = true;
    }
    // P = exp2(s * scale - m) as fp16 pairs over the score columns (keys 2k, 2k+1 in column k),
    // 16 columns per store so each chunk of scores dies as soon as it is used; masked keys
    // hold -inf and give 0.  The argument and the row sum run on packed fp32 pairs; the sum
    // adds the fp16-rounded weights, the values the PV product uses (a sum of the unrounded
    // weights leaves the normalised weights off one by the rounding, which measured 2.7e-2
    // against 2.2e-2 x RMS at the block output in a CPU emulation of the 4096+512-token block).
    const uint64_t scale2 = f32x2(kScaleLog2, kScaleLog2);
    const uint64_t negm2 = f32x2(-m_run, -m_run);
    uint64_t sum_a = f32x2(0.f, 0.f), sum_b = f32x2(0.f, 0.f);
    auto emit = [&](const uint32_t (&sc)[32], uint32_t col) {
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float a, b;
        f32x2_split(ffma2(f32x2(__uint_as_float(sc[2 * i]), __uint_as_float(sc[2 * i + 1])), scale2,
                          negm2),
                    a, b);
        pk[i] = pack_half2(fast_exp2(a), fast_exp2(b));
        // the row sum takes the fp16 weights the PV product multiplies, so the normalised weights
        // sum to one exactly as used
        const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&pk[i]));
        if (i & 1)
          sum_b = fadd2(sum_b, f32x2(e.x, e.y));
        else
          sum_a = fadd2(sum_a, f32x2(e.x, e.y));
      }
      tmem_st16(s_cols + col, pk);
    };
    emit(r0, 0);   // keys [0, 32)   -> columns [0, 16)
    emit(r1, 16);  // keys [32, 64)  -> columns [16, 32)
    emit(r2, 32);  // keys [64, 96)  -> columns [32, 48)
    emit(r3, 48);  // keys [96, 128) -> columns [48, 64)
    float sum;
    {
      float a0, a1, b0, b1;
      f32x2_split(sum_a, a0, a1);
      f32x2_split(sum_b, b0, b1);
      sum = (a0 + a1) + (b0 + b1);
    }
    // O holds sum_{t<j} P_t V_t (PV(j-1) was issued before S(j), whose completion we saw);
    // rescaled after the scores are consumed, so the two never hold registers together
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t r[16];
        tmem_ld16_wait(o_cols + c * 16, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st16(o_cols + c * 16, r);
      }
    }
    tmem_st_wait();
    l_run = l_run * alpha + sum;
    tc_fence_before();
    mbar_arrive(&sb->p_full[X]);
  }
  const bool w = mbar_wait(&sb->o_full, 0, abort_flag, status, kErrAttnWait);
  if (!__all_sync(0xffffffffu, w)) return;
  tc_fence_after();
  const int s_row = q0 + X * kQTile + row;
  const float inv_l = 1.f / l_run;
  // training forward: the row's log-sum-exp in log2 units of the scaled scores, so that the
  // backward recomputes P = exp2(s log2(e) / sqrt(d) - L) (m_run and l_run agree however lazily
  // the maximum moved)
  if (lse && s_row < seq) lse[static_cast<size_t>(bh) * lse_stride + s_row] = m_run + log2f(l_run);
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
    uint32_t r[32];
    tmem_ld32_wait(o_cols + c * 32, r);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * inv_l;
    if (dst) store32(dst + c * 32, v);
  }
}


template <typename OutT>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_vt, int heads, int seq, int split,
                     OutT* out0, OutT* out1, float* lse, int lse_stride, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  AttnBarriers* sb = reinterpret_cast<AttnBarriers*>(smem + kSmemData);
  volatile int* abort_flag = &sb->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * 2 * kQTile;
  const int bh = blockIdx.y;
  const int n_kv = (seq + kKvTile - 1) / kKvTile;

  if (threadIdx.x == 0) {
    mbar_init(&sb->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
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
    tmem_alloc(&sb->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tmem_slot;
  pdl_wait();  // the set-up above overlapped the previous kernel; its results are visible now

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      mbar_arrive_expect_tx(&sb->q_full, 2 * kTileBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(q_tile(smem, x), &tm_q, &sb->q_full, 0, q0 + x * kQTile, bh);
        tma_load_3d(q_tile(smem, x) + kHalfTile, &tm_q, &sb->q_full, 64, q0 + x * kQTile, bh);
      }
      int last_parity[kStages] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        const uint32_t ph = static_cast<uint32_t>(j / kStages) & 1u;
        if (!mbar_wait(&sb->kv_empty[st], ph ^ 1u, abort_flag, status, kErrAttnWait)) break;
        const int kv0 = j * kKvTile;
        mbar_arrive_expect_tx(&sb->k_full[st], kTileBytes);
        tma_load_3d(k_tile(smem, st), &tm_k, &sb->k_full[st], 0, kv0, bh);
        tma_load_3d(k_tile(smem, st) + kHalfTile, &tm_k, &sb->k_full[st], 64, kv0, bh);
        mbar_arrive_expect_tx(&sb->v_full[st], kTileBytes);
        tma_load_3d(v_tile(smem, st), &tm_vt, &sb->v_full[st], kv0, 0, bh);
        tma_load_3d(v_tile(smem, st) + kHalfTile, &tm_vt, &sb->v_full[st], kv0 + 64, 0, bh);
        last_parity[st] = static_cast<int>(ph);
      }
      if (*abort_flag) {
        // give the copies already issued a bounded chance to land before the CTA exits
        int never = 0;
        mbar_wait(&sb->q_full, 0, &never, status, 0);
        for (int s = 0; s < kStages; ++s)
          if (last_parity[s] >= 0) {
            mbar_wait(&sb->k_full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
            mbar_wait(&sb->v_full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer.  Every wait or commit stalls this one thread for tens of
      // cycles while the tensor core drains its short queue, so the loop keeps them few: one
      // wait per K and per V tile (both query tiles read the same one), fences only after the
      // softmax's P hand-off (the TMA barriers need none), one release commit per K/V stage,
      // and shared-memory descriptors built once, each product then adding a constant.
      const uint64_t dq[2] = {sdesc_kmajor_sw128(smem_addr(q_tile(smem, 0))),
                              sdesc_kmajor_sw128(smem_addr(q_tile(smem, 1)))};
      const uint64_t dk[2] = {sdesc_kmajor_sw128(smem_addr(k_tile(smem, 0))),
                              sdesc_kmajor_sw128(smem_addr(k_tile(smem, 1)))};
      const uint64_t dv[2] = {sdesc_kmajor_sw128(smem_addr(v_tile(smem, 0))),
                              sdesc_kmajor_sw128(smem_addr(v_tile(smem, 1)))};
      // K-step k of a 128 x 128 operand tile: 16 elements into its 128-byte swizzle atoms
      auto koff = [](int k) -> uint64_t {
        return static_cast<uint64_t>(((k >> 2) * kHalfTile + (k & 3) * 32) >> 4);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait(bar, parity, abort_flag, status, kErrAttnWait);
      };
      auto mma_s = [&](int x, int j) {  // S_x(j) = Q_x K_j^T into columns [128x, 128x + 128)
        const uint64_t k_desc = (j % kStages) ? dk[1] : dk[0];
        const uint32_t d_s = tmem + static_cast<uint32_t>(x * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma<kKindF16>(d_s, dq[x] + koff(k), k_desc + koff(k), kIdesc, k > 0 ? 1u : 0u);
        tc_commit(&sb->s_full[x]);
      };
      auto mma_pv = [&](int x, int j) {  // O_x += P_x(j) V_j, P read from TMEM over S_x
        const uint64_t v_desc = (j % kStages) ? dv[1] : dv[0];
        const uint32_t p_cols = tmem + static_cast<uint32_t>(x * 128);  // 16 keys per 8 columns
        const uint32_t d_o = tmem + 256u + static_cast<uint32_t>(x * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma_ts_f16(d_o, p_cols + static_cast<uint32_t>(k * 8), v_desc + koff(k), kIdescPV,
                        (j > 0 || k > 0) ? 1u : 0u);
      };
      auto k_ready = [&](int j) {
        return wait(&sb->k_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u);
      };
      auto v_ready = [&](int j) {
        return wait(&sb->v_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u);
      };
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
        // PV_A(j) S_A(j+1) PV_B(j) S_B(j+1): the tensor core works on one tile while the other
        // tile's softmax runs
        if (!(v_ready(j) && p_ready(0, j))) break;
        mma_pv(0, j);
        if (more) {
          if (!k_ready(j + 1)) break;
          mma_s(0, j + 1);
        }
        if (!p_ready(1, j)) break;
        mma_pv(1, j);
        tc_commit(&sb->kv_empty[j % kStages]);  // K_j and V_j fully consumed once this lands
        if (more) mma_s(1, j + 1);
        if (j + 1 == n_kv) tc_commit(&sb->o_full);
      }
      if (*abort_flag) {
        // wait (bounded) for every MMA issued so far before TMEM is released
        int never = 0;
        tc_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, &never, status, 0);
      }
    }
  } else if (warp >= 4) {
    softmax_role<OutT>(sb, (warp - 4) >> 2, tmem, q0, bh, heads, seq, split, n_kv, out0, out1, lse,
                       lse_stride, status);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnProblem& p, uint32_t* status, cudaStream_t stream) {
  const uint64_t bh = static_cast<uint64_t>(p.batch) * p.heads;
  CUtensorMap tq, tk, tv;
  const uint64_t dqk[3] = {128, static_cast<uint64_t>(p.seq), bh};
  const uint64_t sqk[2] = {128 * 2, static_cast<uint64_t>(p.seq) * 128 * 2};
  const uint64_t dv[3] = {static_cast<uint64_t>(p.seq), 128, bh};
  const uint64_t sv[2] = {static_cast<uint64_t>(p.seq_pad) * 2,
                          static_cast<uint64_t>(p.seq_pad) * 128 * 2};
  const uint32_t box[3] = {64, 128, 1};
  if (!encode_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.q, dqk, sqk, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.k, dqk, sqk, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p.vt, dv, sv, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const dim3 grid((p.seq + 2 * kQTile - 1) / (2 * kQTile), static_cast<unsigned>(bh));
  int dev = 0;
  cudaGetDevice(&dev);
  static int configured = -1;
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attention_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kAttnSmem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  if (p.act == 1) {
    const cudaError_t e_ = launch_pdl(attention_kernel<__nv_bfloat16>, dim3(grid), dim3(kAttnThreads), kAttnSmem, stream,
        tq, tk, tv, p.heads, p.seq, p.split, static_cast<__nv_bfloat16*>(p.out0),
        static_cast<__nv_bfloat16*>(p.out1), p.lse, p.seq_pad, status);
    if (e_ != cudaSuccess) return e_;
  } else {
    const cudaError_t e_ = launch_pdl(attention_kernel<float>, dim3(grid), dim3(kAttnThreads), kAttnSmem, stream,
        tq, tk, tv, p.heads, p.seq, p.split, static_cast<float*>(p.out0), static_cast<float*>(p.out1),
        p.lse, p.seq_pad, status);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
