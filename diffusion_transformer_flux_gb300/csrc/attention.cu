// attention.cu -- joint softmax attention on tcgen05 tensor cores (flash-style online softmax).
//
// Computes, per (batch, head), O = softmax(Q K^T / sqrt(128)) V over every key (no mask), the
// attention of "Flux architecture deep dive", §Implementation details (Attention implementation,
// Joint Attention Trick): one call over the concatenated [image; text] sequence.
//
// One CTA owns 128 query rows of one head and streams the keys in tiles of 128:
//   warp 0      TMA producer: Q once, then K and V^T tiles into a two-stage ring;
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM score buffers, then
//               O += P_{j-1} V_{j-1} into a TMEM accumulator, so QK^T of tile j runs while the
//               softmax warps work on tile j-1;
//   warps 2..5  softmax: one query row per thread (its TMEM lane), exp2 with the 1/sqrt(d)
//               scale folded in, P written to shared memory in the tensor core's swizzled
//               layout, and the running-max correction of O applied in TMEM only when the
//               row maximum grows by more than 2^8 (otherwise the stale maximum is kept; the
//               final division by the row sum makes the result exact either way).
// V arrives transposed ([B, H, 128, S_pad]) so both products read K-major operands.
#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kAttnThreads = 192;
constexpr int kQTile = 128;
constexpr int kKvTile = 128;
constexpr int kKvStages = 2;
constexpr int kHalfTile = 128 * 128;                      // one 128-row x 64-element bf16 atom block
constexpr int kQBytes = 2 * kHalfTile;                    // 32 KB
constexpr int kKBytes = 2 * kHalfTile;
constexpr int kVBytes = 2 * kHalfTile;
constexpr int kPBytes = 2 * kHalfTile;
constexpr int kStageBytes = kKBytes + kVBytes;            // 64 KB
constexpr int kSmemData = kQBytes + kKvStages * kStageBytes + 2 * kPBytes;  // 224 KB
constexpr int kAttnSmem = kSmemData + 256 + 1024;
constexpr uint32_t kTmemCols = 512;                       // S0 | S1 | O | (unused)
constexpr uint32_t kIdescQK = make_idesc<kKindF16>(128, 128);
constexpr float kScaleLog2 = 0.12751743074380043f;        // log2(e) / sqrt(128)
constexpr float kRescaleThreshold = 8.0f;                 // in log2 units

struct AttnSmem {
  uint64_t q_full;
  uint64_t kv_full[kKvStages];
  uint64_t kv_empty[kKvStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t p_free[2];
  uint64_t pv_done;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

// Softmax / correction / output role: warps 2..5, one query row per thread.
template <typename OutT>
__device__ __forceinline__ void softmax_role(AttnSmem* sb, uint8_t* s_p, uint32_t tmem,
                                             uint32_t tmem_o, int q0, int bh, int heads, int seq,
                                             int split, int n_kv, OutT* out0, OutT* out1,
                                             uint32_t* status) {
  volatile int* abort_flag = &sb->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int j = 0; j < n_kv; ++j) {
    const int buf = j & 1;
    bool w = mbar_wait(&sb->s_full[buf], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status,
                       kErrAttnWait);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float s[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32_wait(tmem + static_cast<uint32_t>(buf * 128 + c * 32) + lane_off, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
    }
    tc_fence_before();
    mbar_arrive(&sb->s_free[buf]);  // scores are in registers; the buffer may be reused
    const int kv0 = j * kKvTile;
    if (kv0 + kKvTile > seq) {
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (kv0 + i >= seq) s[i] = -INFINITY;
    }
    float mx = s[0];
#pragma unroll
    for (int i = 1; i < 128; ++i) mx = fmaxf(mx, s[i]);
    mx *= kScaleLog2;
    float alpha = 1.f;
    bool rescale = false;
    if (j == 0) {
      m_run = mx;
    } else if (mx > m_run + kRescaleThreshold) {
      alpha = fast_exp2(m_run - mx);
      m_run = mx;
      rescale = true;
    }
    uint32_t pk[64];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float p0 = fast_exp2(fmaf(s[2 * i], kScaleLog2, -m_run));
      const float p1 = fast_exp2(fmaf(s[2 * i + 1], kScaleLog2, -m_run));
      pk[i] = pack_bf16x2(p0, p1);
      // normalise by the sum of the rounded weights that the PV product actually uses
      sum += bf16_lo(pk[i]) + bf16_hi(pk[i]);
    }
    // P_j goes to buffer j&1 once PV_{j-2} has finished reading it.
    w = mbar_wait(&sb->p_free[buf], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag, status,
                  kErrAttnWait);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    // Row `row` of a 128-byte-swizzled K-major tile: 16-byte chunk c sits at c ^ (row % 8).
    uint8_t* prow = s_p + buf * kPBytes + row * 128;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int atom = c >> 3, cc = c & 7;
      uint4 u = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      *reinterpret_cast<uint4*>(prow + atom * kHalfTile + ((cc ^ (row & 7)) << 4)) = u;
    }
    fence_proxy_async_smem();
    if (__any_sync(0xffffffffu, rescale)) {
      // O holds sum_{t<j} P_t V_t only after PV_{j-1} completes.
      w = mbar_wait(&sb->pv_done, static_cast<uint32_t>(j - 1) & 1u, abort_flag, status,
                    kErrAttnWait);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        const uint32_t ta = tmem_o + static_cast<uint32_t>(c * 32) + lane_off;
        tmem_ld32_wait(ta, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(ta, r);
      }
      tmem_st_wait();
    }
    l_run = l_run * alpha + sum;
    tc_fence_before();
    mbar_arrive(&sb->p_full[buf]);
  }
  if (!ok) return;
  bool w = mbar_wait(&sb->o_full, 0, abort_flag, status, kErrAttnWait);
  if (!__all_sync(0xffffffffu, w)) return;
  tc_fence_after();
  const int s_row = q0 + row;
  const float inv_l = 1.f / l_run;
  OutT* dst = nullptr;
  if (s_row < seq) {
    const int b = bh / heads, h = bh % heads;
    if (s_row < split)
      dst = out0 + ((static_cast<size_t>(b) * split + s_row) * heads + h) * 128;
    else
      dst = out1 + ((static_cast<size_t>(b) * (seq - split) + (s_row - split)) * heads + h) * 128;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32_wait(tmem_o + static_cast<uint32_t>(c * 32) + lane_off, r);
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
                     OutT* out0, OutT* out1, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* s_q = smem;
  uint8_t* s_kv = smem + kQBytes;
  uint8_t* s_p = s_kv + kKvStages * kStageBytes;
  AttnSmem* sb = reinterpret_cast<AttnSmem*>(smem + kSmemData);
  volatile int* abort_flag = &sb->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kQTile;
  const int bh = blockIdx.y;
  const int n_kv = (seq + kKvTile - 1) / kKvTile;

  if (threadIdx.x == 0) {
    mbar_init(&sb->q_full, 1);
    for (int s = 0; s < kKvStages; ++s) mbar_init(&sb->kv_full[s], 1), mbar_init(&sb->kv_empty[s], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb->s_full[i], 1);
      mbar_init(&sb->s_free[i], 128);
      mbar_init(&sb->p_full[i], 128);
      mbar_init(&sb->p_free[i], 1);
    }
    mbar_init(&sb->pv_done, 1);
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
  const uint32_t tmem_o = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      mbar_arrive_expect_tx(&sb->q_full, kQBytes);
      tma_load_3d(s_q, &tm_q, &sb->q_full, 0, q0, bh);
      tma_load_3d(s_q + kHalfTile, &tm_q, &sb->q_full, 64, q0, bh);
      int last_parity[kKvStages] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kKvStages;
        const uint32_t ph = static_cast<uint32_t>(j / kKvStages) & 1u;
        if (!mbar_wait(&sb->kv_empty[st], ph ^ 1u, abort_flag, status, kErrAttnWait)) break;
        uint8_t* sk = s_kv + st * kStageBytes;
        uint8_t* sv = sk + kKBytes;
        const int kv0 = j * kKvTile;
        mbar_arrive_expect_tx(&sb->kv_full[st], kStageBytes);
        tma_load_3d(sk, &tm_k, &sb->kv_full[st], 0, kv0, bh);
        tma_load_3d(sk + kHalfTile, &tm_k, &sb->kv_full[st], 64, kv0, bh);
        tma_load_3d(sv, &tm_vt, &sb->kv_full[st], kv0, 0, bh);
        tma_load_3d(sv + kHalfTile, &tm_vt, &sb->kv_full[st], kv0 + 64, 0, bh);
        last_parity[st] = static_cast<int>(ph);
      }
      if (*abort_flag) {
        int never = 0;
        mbar_wait(&sb->q_full, 0, &never, status, 0);
        for (int s = 0; s < kKvStages; ++s)
          if (last_parity[s] >= 0)
            mbar_wait(&sb->kv_full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t aq = smem_addr(s_q);
      const uint32_t ap = smem_addr(s_p);
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(&sb->p_full[i & 1], static_cast<uint32_t>(i >> 1) & 1u, abort_flag, status,
                       kErrAttnWait))
          return false;
        tc_fence_after();
        const uint32_t pa = ap + static_cast<uint32_t>((i & 1) * kPBytes);
        const uint32_t vb = smem_addr(s_kv + (i % kKvStages) * kStageBytes + kKBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = static_cast<uint32_t>((k >> 2) * kHalfTile + (k & 3) * 32);
          tc_mma<kKindF16>(tmem_o, sdesc_kmajor_sw128(pa + off), sdesc_kmajor_sw128(vb + off),
                           kIdescQK, (i > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&sb->pv_done);
        tc_commit(&sb->p_free[i & 1]);
        tc_commit(&sb->kv_empty[i % kKvStages]);
        return true;
      };
      bool ok = mbar_wait(&sb->q_full, 0, abort_flag, status, kErrAttnWait);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % kKvStages;
        if (!mbar_wait(&sb->kv_full[st], static_cast<uint32_t>(j / kKvStages) & 1u, abort_flag,
                       status, kErrAttnWait) ||
            !mbar_wait(&sb->s_free[j & 1], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag,
                       status, kErrAttnWait)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = smem_addr(s_kv + st * kStageBytes);
        const uint32_t d_s = tmem + static_cast<uint32_t>((j & 1) * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = static_cast<uint32_t>((k >> 2) * kHalfTile + (k & 3) * 32);
          tc_mma<kKindF16>(d_s, sdesc_kmajor_sw128(aq + off), sdesc_kmajor_sw128(kb + off),
                           kIdescQK, k > 0 ? 1u : 0u);
        }
        tc_commit(&sb->s_full[j & 1]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok && issue_pv(n_kv - 1)) tc_commit(&sb->o_full);
      if (*abort_flag) {
        int never = 0;
        tc_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, &never, status, 0);
      }
    }
  } else {
    softmax_role<OutT>(sb, s_p, tmem, tmem_o, q0, bh, heads, seq, split, n_kv, out0, out1, status);
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
      !encode_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.vt, dv, sv, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const dim3 grid((p.seq + kQTile - 1) / kQTile, static_cast<unsigned>(bh));
  int dev = 0;
  cudaGetDevice(&dev);
  if (p.act == 1) {
    static int configured = -1;
    if (configured != dev) {
      cudaError_t e = cudaFuncSetAttribute(attention_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
      if (e != cudaSuccess) return e;
      configured = dev;
    }
    attention_kernel<__nv_bfloat16><<<grid, kAttnThreads, kAttnSmem, stream>>>(
        tq, tk, tv, p.heads, p.seq, p.split, static_cast<__nv_bfloat16*>(p.out0),
        static_cast<__nv_bfloat16*>(p.out1), status);
  } else {
    static int configured = -1;
    if (configured != dev) {
      cudaError_t e = cudaFuncSetAttribute(attention_kernel<float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
      if (e != cudaSuccess) return e;
      configured = dev;
    }
    attention_kernel<float><<<grid, kAttnThreads, kAttnSmem, stream>>>(
        tq, tk, tv, p.heads, p.seq, p.split, static_cast<float*>(p.out0),
        static_cast<float*>(p.out1), status);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
