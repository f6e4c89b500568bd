// attention_bwd.cu -- the joint attention's backward on tcgen05 tensor cores (flash style).
//
// The pages train the blocks ("Flux architecture deep dive", §Training data flow) and print no
// backward; this is the chain rule of softmax(Q K^T / sqrt(d)) V.  Per (b, h), with
// P = exp2(c S - L) recomputed from the forward's row log-sum-exp L (log2 units,
// c = log2(e)/sqrt(128)) and D = rowsum(dO * O) from a pre-pass:
//   dV = P^T dO,  dS = P * (dO V^T - D) / sqrt(128),  dK = dS^T Q,  dQ = dS K.
// One CTA per (128-key tile, b*h) loops over 64-query tiles.  Twelve warps:
//   warp 0       TMA: K, V, K^T of its key tile once; per query tile Q, dO (64 x 128), Q^T,
//                dO^T (128 x 64) and L, D (64 floats each) into one stage
//   warp 1       MMA issuer:  S^T = K Q^T, dP^T = V dO^T          (M 128 keys, N 64, K 128)
//                             dV += P^T dO, dK += dS^T Q         (A from TMEM, N 128, K 64)
//                             dQ^T = K^T dS^T                    (M 128 = d, N 64, K 128 keys)
//   warps 4..7   one key row per thread: P^T and dS^T from S^T and dP^T (written back over them as
//                packed fp16 pairs, the A operands of dV and dK), dS into shared memory as
//                [query][key] (the B operand of dQ^T); at the end the dK, dV rows to global memory
//   warps 8..11  dQ^T out of TMEM (one d row per thread), added into the fp32 dQ [B, H, S, 128]
//                with coalesced atomic additions (lanes = consecutive d)
// TMEM columns: S^T [0,64) (P^T packed in [0,32)), dP^T [64,128) (dS^T packed in [64,96)),
// dV [128,256), dK [256,384), dQ^T [384,448).  Shared memory: K, V, K^T 32 KB each; one stage of
// Q, dO, Q^T, dO^T 16 KB each; dS 16 KB; L, D.  About 178 KB.
//
// Precision: S^T and dP^T from bf16 operands; P^T, dS^T and the transposed copies K^T, Q^T, dO^T
// in fp16 (10-bit mantissa: a CPU emulation of these tiles and roundings measured 2e-3 x RMS
// against the float64 gradients, 1.7e-2 with bf16).  dO (and so D, dS and every gradient)
// arrives multiplied by the power-of-two gradient scale the pre-pass chose, so that it sits in
// fp16's normal range; the consumers divide it out.
// Inputs: Q, K, V, dO [B, H, S, 128] bf16; K^T, Q^T, dO^T [B, H, 128, S_pad] fp16; L, D
// [B, H, S_pad] fp32 read in 64-row tiles with bulk copies (64 floats of slack past the end;
// rows at or past S are read but masked).  Outputs: dQ [B, H, S, 128] fp32 (zeroed by the
// launcher, added into), dK, dV [B, H, S, 128] fp32.  S_pad a multiple of 8.
#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kBwdThreads = 384;
constexpr int kKeyTile = 128;
constexpr int kQryTile = 64;
constexpr uint32_t kErrAttnBwdWait = 1u << 1;  // shares the attention's status bit
constexpr int kKTileBytes = 128 * 128 * 2;     // 128 rows x 128 bf16
constexpr int kKHalf = 128 * 128;              // 128 rows x 64 bf16 (one swizzle column block)
constexpr int kQTileBytes = 64 * 128 * 2;      // 64 rows x 128 bf16
constexpr int kQHalf = 64 * 128;               // 64 rows x 64 bf16
constexpr int kTTileBytes = 128 * 64 * 2;      // 128 rows x 64 bf16 (transposed 64-query tile)
// offsets in the 1024-aligned dynamic shared memory
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKTileBytes;
constexpr int kOffKT = kOffV + kKTileBytes;
constexpr int kOffQ = kOffKT + kKTileBytes;
constexpr int kOffDO = kOffQ + kQTileBytes;
constexpr int kOffQT = kOffDO + kQTileBytes;
constexpr int kOffDOT = kOffQT + kTTileBytes;
constexpr int kOffDS = kOffDOT + kTTileBytes;
constexpr int kOffL = kOffDS + kQTileBytes;
constexpr int kOffD = kOffL + kQryTile * 4;
constexpr int kOffBar = kOffD + kQryTile * 4;
constexpr int kBwdSmem = kOffBar + 256 + 1024;
constexpr uint32_t kBwdTmemCols = 512;
constexpr uint32_t kIdescN64 = make_idesc<kKindF16>(128, 64);        // S^T, dP^T: bf16 operands
constexpr uint32_t kIdescN64h = make_idesc_fp16(128, 64);          // dQ^T: fp16 K^T and dS
constexpr uint32_t kIdescN128h = make_idesc_fp16(128, 128);        // dV, dK: fp16 P^T / dS^T and copies
constexpr float kScaleLog2 = 0.12751743074380043f;  // log2(e) / sqrt(128)
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)

struct BwdBarriers {
  uint64_t kv_full;     // K, V, K^T landed
  uint64_t st_full;     // the stage (Q, dO, Q^T, dO^T, L, D) landed
  uint64_t st_empty;    // the stage's last reader (dK) completed
  uint64_t sp_full;     // S^T and dP^T in TMEM
  uint64_t p_full;      // P^T, dS^T in TMEM and dS in shared memory (128 arrivals)
  uint64_t ds_empty;    // dQ^T's MMA (the reader of dS) completed
  uint64_t dq_full;     // dQ^T in TMEM
  uint64_t dq_empty;    // dQ^T read out (128 arrivals)
  uint64_t kv_done;     // every MMA completed: dK, dV final
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// 128-byte swizzle: 16-byte chunk c of 128-byte line r lands at chunk c ^ (r & 7)
__device__ __forceinline__ uint32_t sw128(uint32_t line, uint32_t byte_in_line) {
  return line * 128u + ((((byte_in_line >> 4) ^ (line & 7u)) << 4) | (byte_in_line & 15u));
}


__global__ void __launch_bounds__(kBwdThreads, 1)
    attention_bwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_qt,
                         const __grid_constant__ CUtensorMap tm_dot, const float* __restrict__ lse,
                         const float* __restrict__ dsum, int seq, int seq_pad, float* __restrict__ dq,
                         float* __restrict__ dk, float* __restrict__ dv, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  BwdBarriers* sb = reinterpret_cast<BwdBarriers*>(smem + kOffBar);
  volatile int* abort_flag = &sb->abort_flag;
  float* sL = reinterpret_cast<float*>(smem + kOffL);
  float* sD = reinterpret_cast<float*>(smem + kOffD);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = blockIdx.x * kKeyTile;
  const int bh = blockIdx.y;
  const int n_q = (seq + kQryTile - 1) / kQryTile;
  // The key tiles of one head start their walk over the query tiles at staggered offsets, so
  // that their dQ additions do not land on the same rows at the same time.
  const int q_first = static_cast<int>((static_cast<int64_t>(blockIdx.x) * n_q) / gridDim.x);
  auto q_tile = [&](int i) { const int t = q_first + i; return (t >= n_q ? t - n_q : t) * kQryTile; };

  if (threadIdx.x == 0) {
    mbar_init(&sb->kv_full, 1);
    mbar_init(&sb->st_full, 1);
    mbar_init(&sb->st_empty, 1);
    mbar_init(&sb->sp_full, 1);
    mbar_init(&sb->p_full, 128);
    mbar_init(&sb->ds_empty, 1);
    mbar_init(&sb->dq_full, 1);
    mbar_init(&sb->dq_empty, 128);
    mbar_init(&sb->kv_done, 1);
    mbar_init(&sb->drain, 1);
    sb->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sb->tmem_slot, kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tmem_slot;
  pdl_wait();

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, abort_flag, status, kErrAttnBwdWait);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(&sb->kv_full, 3 * kKTileBytes);
      tma_load_3d(smem + kOffK, &tm_k, &sb->kv_full, 0, k0, bh);
      tma_load_3d(smem + kOffK + kKHalf, &tm_k, &sb->kv_full, 64, k0, bh);
      tma_load_3d(smem + kOffV, &tm_v, &sb->kv_full, 0, k0, bh);
      tma_load_3d(smem + kOffV + kKHalf, &tm_v, &sb->kv_full, 64, k0, bh);
      tma_load_3d(smem + kOffKT, &tm_kt, &sb->kv_full, k0, 0, bh);
      tma_load_3d(smem + kOffKT + kKHalf, &tm_kt, &sb->kv_full, k0 + 64, 0, bh);
      int issued = -1;
      for (int i = 0; i < n_q; ++i) {
        if (!wait(&sb->st_empty, (static_cast<uint32_t>(i) & 1u) ^ 1u)) break;
        const int q0 = q_tile(i);
        mbar_arrive_expect_tx(&sb->st_full, 2 * kQTileBytes + 2 * kTTileBytes + 2 * kQryTile * 4);
        tma_load_3d(smem + kOffQ, &tm_q, &sb->st_full, 0, q0, bh);
        tma_load_3d(smem + kOffQ + kQHalf, &tm_q, &sb->st_full, 64, q0, bh);
        tma_load_3d(smem + kOffDO, &tm_do, &sb->st_full, 0, q0, bh);
        tma_load_3d(smem + kOffDO + kQHalf, &tm_do, &sb->st_full, 64, q0, bh);
        tma_load_3d(smem + kOffQT, &tm_qt, &sb->st_full, q0, 0, bh);
        tma_load_3d(smem + kOffDOT, &tm_dot, &sb->st_full, q0, 0, bh);
        bulk_load(sL, lse + static_cast<size_t>(bh) * seq_pad + q0, kQryTile * 4, &sb->st_full);
        bulk_load(sD, dsum + static_cast<size_t>(bh) * seq_pad + q0, kQryTile * 4, &sb->st_full);
        issued = i;
      }
      if (*abort_flag) {
        // give the copies already issued a bounded chance to land before the CTA exits
        int never = 0;
        mbar_wait(&sb->kv_full, 0, &never, status, 0);
        if (issued >= 0) mbar_wait(&sb->st_full, static_cast<uint32_t>(issued) & 1u, &never, status, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint64_t dK = sdesc_kmajor_sw128(smem_addr(smem + kOffK));
      const uint64_t dV = sdesc_kmajor_sw128(smem_addr(smem + kOffV));
      const uint64_t dKT = sdesc_kmajor_sw128(smem_addr(smem + kOffKT));
      const uint64_t dQ = sdesc_kmajor_sw128(smem_addr(smem + kOffQ));
      const uint64_t dDO = sdesc_kmajor_sw128(smem_addr(smem + kOffDO));
      const uint64_t dQT = sdesc_kmajor_sw128(smem_addr(smem + kOffQT));
      const uint64_t dDOT = sdesc_kmajor_sw128(smem_addr(smem + kOffDOT));
      const uint64_t dDS = sdesc_kmajor_sw128(smem_addr(smem + kOffDS));
      // K-step k (16 elements) of a K-major operand whose 64-element column blocks are
      // `half` bytes apart
      auto koff = [](int k, int half) -> uint64_t {
        return static_cast<uint64_t>(((k >> 2) * half + (k & 3) * 32) >> 4);
      };
      const uint32_t t_s = tmem, t_dp = tmem + 64u, t_dv = tmem + 128u, t_dk = tmem + 256u,
                     t_dq = tmem + 384u;
      bool ok = wait(&sb->kv_full, 0);
      for (int i = 0; ok && i < n_q; ++i) {
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        if (!wait(&sb->st_full, ph)) break;
        tc_fence_after();
        // S^T = K Q_i^T and dP^T = V dO_i^T (128 keys x 64 queries, K = 128)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma<kKindF16>(t_s, dK + koff(k, kKHalf), dQ + koff(k, kQHalf), kIdescN64, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma<kKindF16>(t_dp, dV + koff(k, kKHalf), dDO + koff(k, kQHalf), kIdescN64, k > 0 ? 1u : 0u);
        tc_commit(&sb->sp_full);
        if (!wait(&sb->p_full, ph)) break;
        tc_fence_after();
        // dV += P^T dO_i and dK += dS^T Q_i: A from TMEM (8 columns per 16 queries), B the
        // transposed 128 x 64 tiles (one swizzle column block)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_ts_f16(t_dv, t_s + static_cast<uint32_t>(k * 8), dDOT + koff(k, 0), kIdescN128h,
                        (i > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_ts_f16(t_dk, t_dp + static_cast<uint32_t>(k * 8), dQT + koff(k, 0), kIdescN128h,
                        (i > 0 || k > 0) ? 1u : 0u);
        tc_commit(&sb->st_empty);  // the stage may be refilled once dK's reads are done
        // dQ^T = K^T dS^T (128 d x 64 queries, K = 128 keys) once the previous dQ^T is out
        if (i > 0 && !wait(&sb->dq_empty, ph ^ 1u)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma<kKindF16>(t_dq, dKT + koff(k, kKHalf), dDS + koff(k, kQHalf), kIdescN64h, k > 0 ? 1u : 0u);
        tc_commit(&sb->ds_empty);
        tc_commit(&sb->dq_full);
        if (i + 1 == n_q) tc_commit(&sb->kv_done);
      }
      if (*abort_flag) {
        int never = 0;
        tc_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, &never, status, 0);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- P^T and dS^T, one key row per thread
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key k0 + row
    const bool key_ok = k0 + row < seq;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off, t_dp = tmem + 64u + lane_off;
    uint8_t* ds_tile = smem + kOffDS;
    const uint32_t key_half = static_cast<uint32_t>(row >> 6);       // dS column block
    const uint32_t key_byte = static_cast<uint32_t>(row & 63) * 2u;  // byte within the 128-byte line
    for (int i = 0; i < n_q; ++i) {
      const uint32_t ph = static_cast<uint32_t>(i) & 1u;
      const int q0 = q_tile(i);
      // the stage (L, D) was written by the bulk copies: observe its barrier here too
      bool w = wait(&sb->st_full, ph);
      if (w) w = wait(&sb->sp_full, ph);
      // dS of the previous tile must have been consumed by its dQ^T product
      if (w && i > 0) w = wait(&sb->ds_empty, ph ^ 1u);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
#pragma unroll 1
      for (int h2 = 0; h2 < 2; ++h2) {  // 32 queries at a time
        uint32_t s[32], dp[32];
        tmem_ld32_wait(t_s + static_cast<uint32_t>(h2 * 32), s);
        tmem_ld32_wait(t_dp + static_cast<uint32_t>(h2 * 32), dp);
        uint32_t pk[16], dk2[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float p2[2], d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int q = h2 * 32 + 2 * c + e;
            const bool ok = key_ok && (q0 + q < seq);
            const float p = ok ? fast_exp2(__uint_as_float(s[2 * c + e]) * kScaleLog2 - sL[q]) : 0.f;
            p2[e] = p;
            d2[e] = ok ? p * (__uint_as_float(dp[2 * c + e]) - sD[q]) * kInvSqrtD : 0.f;
          }
          pk[c] = pack_half2(p2[0], p2[1]);
          dk2[c] = pack_half2(d2[0], d2[1]);
          // dS[q][key] into the [query][key] tile (128-byte swizzle, two 64-key blocks)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t q = static_cast<uint32_t>(h2 * 32 + 2 * c + e);
            const uint32_t off = key_half * kQHalf + sw128(q, key_byte);
            *reinterpret_cast<__half*>(ds_tile + off) = __float2half_rn(d2[e]);
          }
        }
        tmem_st16(t_s + static_cast<uint32_t>(h2 * 16), pk);    // P^T packed: columns [0, 32)
        tmem_st16(t_dp + static_cast<uint32_t>(h2 * 16), dk2);  // dS^T packed: columns [64, 96)
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sb->p_full);
    }
    // dK and dV rows once every product is done
    const bool w = wait(&sb->kv_done, 0);
    if (__all_sync(0xffffffffu, w)) {
      tc_fence_after();
      const size_t grow = (static_cast<size_t>(bh) * seq + k0 + row) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tmem + 128u + lane_off + static_cast<uint32_t>(c * 32), r);
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (key_ok) store32(dv + grow + c * 32, v);
        tmem_ld32_wait(tmem + 256u + lane_off + static_cast<uint32_t>(c * 32), r);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (key_ok) store32(dk + grow + c * 32, v);
      }
    }
  } else if (warp >= 8) {
    // ---------------- dQ^T out of TMEM, added into dQ (thread = d row)
    const int quarter = warp & 3;
    const int d = quarter * 32 + lane;
    const uint32_t t_dq = tmem + 384u + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int i = 0; i < n_q; ++i) {
      const bool w = wait(&sb->dq_full, static_cast<uint32_t>(i) & 1u);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      uint32_t a[32], b[32];
      tmem_ld32_wait(t_dq, a);
      tmem_ld32_wait(t_dq + 32u, b);
      tc_fence_before();
      mbar_arrive(&sb->dq_empty);
      const int q0 = q_tile(i);
      float* base = dq + (static_cast<size_t>(bh) * seq + q0) * 128 + d;
#pragma unroll 4
      for (int q = 0; q < 32; ++q)
        if (q0 + q < seq) atomicAdd(base + static_cast<size_t>(q) * 128, __uint_as_float(a[q]));
#pragma unroll 4
      for (int q = 0; q < 32; ++q)
        if (q0 + 32 + q < seq) atomicAdd(base + static_cast<size_t>(32 + q) * 128, __uint_as_float(b[q]));
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention_bwd(const AttnBwdProblem& p, uint32_t* status, cudaStream_t stream) {
  const uint64_t bh = static_cast<uint64_t>(p.batch) * p.heads;
  if (bh == 0 || p.seq == 0) return cudaSuccess;
  if (p.seq_pad % 8 != 0 || p.seq_pad < p.seq) return cudaErrorInvalidValue;  // 16-byte rows for TMA and the L, D bulk loads
  CUtensorMap tk, tv, tkt, tq, tdo, tqt, tdot;
  const uint64_t drow[3] = {128, static_cast<uint64_t>(p.seq), bh};
  const uint64_t srow[2] = {128 * 2, static_cast<uint64_t>(p.seq) * 128 * 2};
  const uint64_t dcol[3] = {static_cast<uint64_t>(p.seq), 128, bh};
  const uint64_t scol[2] = {static_cast<uint64_t>(p.seq_pad) * 2, static_cast<uint64_t>(p.seq_pad) * 128 * 2};
  const uint32_t box_k[3] = {64, 128, 1};   // 128 rows x 64 elements
  const uint32_t box_q[3] = {64, 64, 1};    // 64 rows x 64 elements
  const uint32_t box_t[3] = {64, 128, 1};   // 64 queries x 128 d rows (transposed tiles)
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto HF = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_tmap(&tk, BF, 3, p.k, drow, srow, box_k, SW) || !encode_tmap(&tv, BF, 3, p.v, drow, srow, box_k, SW) ||
      !encode_tmap(&tkt, HF, 3, p.kt, dcol, scol, box_k, SW) ||
      !encode_tmap(&tq, BF, 3, p.q, drow, srow, box_q, SW) ||
      !encode_tmap(&tdo, BF, 3, p.dout, drow, srow, box_q, SW) ||
      !encode_tmap(&tqt, HF, 3, p.qt, dcol, scol, box_t, SW) ||
      !encode_tmap(&tdot, HF, 3, p.dout_t, dcol, scol, box_t, SW))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(p.dq, 0, bh * p.seq * 128 * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  pdl_begin_call();  // the kernel follows a memset: an ordinary launch
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    e = cudaFuncSetAttribute(attention_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const dim3 grid((p.seq + kKeyTile - 1) / kKeyTile, static_cast<unsigned>(bh));
  e = launch_pdl(attention_bwd_kernel, grid, dim3(kBwdThreads), kBwdSmem, stream, tk, tv, tkt, tq, tdo, tqt, tdot,
                 p.lse, p.dsum, p.seq, p.seq_pad, p.dq, p.dk, p.dv, status);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
