// gemm_pair.cuh -- the persistent GEMM  C = A * W^T  on CTA pairs (tcgen05 cta_group::2).
//
// A cluster of two CTAs on two SMs computes 256 x BN output tiles.  CTA r of the pair loads
// rows [128 r, 128 r + 128) of the tile's A slice and rows [r BN/2, (r + 1) BN/2) of its W
// slice into its own shared memory; the leader (r = 0) issues one M = 256 MMA per K step that
// reads both CTAs' operands and writes each CTA's 128 accumulator rows into that CTA's TMEM.
// Each SM therefore streams 32 KB per 128-byte K slice instead of the 48 KB a single-CTA
// 128 x 256 tile needs for the same MMA work, which is what bounds the single-CTA kernel.
//
// Roles (per CTA, as in gemm_tc_kernel):
//   warp 0   TMA producer: loads this CTA's A and W rows; the bytes complete on the leader's
//            stage barrier, which the leader alone arms with the pair's total byte count;
//   warp 1   (leader) MMA issuer; its commits arrive on the stage-empty and accumulator-full
//            barriers of both CTAs; (peer) idle after the tensor-memory allocation;
//   warps 2+ epilogue on this CTA's TMEM rows; each warp then arrives on the leader's
//            accumulator-empty barrier.
// Every mbarrier wait is bounded (common.cuh); cluster barriers after set-up and before
// teardown keep either CTA from leaving while the other may still address it.
//
// MAJ selects how the operands are stored (16-bit kinds): bit 0 set, A is held as A^T [K, M];
// bit 1 set, W is held as W^T [K, N].  Such an operand is loaded as two 64-wide MN blocks of
// 64 k lines each (the same 16 KB per CTA and stage) and read by the MMA through MN-major
// descriptors, so a transposed product (a weight or input gradient) needs no transpose pass.
#pragma once

#include "gemm_kernel.cuh"

namespace mmdit {

template <int BN>
struct PairCfg {
  static constexpr int kStages = 6;
  static constexpr int kABytes = kBM * 128;       // this CTA's 128 rows of A
  static constexpr int kBBytes = (BN / 2) * 128;  // this CTA's BN/2 rows of W
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;        // double-buffered accumulator
  static constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
};

template <int KIND, int BN, int EPI, int MAJ = 0>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads<EPI>(), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_b0,
                     const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_b1,
                     int M0, int M1, int N, int K, int K1, int interleave, const __grid_constant__ EpiArgs ep0,
                     const __grid_constant__ EpiArgs ep1, uint32_t* status) {
  using Cfg = PairCfg<BN>;
  using TE = typename KindTraits<KIND>::TE;
  constexpr int kBK = 128 / KindTraits<KIND>::kEltBytes;    // elements per 128-byte K slice
  constexpr int kUmmaK = 32 / KindTraits<KIND>::kEltBytes;  // K of one tcgen05.mma
  constexpr int kKSteps = kBK / kUmmaK;
  constexpr uint32_t kIdesc = make_idesc<KIND>(2 * kBM, BN) | ((MAJ & 1) ? kIdescAMnMajor : 0u) |
                              ((MAJ & 2) ? kIdescBMnMajor : 0u);
  static_assert(MAJ == 0 || (KindTraits<KIND>::kEltBytes == 2 && BN == 256), "MN-major: 16-bit kinds, BN 256");
  constexpr int kMnBlock = 128 / KindTraits<KIND>::kEltBytes;  // MN elements per 128-byte line
  constexpr uint32_t kMnBoxBytes = static_cast<uint32_t>(kBK) * 128u;  // one MN block of kBK k lines
  constexpr int kEpiWarps = 4 * EpiGroups<EPI>::value;

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

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb0 = (K + kBK - 1) / kBK, num_kb1 = (K1 + kBK - 1) / kBK;
  // Pair tiles: problem 0's (M fastest), then problem 1's (or, interleaved, alternating); CTA r
  // takes M block 2 mp + r.
  const int num_n = N / BN;
  const int pm0 = (M0 + 2 * kBM - 1) / (2 * kBM), pm1 = (M1 + 2 * kBM - 1) / (2 * kBM);
  const int tiles0 = pm0 * num_n;
  const int tiles = tiles0 + pm1 * num_n;
  const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
  auto decode = [&](int tile, int& prob, int& m0, int& nb) {
    // Interleaved (equal tile counts): every pair walks tile, tile + pairs, ...; the problem
    // alternates along that walk, and each problem's tiles are numbered without gaps.
    int t;
    if (!interleave) {
      prob = tile >= tiles0;
      t = prob ? tile - tiles0 : tile;
    } else if (pairs & 1) {
      prob = tile & 1;
      t = tile >> 1;
    } else {
      const int blk = tile / pairs, r = tile - blk * pairs;
      prob = (r + blk) & 1;
      t = blk * (pairs >> 1) + (r >> 1);
    }
    const int pm = prob ? pm1 : pm0;
    m0 = (t % pm) * 2 * kBM + static_cast<int>(rank) * kBM;
    nb = t / pm;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], 1);
    for (int a = 0; a < 2; ++a) mbar_init(&tfull[a], 1), mbar_init(&tempty[a], 2 * kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the set-up above overlapped the previous kernel; its results are visible now
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      tma_prefetch_desc(&tm_a0);
      tma_prefetch_desc(&tm_b0);
      if (M1 > 0) tma_prefetch_desc(&tm_a1), tma_prefetch_desc(&tm_b1);
      const uint32_t full_leader = mapa_shared(smem_addr(full), 0);
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[Cfg::kStages];
      for (int s = 0; s < Cfg::kStages; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int tile = pair; ok && tile < tiles; tile += pairs) {
        int prob, m0, nb;
        decode(tile, prob, m0, nb);
        const CUtensorMap* ma = prob ? &tm_a1 : &tm_a0;
        const CUtensorMap* mw = prob ? &tm_b1 : &tm_b0;
        const int num_kb = prob ? num_kb1 : num_kb0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1, abort_flag, status, kErrGemmWait)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * Cfg::kStageBytes;
          const uint32_t bar = full_leader + static_cast<uint32_t>(stage * sizeof(uint64_t));
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::kStageBytes);
          const int n_base = nb * BN + static_cast<int>(rank) * (BN / 2);
          if constexpr ((MAJ & 1) != 0) {
            tma_load_2d_pair(sa, ma, bar, m0, kb * kBK);
            tma_load_2d_pair(sa + kMnBoxBytes, ma, bar, m0 + kMnBlock, kb * kBK);
          } else {
            tma_load_2d_pair(sa, ma, bar, kb * kBK, m0);
          }
          if constexpr ((MAJ & 2) != 0) {
            tma_load_2d_pair(sa + Cfg::kABytes, mw, bar, n_base, kb * kBK);
            tma_load_2d_pair(sa + Cfg::kABytes + kMnBoxBytes, mw, bar, n_base + kMnBlock, kb * kBK);
          } else {
            tma_load_2d_pair(sa + Cfg::kABytes, mw, bar, kb * kBK, n_base);
          }
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == Cfg::kStages) stage = 0, phase ^= 1;
        }
      }
      if (*abort_flag && leader) {
        // Give the copies already issued (both CTAs' bytes land on these barriers) a bounded
        // chance to land before the pair exits.
        int never = 0;
        for (int s = 0; s < Cfg::kStages; ++s)
          if (last_parity[s] >= 0)
            mbar_wait_cluster(&full[s], static_cast<uint32_t>(last_parity[s]), &never, status, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader)
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < tiles; tile += pairs) {
        if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1, abort_flag, status, kErrGemmWait)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        int prob, m0_unused, nb_unused;
        decode(tile, prob, m0_unused, nb_unused);
        const int num_kb = prob ? num_kb1 : num_kb0;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, abort_flag, status, kErrGemmWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
          // K step k: 32 bytes into each 128-byte line (K-major), or kUmmaK lines further (MN-major)
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {
            const uint64_t da = (MAJ & 1) ? sdesc_mnmajor_sw128(sa + k * kUmmaK * 128, kMnBoxBytes)
                                          : sdesc_kmajor_sw128(sa + k * 32);
            const uint64_t db = (MAJ & 2) ? sdesc_mnmajor_sw128(sb + k * kUmmaK * 128, kMnBoxBytes)
                                          : sdesc_kmajor_sw128(sb + k * 32);
            tc_mma_pair<KIND>(d_tmem, da, db, kIdesc, (kb != 0 || k != 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == Cfg::kStages) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull[acc], 0x3);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (*abort_flag) {
        // Wait (bounded) for every MMA issued so far before either CTA releases its TMEM.
        int never = 0;
        tc_commit_pair(drain);
        mbar_wait(drain, 0, &never, status, 0);
      }
    }
  } else {
    // ---------------- epilogue warps 2..: warp w reads TMEM lanes 32*(w%4) .. +31 of this CTA
    const int quarter = warp & 3;
    const int group = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_addr(tempty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < tiles; tile += pairs) {
      int prob, m0, nb;
      decode(tile, prob, m0, nb);
      bool ok = mbar_wait_cluster(&tfull[acc], acc_phase, abort_flag, status, kErrGemmWait);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      EpiArgs ep = prob ? ep1 : ep0;
      gemm_epilogue<TE, BN, EPI, (KIND == kKindF8 || KIND == kKindF8E5M2)>(group, taddr, m0 + row, nb * BN, prob ? M1 : M0, N, ep);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_leader + static_cast<uint32_t>(acc * sizeof(uint64_t)));
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }

  __syncthreads();
  cluster_sync();  // no MMA, copy or remote arrival of the pair is still outstanding
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

// Host side: 256 x BN pair tiles; N % BN == 0 and no split K.  The grid is as many pairs as can
// be resident at once (every pair walks its share of the tile list).  MAJ as for the kernel.
template <int KIND, int BN, int EPI, int MAJ>
cudaError_t run_gemm_pair(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  using Cfg = PairCfg<BN>;
  constexpr int kElt = KindTraits<KIND>::kEltBytes;
  constexpr int kBK = 128 / kElt;
  if (p.N % BN != 0) return cudaErrorInvalidValue;
  const CUtensorMapDataType dt = KindTraits<KIND>::kMapType;
  const bool two = p.M1 > 0;
  const int K1 = two && p.K1 > 0 ? p.K1 : p.K;  // the second problem's K
  if (K1 < 1) return cudaErrorInvalidValue;
  CUtensorMap ta0, tb0, ta1, tb1;
  const uint64_t stride[1] = {static_cast<uint64_t>(p.K) * kElt};
  const uint64_t stride1[1] = {static_cast<uint64_t>(K1) * kElt};
  const uint32_t box_a[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
  const uint32_t box_b[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(BN / 2)};
  const uint64_t da0[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
  const uint64_t db[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
  const uint64_t da1[2] = {static_cast<uint64_t>(K1), static_cast<uint64_t>(two ? p.M1 : p.M)};
  const uint64_t db1[2] = {static_cast<uint64_t>(K1), static_cast<uint64_t>(p.N)};
  if constexpr (MAJ != 0) {
    // transposed operands: [K, M] and [K, N] tensors read in (64 MN x kBK k) boxes
    if ((p.a_mn && (p.M % 8 != 0 || (two && p.M1 % 8 != 0)))) return cudaErrorInvalidValue;
    const uint32_t box_mn[2] = {128u / kElt, static_cast<uint32_t>(kBK)};
    auto encode_pair = [&](CUtensorMap* ta, CUtensorMap* tb, const void* A, const void* W, int M, int K) {
      const uint64_t dak[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
      const uint64_t dbk[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(p.N)};
      const uint64_t sk[1] = {static_cast<uint64_t>(K) * kElt};
      const uint64_t dat[2] = {static_cast<uint64_t>(M), static_cast<uint64_t>(K)};
      const uint64_t dbt[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(K)};
      const uint64_t sat[1] = {static_cast<uint64_t>(M) * kElt};
      const uint64_t sbt[1] = {static_cast<uint64_t>(p.N) * kElt};
      const bool ok_a = (MAJ & 1) ? encode_tmap(ta, dt, 2, A, dat, sat, box_mn, CU_TENSOR_MAP_SWIZZLE_128B)
                                  : encode_tmap(ta, dt, 2, A, dak, sk, box_a, CU_TENSOR_MAP_SWIZZLE_128B);
      const bool ok_b = (MAJ & 2) ? encode_tmap(tb, dt, 2, W, dbt, sbt, box_mn, CU_TENSOR_MAP_SWIZZLE_128B)
                                  : encode_tmap(tb, dt, 2, W, dbk, sk, box_b, CU_TENSOR_MAP_SWIZZLE_128B);
      return ok_a && ok_b;
    };
    if (!encode_pair(&ta0, &tb0, p.A, p.W, p.M, p.K)) return cudaErrorInvalidValue;
    if (two) {
      if (!encode_pair(&ta1, &tb1, p.A1, p.W1, p.M1, K1)) return cudaErrorInvalidValue;
    } else {
      ta1 = ta0, tb1 = tb0;
    }
  } else if (!encode_tmap(&ta0, dt, 2, p.A, da0, stride, box_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !encode_tmap(&tb0, dt, 2, p.W, db, stride, box_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !encode_tmap(&ta1, dt, 2, two ? p.A1 : p.A, da1, two ? stride1 : stride, box_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !encode_tmap(&tb1, dt, 2, two ? p.W1 : p.W, two ? db1 : db, two ? stride1 : stride, box_b,
                          CU_TENSOR_MAP_SWIZZLE_128B)) {
    return cudaErrorInvalidValue;
  }
  auto kern = gemm_pair_kernel<KIND, BN, EPI, MAJ>;
  static int configured_device = -1;
  static int max_pairs = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(gemm_threads<EPI>(), 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2, attr.val.clusterDim.y = 1, attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_pairs = n;
    configured_device = dev;
  }
  const int num_n = p.N / BN;
  const int tiles0 = (p.M + 2 * kBM - 1) / (2 * kBM) * num_n;
  const int tiles1 = two ? (p.M1 + 2 * kBM - 1) / (2 * kBM) * num_n : 0;
  const int tiles = tiles0 + tiles1;
  const int interleave = p.interleave && two && tiles0 == tiles1 ? 1 : 0;
  if (tiles == 0) return cudaSuccess;
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  {
    const cudaError_t e_ = launch_pdl(kern, dim3(2 * pairs), dim3(gemm_threads<EPI>()), Cfg::kSmemBytes, stream,
                                        ta0, tb0, ta1, tb1, p.M, two ? p.M1 : 0, p.N, p.K, K1, interleave, p.ep,
                                        two ? p.ep1 : p.ep, status);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
