// gemm_blockwise.cu -- the blockwise FP8 recipe of the block linears: current per-tile scaling
// of both operands and a GEMM that applies each K slice's two scales as it accumulates.
//
// "FP8 training for Flux models", §Configuration › FP8 model configuration offers
// `fp8_recipe: "blockwise"` and prints the name only.  The reading taken (the same as the
// oracle's): every tile gets its own scale s = 448 / amax(tile) (1 for a tile of zeros) and is
// cast to E4M3 as Q(x s) (round to nearest even, saturating); activations [M, K] in 1 x 128
// tiles, weights [N, K] in 128 x 128 tiles; the linear is
//   y[m, n] = sum over 128-wide K slices j of  (Q_j(x) Q_j(W)^T)[m, n] / (s_x[m, j] s_w[n / 128, j]) + b[n].
//
// The casts: one warp per activation tile (four elements per lane), one 256-thread block per
// weight tile; the scale is the float32 quotient 448 / amax and the product x * s is float32, so
// a float32 emulation of the cast reproduces every code.  Scales are stored s_x [K/128, M] (a
// K slice's scales of consecutive rows adjacent) and s_w [N/128, K/128].
//
// The GEMM: one CTA per 128 x 128 output tile.  The MMA warp runs each 128-wide K slice (four
// kind::f8f6f4 MMAs of K = 32) into one of two TMEM buffers of 128 columns; eight promotion warps
// (a row and 64 columns per thread) take the slice out of TMEM as soon as it is complete, multiply
// it by 1 / (s_x s_w) and add it to float32 registers, while the tensor cores fill the other buffer.
// After the last slice the same warps add the bias and store bf16 rows.  Every wait is bounded
// (common.cuh).
#include "gemm_kernel.cuh"

namespace mmdit {
namespace {

constexpr int kBwTile = 128;             // M, N and K extent of a tile (K: 128 E4M3 = 128 bytes)
constexpr int kBwStages = 4;
constexpr int kBwStageBytes = 2 * kBwTile * kBwTile;  // A and B slices, 16 KB each
constexpr int kBwThreads = 64 + 256;     // producer, MMA, 8 promotion warps
constexpr int kBwSmem = kBwStages * kBwStageBytes + 256 + 1024;
constexpr uint32_t kBwTmemCols = 256;
constexpr uint32_t kBwIdesc = make_idesc<kKindF8>(kBwTile, kBwTile);

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct BwBarriers {
  uint64_t full[kBwStages];
  uint64_t empty[kBwStages];
  uint64_t pfull[2];   // a K slice's product in TMEM buffer b
  uint64_t pempty[2];  // buffer b read out (8 warp arrivals)
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

// EPI: the epilogue applied to the promoted sums (kEpiBias, kEpiQkv, kEpiGelu, kEpiGateResid, as
// for the other GEMMs).  Two problems of the same N and K (the image and text streams) share a
// launch: blockIdx.x enumerates problem 0's row tiles, then problem 1's.  Per problem, ep.bw_sx
// holds s_x [K/128, M] and ep.bw_sw s_w [N/128, K/128].
template <int EPI>
__global__ void __launch_bounds__(kBwThreads, 1)
    gemm_blockwise_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_b0,
                          const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_b1,
                          int M0, int M1, int N, int K, const __grid_constant__ EpiArgs ep0,
                          const __grid_constant__ EpiArgs ep1, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  BwBarriers* sb = reinterpret_cast<BwBarriers*>(smem + kBwStages * kBwStageBytes);
  volatile int* abort_flag = &sb->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles0 = (M0 + kBwTile - 1) / kBwTile;
  const int prob = static_cast<int>(blockIdx.x) >= tiles0;
  const int M = prob ? M1 : M0;
  const int m0 = (prob ? static_cast<int>(blockIdx.x) - tiles0 : static_cast<int>(blockIdx.x)) * kBwTile;
  const int nb = blockIdx.y, n0 = nb * kBwTile;
  const int num_kb = K / kBwTile;
  const CUtensorMap* tm_a = prob ? &tm_a1 : &tm_a0;
  const CUtensorMap* tm_b = prob ? &tm_b1 : &tm_b0;
  const EpiArgs& ep = prob ? ep1 : ep0;
  const float* __restrict__ sx = ep.bw_sx;
  const float* __restrict__ sw = ep.bw_sw;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBwStages; ++s) mbar_init(&sb->full[s], 1), mbar_init(&sb->empty[s], 1);
    for (int b = 0; b < 2; ++b) mbar_init(&sb->pfull[b], 1), mbar_init(&sb->pempty[b], 8);
    mbar_init(&sb->drain, 1);
    sb->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sb->tmem_slot, kBwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tmem_slot;
  pdl_wait();

  auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort_flag, status, kErrGemmWait); };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(tm_a);
      tma_prefetch_desc(tm_b);
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kBwStages;
        if (!wait(&sb->empty[s], (static_cast<uint32_t>(kb / kBwStages) & 1u) ^ 1u)) break;
        uint8_t* st = smem + s * kBwStageBytes;
        mbar_arrive_expect_tx(&sb->full[s], kBwStageBytes);
        tma_load_2d(st, tm_a, &sb->full[s], kb * kBwTile, m0);
        tma_load_2d(st + kBwTile * kBwTile, tm_b, &sb->full[s], kb * kBwTile, n0);
        issued = kb + 1;
      }
      if (*abort_flag) {
        // give the copies already issued a bounded chance to land before the CTA exits
        int never = 0;
        for (int t = issued - kBwStages > 0 ? issued - kBwStages : 0; t < issued; ++t)
          mbar_wait(&sb->full[t % kBwStages], static_cast<uint32_t>(t / kBwStages) & 1u, &never, status, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: K slice kb into TMEM buffer kb & 1
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kBwStages, b = kb & 1;
        if (!wait(&sb->full[s], static_cast<uint32_t>(kb / kBwStages) & 1u)) break;
        if (!wait(&sb->pempty[b], (static_cast<uint32_t>(kb >> 1) & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t sa = smem_addr(smem + s * kBwStageBytes);
        const uint32_t sbb = sa + kBwTile * kBwTile;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma<kKindF8>(tmem + static_cast<uint32_t>(b * kBwTile), sdesc_kmajor_sw128(sa + k * 32),
                          sdesc_kmajor_sw128(sbb + k * 32), kBwIdesc, k > 0 ? 1u : 0u);
        tc_commit(&sb->empty[s]);
        tc_commit(&sb->pfull[b]);
      }
      if (*abort_flag) {
        int never = 0;
        tc_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, &never, status, 0);
      }
    }
  } else {
    // ---------------- promotion: warp w reads TMEM lanes 32 (w % 4) .. (its row) and columns
    // [64 g, 64 g + 64) of each buffer, g its warp group
    const int quarter = warp & 3, g = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int m = m0 + row;
    const bool row_ok = m < M;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int b = kb & 1;
      // this slice's factor 1 / (s_x[m, kb] s_w[nb, kb]), fetched before the wait
      const float f = row_ok ? 1.f / (__ldg(sx + static_cast<size_t>(kb) * M + m) *
                                      __ldg(sw + static_cast<size_t>(nb) * num_kb + kb))
                             : 0.f;
      ok = wait(&sb->pfull[b], static_cast<uint32_t>(kb >> 1) & 1u);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t p0[32], p1[32];
      const uint32_t t = tmem + static_cast<uint32_t>(b * kBwTile + g * 64) + lane_off;
      tmem_ld32(t, p0);
      tmem_ld32(t + 32u, p1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->pempty[b]);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        acc[i] = fmaf(__uint_as_float(p0[i]), f, acc[i]);
        acc[32 + i] = fmaf(__uint_as_float(p1[i]), f, acc[32 + i]);
      }
    }
    // the promoted sums back into TMEM (buffer 0: every product has been read out of it), then
    // the epilogue every GEMM shares reads them there
    ok = ok && !*abort_flag;
    if (ok) {
      uint32_t w0[32], w1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w0[i] = __float_as_uint(acc[i]), w1[i] = __float_as_uint(acc[32 + i]);
      const uint32_t t = tmem + static_cast<uint32_t>(g * 64) + lane_off;
      tmem_st32(t, w0);
      tmem_st32(t + 32u, w1);
      tmem_st_wait();
      tc_fence_before();
    }
    // the eight promotion warps (an epilogue group may read columns another group wrote)
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok && g < EpiGroups<EPI>::value) {
      tc_fence_after();
      gemm_epilogue<__nv_bfloat16, kBwTile, EPI, false>(g, tmem + lane_off, m, n0, M, N, ep);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwTmemCols);
  }
}

// Activation casts: one warp per (row, 128-wide tile), four elements per lane.
__global__ void blockwise_cast_act_kernel(const __nv_bfloat16* __restrict__ x, int M, int K, uint8_t* __restrict__ q,
                                          float* __restrict__ s_out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int tiles = K / kBwTile;
  const int64_t total = static_cast<int64_t>(M) * tiles;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total;
       w += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int m = static_cast<int>(w / tiles), j = static_cast<int>(w - static_cast<int64_t>(m) * tiles);
    const size_t off = static_cast<size_t>(m) * K + j * kBwTile + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + off);
    const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = a > 0.f ? 448.f / a : 1.f;
    *reinterpret_cast<uint32_t*>(q + off) = e4m3x2(v[0] * s, v[1] * s) | (e4m3x2(v[2] * s, v[3] * s) << 16);
    if (lane == 0) s_out[static_cast<size_t>(j) * M + m] = s;
  }
}

// Weight casts: one 256-thread block per 128 x 128 tile (a thread: half a row of 64 elements).
__global__ void __launch_bounds__(256) blockwise_cast_weight_kernel(const __nv_bfloat16* __restrict__ w, int N, int K,
                                                                    uint8_t* __restrict__ q, float* __restrict__ s_out) {
  pdl_wait();
  __shared__ float red[8];
  const int tiles_k = K / kBwTile;
  const int ti = blockIdx.x / tiles_k, tj = blockIdx.x - ti * tiles_k;
  const int r = ti * kBwTile + (threadIdx.x >> 1), c = tj * kBwTile + (threadIdx.x & 1) * 64;
  const __nv_bfloat16* src = w + static_cast<size_t>(r) * K + c;
  float v[64];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = *reinterpret_cast<const uint4*>(src + 8 * i);
    v[8 * i + 0] = bf16_lo(u.x), v[8 * i + 1] = bf16_hi(u.x), v[8 * i + 2] = bf16_lo(u.y), v[8 * i + 3] = bf16_hi(u.y);
    v[8 * i + 4] = bf16_lo(u.z), v[8 * i + 5] = bf16_hi(u.z), v[8 * i + 6] = bf16_lo(u.w), v[8 * i + 7] = bf16_hi(u.w);
  }
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) a = fmaxf(a, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  const float s = a > 0.f ? 448.f / a : 1.f;
  uint8_t* dst = q + static_cast<size_t>(r) * K + c;
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(dst + 8 * i) = e4m3x8(v + 8 * i, s);
  if (threadIdx.x == 0) s_out[blockIdx.x] = s;  // [N/128, K/128]: blockIdx.x = ti * tiles_k + tj
}




// The blockwise GEMM for a GemmProblem whose per-problem ep.bw_sx / ep.bw_sw are set: A, W (and
// A1, W1) are E4M3 codes [M, K], [N, K]; N % 128 == 0, K % 128 == 0.
template <int EPI>
cudaError_t run_gemm_blockwise(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  const bool two = p.M1 > 0;
  if (p.N % kBwTile != 0 || p.K % kBwTile != 0 || p.K < kBwTile || (two && p.K1 > 0 && p.K1 != p.K))
    return cudaErrorInvalidValue;
  if (!p.ep.bw_sx || !p.ep.bw_sw || (two && (!p.ep1.bw_sx || !p.ep1.bw_sw))) return cudaErrorInvalidValue;
  const uint64_t k = static_cast<uint64_t>(p.K), n = static_cast<uint64_t>(p.N);
  const uint64_t stride[1] = {k};
  const uint32_t box[2] = {static_cast<uint32_t>(kBwTile), static_cast<uint32_t>(kBwTile)};
  CUtensorMap ta0, tb0, ta1, tb1;
  const uint64_t da0[2] = {k, static_cast<uint64_t>(p.M)}, db[2] = {k, n};
  const uint64_t da1[2] = {k, static_cast<uint64_t>(two ? p.M1 : p.M)};
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_tmap(&ta0, U8, 2, p.A, da0, stride, box, SW) || !encode_tmap(&tb0, U8, 2, p.W, db, stride, box, SW) ||
      !encode_tmap(&ta1, U8, 2, two ? p.A1 : p.A, da1, stride, box, SW) ||
      !encode_tmap(&tb1, U8, 2, two ? p.W1 : p.W, db, stride, box, SW))
    return cudaErrorInvalidValue;
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_blockwise_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwSmem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const int tiles_m = (p.M + kBwTile - 1) / kBwTile + (two ? (p.M1 + kBwTile - 1) / kBwTile : 0);
  if (tiles_m == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(tiles_m), static_cast<unsigned>(p.N / kBwTile));
  cudaError_t e = launch_pdl(gemm_blockwise_kernel<EPI>, grid, dim3(kBwThreads), kBwSmem, stream, ta0, tb0, ta1, tb1,
                             p.M, two ? p.M1 : 0, p.N, p.K, p.ep, two ? p.ep1 : p.ep, status);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace

size_t blockwise_linear_scratch(int M, int N, int K) {
  const size_t m = static_cast<size_t>(M), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
  return round256(m * k) + round256(n * k) + round256((k / kBwTile) * m * 4) +
         round256((n / kBwTile) * (k / kBwTile) * 4);
}

cudaError_t launch_blockwise_cast_act(const __nv_bfloat16* x, int M, int K, uint8_t* q, float* s, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (M < 0 || K % kBwTile != 0) return cudaErrorInvalidValue;
  const int64_t warps = static_cast<int64_t>(M) * (K / kBwTile);
  int64_t blocks = (warps + 7) / 8;
  if (blocks > num_sms() * 16) blocks = num_sms() * 16;
  cudaError_t e = launch_pdl(blockwise_cast_act_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, x, M,
                             K, q, s);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_blockwise_cast_weight(const __nv_bfloat16* w, int N, int K, uint8_t* q, float* s, cudaStream_t stream) {
  if (N % kBwTile != 0 || K % kBwTile != 0) return cudaErrorInvalidValue;
  const unsigned tiles = static_cast<unsigned>((N / kBwTile) * (K / kBwTile));
  if (tiles == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(blockwise_cast_weight_kernel, dim3(tiles), dim3(256), 0, stream, w, N, K, q, s);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_gemm_blockwise(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  switch (p.epi) {
    case kEpiBias: return run_gemm_blockwise<kEpiBias>(p, status, stream);
    case kEpiQkv: return run_gemm_blockwise<kEpiQkv>(p, status, stream);
    case kEpiGelu: return run_gemm_blockwise<kEpiGelu>(p, status, stream);
    case kEpiGateResid: return run_gemm_blockwise<kEpiGateResid>(p, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_blockwise_linear(int M, int N, int K, const __nv_bfloat16* x, const __nv_bfloat16* w,
                                    const __nv_bfloat16* bias, __nv_bfloat16* y, void* scratch, uint32_t* status,
                                    cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (M < 0 || N % kBwTile != 0 || K % kBwTile != 0 || N == 0 || K == 0) return cudaErrorInvalidValue;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  const size_t m = static_cast<size_t>(M), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
  uint8_t* xq = base;
  uint8_t* wq = xq + round256(m * k);
  float* sx = reinterpret_cast<float*>(wq + round256(n * k));
  float* sw = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sx) + round256((k / kBwTile) * m * 4));
  cudaError_t e = launch_blockwise_cast_act(x, M, K, xq, sx, stream);
  if (e != cudaSuccess) return e;
  if ((e = launch_blockwise_cast_weight(w, N, K, wq, sw, stream)) != cudaSuccess) return e;
  GemmProblem g;
  g.act = 2, g.epi = kEpiBias, g.M = M, g.N = N, g.K = K, g.A = xq, g.W = wq;
  g.ep.bias = bias, g.ep.out = y, g.ep.bw_sx = sx, g.ep.bw_sw = sw;
  return launch_gemm_blockwise(g, status, stream);
}

}  // namespace mmdit
