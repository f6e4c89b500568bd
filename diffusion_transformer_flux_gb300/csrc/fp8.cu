// fp8.cu -- E4M3 casts with per-tensor delayed scaling ("FP8 training for Flux models",
// §Configuration, FP8 model configuration: E4M3, amax history 1024, most_recent, margin 0).
//
//   quantize_e4m3_kernel   bf16 -> E4M3 codes of x * scale, recording max |x| (one launch casts
//                          up to eight tensors, e.g. every weight of a block); a job without a
//                          destination records max |x| only (the first pass of current scaling)
//   amax_reset_kernel      zeroes the history slot a call is about to record into
//   scale_update_kernel    scale = 448 / amax / 2^margin, amax of that slot (most_recent) or the
//                          largest in the history (max), where amax > 0
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kQThreads = 256;
constexpr int kQVec = 16;                        // elements per thread and round (32 bytes in)
constexpr int kQRounds = 4;                      // rounds per tile, loads issued together
constexpr int64_t kQTile = static_cast<int64_t>(kQThreads) * kQVec * kQRounds;  // 16384

struct QuantJobs {
  QuantJob j[kQuantMaxJobs];
  int64_t tile_start[kQuantMaxJobs + 1];  // first tile of each job; tile_start[njobs] = total
  int njobs;
};

// Every tile lies inside one job; a thread converts kQRounds groups of 16 elements.
__global__ void __launch_bounds__(kQThreads) quantize_e4m3_kernel(const __grid_constant__ QuantJobs jobs,
                                                                  int64_t tiles) {
  pdl_wait();  // the previous kernel's results are visible from here on
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    int j = 0;
    while (j + 1 < jobs.njobs && t >= jobs.tile_start[j + 1]) ++j;
    const QuantJob& q = jobs.j[j];
    const int64_t base = (t - jobs.tile_start[j]) * kQTile;
    const float s = q.dst ? __ldg(q.scale) : 1.f;
    uint4 raw[kQRounds][2];
#pragma unroll
    for (int r = 0; r < kQRounds; ++r) {
      const int64_t i = base + (static_cast<int64_t>(r) * kQThreads + threadIdx.x) * kQVec;
      if (i < q.n) {
        const uint4* src = reinterpret_cast<const uint4*>(q.src + i);
        raw[r][0] = __ldg(src);
        raw[r][1] = __ldg(src + 1);
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int r = 0; r < kQRounds; ++r) {
      const int64_t i = base + (static_cast<int64_t>(r) * kQThreads + threadIdx.x) * kQVec;
      if (i < q.n) {
        float v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 u = raw[r][h];
          v[8 * h + 0] = bf16_lo(u.x), v[8 * h + 1] = bf16_hi(u.x);
          v[8 * h + 2] = bf16_lo(u.y), v[8 * h + 3] = bf16_hi(u.y);
          v[8 * h + 4] = bf16_lo(u.z), v[8 * h + 5] = bf16_hi(u.z);
          v[8 * h + 6] = bf16_lo(u.w), v[8 * h + 7] = bf16_hi(u.w);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) mx = fmaxf(mx, fabsf(v[e]));
        if (q.dst) {  // (a job without a destination records its amax only)
          const uint2 a = q.e5m2 ? e5m2x8(v, s) : e4m3x8(v, s), b = q.e5m2 ? e5m2x8(v + 8, s) : e4m3x8(v + 8, s);
          *reinterpret_cast<uint4*>(q.dst + i) = make_uint4(a.x, a.y, b.x, b.y);
        }
      }
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0 && mx > 0.f) atomic_max_nonneg(q.amax, mx);
  }
}

// out [C, ld_out] = in [R, C]^T for bytes through a 64 x 64 shared tile (one byte per thread
// and element); the padding columns R .. ld_out - 1 are written as zero codes.
__global__ void transpose_u8_kernel(const uint8_t* __restrict__ in, int R, int C, int ld_out,
                                    uint8_t* __restrict__ out) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ uint8_t tile[64][65];
  const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  for (int i = threadIdx.y; i < 64; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < R && c < C) ? in[static_cast<size_t>(r) * C + c] : 0;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 64; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < ld_out) out[static_cast<size_t>(c) * ld_out + r] = tile[threadIdx.x][i];
  }
}

__global__ void amax_reset_kernel(float* hist, int hist_len, int n, int pos) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) hist[static_cast<size_t>(i) * hist_len + pos] = 0.f;
}

// One warp per tensor: lane 0 reads the most recent entry (algo 0), or the warp takes the
// largest entry of the tensor's history row (algo 1).
__global__ void scale_update_kernel(const float* hist, float* scale, int hist_len, int n, int pos,
                                    int margin, int algo) {
  pdl_wait();  // the previous kernel's results are visible from here on
  const int i = blockIdx.x;
  if (i >= n) return;
  const float* row = hist + static_cast<size_t>(i) * hist_len;
  float a;
  if (algo == 1) {
    a = 0.f;
    for (int j = threadIdx.x; j < hist_len; j += 32) a = fmaxf(a, row[j]);
    a = warp_max(a);
  } else {
    a = row[pos];
  }
  if (threadIdx.x == 0 && a > 0.f && isfinite(a)) scale[i] = ldexpf(448.f / a, -margin);
}

}  // namespace

cudaError_t launch_quantize_e4m3(const QuantJob* jobs, int njobs, cudaStream_t stream) {
  if (njobs < 0 || njobs > kQuantMaxJobs) return cudaErrorInvalidValue;
  QuantJobs q{};
  int64_t tiles = 0;
  int k = 0;
  for (int i = 0; i < njobs; ++i) {
    if (jobs[i].n <= 0) continue;
    if (jobs[i].n % kQVec != 0) return cudaErrorInvalidValue;
    q.j[k] = jobs[i];
    q.tile_start[k] = tiles;
    tiles += (jobs[i].n + kQTile - 1) / kQTile;
    ++k;
  }
  q.njobs = k;
  q.tile_start[k] = tiles;
  if (tiles == 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  {
    const cudaError_t e_ = launch_pdl(quantize_e4m3_kernel, dim3(grid), dim3(kQThreads), 0, stream, q, tiles);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_transpose_u8(const uint8_t* in, int R, int C, int ld_out, uint8_t* out, cudaStream_t stream) {
  if (C == 0 || ld_out == 0) return cudaSuccess;
  if (ld_out < R) return cudaErrorInvalidValue;
  const dim3 grid((ld_out + 63) / 64, (C + 63) / 64), block(64, 4);
  {
    const cudaError_t e_ = launch_pdl(transpose_u8_kernel, grid, block, 0, stream, in, R, C, ld_out, out);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_amax_reset(float* hist, int hist_len, int n, int pos, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  {
    const cudaError_t e_ = launch_pdl(amax_reset_kernel, dim3((n + 127) / 128), dim3(128), 0, stream, hist, hist_len, n, pos);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_scale_update(const float* hist, float* scale, int hist_len, int n, int pos,
                                int margin, int algo, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  {
    const cudaError_t e_ = launch_pdl(scale_update_kernel, dim3(n), dim3(32), 0, stream, hist, scale,
                                      hist_len, n, pos, margin, algo);
    if (e_ != cudaSuccess) return e_;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mmdit
