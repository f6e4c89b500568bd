// mxfp8.cu -- the MXFP8 recipe of the block linears: E4M3 elements that share one power-of-two
// (E8M0) scale per 32 consecutive elements along the contraction dimension K.
//
// "FP8 training for Flux models", §Configuration › FP8 model configuration offers
// `fp8_recipe: "mxfp8"` and prints the name only.  The reading taken (the same as the oracle's)
// is the OCP Microscaling formats specification v1.0 with E4M3 elements: a block's shared
// exponent is e = floor(log2 amax) - 8 (8 is the exponent of E4M3's largest normal,
// 448 = 1.75 * 2^8), clamped to [-127, 127], and -127 for a block of zeros; each element is
// stored as P = E4M3(v / 2^e) (round to nearest even, saturating at 448) and stands for P * 2^e.
//
// How the products run: a represented value P * 2^e has at most four significant bits, so bf16
// holds it exactly whenever its lowest bit is at or above 2^-133 (for every block whose largest
// magnitude is at least 2^-116).  The cast therefore writes, beside the codes and the E8M0 scale
// codes, the represented values as bf16, and the linear is the bf16 tensor-core GEMM of those
// values: every product is exact and the sums are fp32, so the result is the MX product up to
// the order of the fp32 additions.  The block-scaled MMA, which would read the codes and scales
// directly at the FP8 rate, is not used; the recipe runs at the bf16 rate.
//
// The cast: one thread per 8 consecutive elements (one 16-byte load), four neighbouring lanes per
// 32-element block, the block maximum by two shuffles.  e comes from the exponent field of the
// float32 maximum (exact, no logarithm); 1 / 2^e and 2^e are built from exponent fields, the
// latter as two normal factors so that a subnormal result is formed exactly.
#include "common.cuh"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kMxBlock = 32;

// two E4M3 codes (low byte first) -> two fp16 values (exact: E4M3 is a subset of fp16)
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t codes) {
  uint32_t h2;
  const uint16_t c = static_cast<uint16_t>(codes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

__device__ __forceinline__ float pow2f(int k) {  // 2^k for k in [-126, 127]
  return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

__global__ void __launch_bounds__(256) mx_cast_kernel(MxJobs jobs) {
  pdl_wait();
  const MxJob jb = jobs.j[blockIdx.y];
  const int64_t units = jb.rows * (jb.K / 8);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  // whole warps walk the units so that the shuffles always see all 32 lanes
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < units;
       base += stride) {
    const int64_t u = base + lane;
    const bool act = u < units;
    float v[8];
    if (act) {
      const uint4 raw = *reinterpret_cast<const uint4*>(jb.src + u * 8);
      v[0] = bf16_lo(raw.x), v[1] = bf16_hi(raw.x), v[2] = bf16_lo(raw.y), v[3] = bf16_hi(raw.y);
      v[4] = bf16_lo(raw.z), v[5] = bf16_hi(raw.z), v[6] = bf16_lo(raw.w), v[7] = bf16_hi(raw.w);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    if (!act) continue;
    // floor(log2 a) is the unbiased exponent of a normal a; a zero or subnormal a (below 2^-126)
    // clamps to -127.  For bf16 inputs e <= 120, so 1 / 2^e = 2^-e is a normal float.
    const int eb = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu);
    const int e = eb == 0 ? -127 : min(127, max(-127, eb - 127 - 8));
    const float inv = pow2f(-e);
    uint2 q;
    q.x = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
    q.y = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
    // the represented values P * 2^e, as (P * 2^(e/2)) * 2^(e - e/2): both factors normal
    const float s1 = pow2f(e / 2), s2 = pow2f(e - e / 2);
    float d[8];
    const uint32_t w4[4] = {q.x & 0xFFFFu, q.x >> 16, q.y & 0xFFFFu, q.y >> 16};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = e4m3x2_decode(w4[i]);
      d[2 * i] = (p.x * s1) * s2, d[2 * i + 1] = (p.y * s1) * s2;
    }
    uint4 o;
    o.x = pack_bf16x2(d[0], d[1]), o.y = pack_bf16x2(d[2], d[3]);
    o.z = pack_bf16x2(d[4], d[5]), o.w = pack_bf16x2(d[6], d[7]);
    *reinterpret_cast<uint4*>(jb.deq + u * 8) = o;
    if (jb.codes) *reinterpret_cast<uint2*>(jb.codes + u * 8) = q;
    if (jb.scales && (lane & 3) == 0) jb.scales[u >> 2] = static_cast<uint8_t>(e + 127);
  }
}

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

cudaError_t launch_mx_cast(const MxJob* jobs, int n, cudaStream_t stream) {
  if (n < 0 || n > kMxMaxJobs) return cudaErrorInvalidValue;
  MxJobs js;
  js.n = n;
  int64_t most = 0;
  for (int i = 0; i < n; ++i) {
    const MxJob& j = jobs[i];
    if (j.rows < 0 || j.K < 0 || j.K % kMxBlock != 0 || (j.rows * j.K > 0 && (!j.src || !j.deq)))
      return cudaErrorInvalidValue;
    js.j[i] = j;
    const int64_t units = j.rows * (j.K / 8);
    if (units > most) most = units;
  }
  if (n == 0 || most == 0) return cudaSuccess;
  // a few waves of 256-thread blocks per job; the loop strides over the rest
  const int64_t blocks = (most + 255) / 256 < 152 * 8 ? (most + 255) / 256 : 152 * 8;
  cudaError_t e = launch_pdl(mx_cast_kernel, dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(n)), dim3(256),
                             0, stream, js);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaSuccess;
}

size_t mx_linear_scratch(int M, int N, int K) {
  const size_t m = M > 0 ? M : 0, n = N > 0 ? N : 0, k = K > 0 ? K : 0;
  return round256(m * k * 2) + round256(n * k * 2) + round256(m * k) + round256(n * k) + round256(m * (k / kMxBlock)) +
         round256(n * (k / kMxBlock));
}

cudaError_t launch_mx_linear(int M, int N, int K, const __nv_bfloat16* x, const __nv_bfloat16* w,
                             const __nv_bfloat16* bias, __nv_bfloat16* y, void* scratch, uint32_t* status,
                             cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (M < 0 || N <= 0 || K <= 0 || K % kMxBlock != 0) return cudaErrorInvalidValue;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  const size_t m = static_cast<size_t>(M), n = static_cast<size_t>(N), k = static_cast<size_t>(K);
  __nv_bfloat16* xd = reinterpret_cast<__nv_bfloat16*>(base);
  __nv_bfloat16* wd = reinterpret_cast<__nv_bfloat16*>(base + round256(m * k * 2));
  uint8_t* xq = reinterpret_cast<uint8_t*>(wd) + round256(n * k * 2);
  uint8_t* wq = xq + round256(m * k);
  uint8_t* xs = wq + round256(n * k);
  uint8_t* wsc = xs + round256(m * (k / kMxBlock));
  const MxJob jobs[2] = {{x, xd, xq, xs, static_cast<int64_t>(M), K}, {w, wd, wq, wsc, static_cast<int64_t>(N), K}};
  cudaError_t e = launch_mx_cast(jobs, 2, stream);
  if (e != cudaSuccess) return e;
  GemmProblem g;
  g.act = 1, g.epi = kEpiBias, g.M = M, g.N = N, g.K = K, g.A = xd, g.W = wd;
  g.ep.bias = bias, g.ep.out = y;
  return launch_gemm(g, status, stream);
}

}  // namespace mmdit
