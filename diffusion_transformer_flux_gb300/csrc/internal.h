// internal.h -- interfaces between the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mmdit {

// Epilogues of the tensor-core GEMM  C[M, N] = A[M, K] * W[N, K]^T (fp32 accumulation).
enum EpiKind : int {
  kEpiBias = 0,       // out[m, n] = acc + bias[n]
  kEpiGelu = 1,       // out[m, n] = GELU(acc + bias[n])
  kEpiGateResid = 2,  // out[m, n] = resid[m, n] + gate[b(m), n] * (acc + bias[n])
  kEpiQkv = 3,        // bias, per-head RMSNorm of q and k, RoPE, scatter to Q, K, Vt
  kEpiUnpatchify = 4, // pred[b, n, s] (fp32) = acc + bias[n], m = b * rows_per_batch + s
  kEpiPartial = 5,    // split-K: partial[split][m][n] (fp32) = acc over the split's K range
  kEpiGeluF8 = 6,     // out[m, n] (E4M3) = GELU(acc + bias[n]) * out_scale, amax recorded
  kEpiDGelu = 7       // out[m, n] = (acc + bias[n]) * GELU'(aux[m, n]) (a GELU's input gradient)
};

struct EpiArgs {
  const void* bias = nullptr;  // [N], activation type, may be null
  void* out = nullptr;         // [M, N] activation type (fp32 [B, N, rows_per_batch] for unpatchify)
  int out_f32 = 0;             // store `out` as fp32 whatever the operand type
  const void* resid = nullptr; // [M, N] (gated residual)
  int resid_f32 = 0;           // `resid` is fp32 whatever the operand type
  const float* gate = nullptr; // gate for batch b at gate + b * gate_bstride
  int64_t gate_bstride = 0;
  int rows_per_batch = 1;      // m -> (b = m / rows_per_batch, s = m % rows_per_batch)
  int gelu_tanh = 0;
  // kEpiQkv, kEpiGelu, kEpiGateResid: when set, [M, N] (activation type) also receives the
  // product plus bias before the epilogue's norm, activation or gate (what a backward reads)
  void* pre = nullptr;
  const void* aux = nullptr;   // kEpiDGelu: [M, N] activation type, the GELU's input
  // QKV scatter
  const void* g_q = nullptr;   // [128] activation type
  const void* g_k = nullptr;
  const float* rope_cos = nullptr;  // [B, seq_joint, 64]
  const float* rope_sin = nullptr;
  __nv_bfloat16* q = nullptr;  // [B, H, seq_joint, 128]
  __nv_bfloat16* k = nullptr;
  __half* vt = nullptr;        // [B, H, 128, seq_pad] fp16 holding bf16-rounded values
  int seq_offset = 0;          // joint index of this stream's token 0
  int seq_joint = 0;
  int seq_pad = 0;
  int heads = 0;
  int hidden = 0;
  float rms_eps = 1e-6f;
  int rope_interleaved = 1;
  // E4M3 operands: the accumulator is first multiplied by 1 / (scale_a[0] * scale_w[0]), the
  // scales the operands were cast with
  const float* scale_a = nullptr;
  const float* scale_w = nullptr;
  // blockwise FP8 (gemm_blockwise.cu): per-tile scales s_x [K/128, M] and s_w [N/128, K/128]; the
  // GEMM divides each 128-wide K slice's product by them before the epilogue
  const float* bw_sx = nullptr;
  const float* bw_sw = nullptr;
  // kEpiGeluF8: `out` receives E4M3 codes of GELU(.) * out_scale[0]; out_amax[0] is raised to
  // the largest |GELU(.)| of the tile
  const float* out_scale = nullptr;
  float* out_amax = nullptr;
};

struct GemmProblem {
  int act = 1;           // 0 = fp32 operands (tf32 MMA), 1 = bf16, 2 = E4M3 (epilogue I/O bf16),
                         // 3 = E5M2 A with E4M3 B (kEpiBias only)
  int epi = kEpiBias;
  int M = 0, N = 0, K = 0;
  const void* A = nullptr;  // [M, K]
  const void* W = nullptr;  // [N, K]
  EpiArgs ep;
  int splits = 1;  // K split into this many ranges (kEpiPartial only), one work item each
  // Operands stored MN-major (bf16, kEpiBias, N % 256 == 0, no second problem): with a_mn, A is
  // held as A^T [K, M] (M contiguous, M % 8 == 0); with b_mn, W is held as W^T [K, N].
  int a_mn = 0, b_mn = 0;
  // optional second problem with the same N and epilogue kind, run in the same launch; its K is
  // K1 (pair kernel only; 0: the same K).  With interleave (pair kernel, equal tile counts) the
  // two problems' tiles alternate in the tile list instead of following one another.
  int M1 = 0;
  int K1 = 0;
  int interleave = 0;
  const void* A1 = nullptr;  // [M1, K]
  const void* W1 = nullptr;  // [N, K]
  EpiArgs ep1;
};

// Programmatic dependent launch within one library call.  pdl_begin_call() marks the start of
// a call on the calling thread; its first kernel then launches as an ordinary launch (it must
// wait for whatever the caller enqueued before it: copies, memsets, other libraries' kernels),
// and each later kernel of the call launches with programmatic stream serialization, so it may
// be scheduled while the call's previous kernel finishes.  Every kernel calls pdl_wait()
// (common.cuh) before it touches global memory, so results are those of ordinary launches.
void pdl_begin_call();
bool pdl_next_launch();  // false for the call's first launch, true afterwards

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_next_launch() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Device status word layout: the first 4 bytes of every workspace.
constexpr size_t kStatusBytes = 256;

// Launch accounting for diagnostics.
void count_launch(int n = 1);

// Records `msg` as the calling thread's last error (returned by mmdit_last_error) and returns
// `status`; for translation units other than the one holding the C ABI's bookkeeping.
int set_last_error(int status, const char* msg);

// Number of SMs of the current device.
int num_sms();

// Tensor-map encoding through the driver entry point (no link-time libcuda dependency).
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// gemm_bf16.cu / gemm_tf32.cu / gemm_fp8.cu
cudaError_t launch_gemm_bf16(const GemmProblem& p, uint32_t* status, cudaStream_t stream);
cudaError_t launch_gemm_tf32(const GemmProblem& p, uint32_t* status, cudaStream_t stream);
// E4M3 operands (K a multiple of 16, N a multiple of 128); epilogues kEpiBias, kEpiQkv,
// kEpiGateResid and kEpiGeluF8, with scale_a / scale_w set in every EpiArgs.
cudaError_t launch_gemm_fp8(const GemmProblem& p, uint32_t* status, cudaStream_t stream);
inline cudaError_t launch_gemm(const GemmProblem& p, uint32_t* status, cudaStream_t stream) {
  return p.act >= 2 ? launch_gemm_fp8(p, status, stream)
                    : (p.act == 1 ? launch_gemm_bf16(p, status, stream) : launch_gemm_tf32(p, status, stream));
}

// attention.cu: O = softmax(Q K^T / sqrt(128)) V per (b, h); rows [0, split) of each batch go
// to out0 ([B, split, H*128]), rows [split, S) to out1 ([B, S - split, H*128]).
struct AttnProblem {
  int act = 1;  // output type: 0 fp32, 1 bf16
  int batch = 0, heads = 0, seq = 0, seq_pad = 0, split = 0;
  const __nv_bfloat16* q = nullptr;   // [B, H, S, 128]
  const __nv_bfloat16* k = nullptr;   // [B, H, S, 128]
  const __half* vt = nullptr;         // [B, H, 128, seq_pad] fp16 (bf16-rounded values)
  void* out0 = nullptr;
  void* out1 = nullptr;
  // training forward: each row's log-sum-exp of the scaled scores in log2 units,
  // L = log2 sum_t exp2(q . k_t log2(e) / sqrt(d)), at lse[(b * H + h) * seq_pad + s]; or null
  float* lse = nullptr;
};
cudaError_t launch_attention(const AttnProblem& p, uint32_t* status, cudaStream_t stream);

// attention_fp8.cu: the joint attention on E4M3 operands (fp8_dot_product_attention): the launcher
// casts q, k (to q8, k8 [B, H, S, 128]) and v (to vt8 [B, H, 128, seq_pad], seq_pad a multiple of
// 16) with the given device scales, recording their amax into amax[0..1] (q, k), then
// O = E4M3(Pt 448) E4M3(v s_v) / (448 s_v) / rowsum(Pt), Pt = exp(S - rowmax), S from the casts.
struct AttnFp8Problem {
  int act = 1;  // output type: 0 fp32, 1 bf16
  int batch = 0, heads = 0, seq = 0, seq_pad = 0, split = 0;
  const __nv_bfloat16 *q = nullptr, *k = nullptr, *v = nullptr;  // [B, H, S, 128]
  uint8_t *q8 = nullptr, *k8 = nullptr, *vt8 = nullptr;           // cast codes (workspace)
  const float *scale_q = nullptr, *scale_k = nullptr, *scale_v = nullptr;
  float* amax = nullptr;  // [2]
  void* out0 = nullptr;
  void* out1 = nullptr;
};
cudaError_t launch_attention_fp8(const AttnFp8Problem& p, uint32_t* status, cudaStream_t stream);

// attention_bwd.cu: the joint attention's backward from the forward's log-sum-exp L and the
// pre-pass's D = rowsum(dO * O): dV = P^T dO, dS = P (dO V^T - D) / sqrt(d), dK = dS^T Q, dQ = dS K,
// P = exp2(q . k log2(e) / sqrt(d) - L).  dO (and so D and every output) carries the pre-pass's
// power-of-two gradient scale.
// gemm_blockwise.cu: the blockwise FP8 linear y = x W^T + b (bf16 x, W, b, y): per-tile E4M3 casts
// of x (1 x 128 tiles) and W (128 x 128 tiles) into `scratch` (blockwise_linear_scratch bytes),
// then the GEMM that scales each 128-wide K slice's product.  N % 128 == 0, K % 128 == 0.
size_t blockwise_linear_scratch(int M, int N, int K);
// The casts alone: x [M, K] -> codes q [M, K], scales s [K/128, M]; W [N, K] -> q [N, K], s [N/128, K/128].
cudaError_t launch_blockwise_cast_act(const __nv_bfloat16* x, int M, int K, uint8_t* q, float* s, cudaStream_t stream);
cudaError_t launch_blockwise_cast_weight(const __nv_bfloat16* w, int N, int K, uint8_t* q, float* s,
                                         cudaStream_t stream);
// The blockwise GEMM of a problem whose ep.bw_sx / ep.bw_sw (and ep1's) are set (E4M3 codes as A, W).
struct GemmProblem;
cudaError_t launch_gemm_blockwise(const GemmProblem& p, uint32_t* status, cudaStream_t stream);
cudaError_t launch_blockwise_linear(int M, int N, int K, const __nv_bfloat16* x, const __nv_bfloat16* w,
                                    const __nv_bfloat16* bias, __nv_bfloat16* y, void* scratch, uint32_t* status,
                                    cudaStream_t stream);

// mxfp8.cu: MXFP8 casts (E4M3 elements, one E8M0 scale per 32 consecutive elements along K).
// Each job casts src [rows, K] (bf16, K % 32 == 0) and writes the represented values P * 2^e
// as bf16 into deq (may be src itself), and, when not null, the E4M3 codes [rows, K] and the
// E8M0 scale codes e + 127 [rows, K/32].
struct MxJob {
  const __nv_bfloat16* src = nullptr;
  __nv_bfloat16* deq = nullptr;
  uint8_t* codes = nullptr;
  uint8_t* scales = nullptr;
  int64_t rows = 0;
  int K = 0;
};
constexpr int kMxMaxJobs = 8;
struct MxJobs {
  MxJob j[kMxMaxJobs];
  int n = 0;
};
cudaError_t launch_mx_cast(const MxJob* jobs, int n, cudaStream_t stream);
// The MXFP8 linear y = x W^T + b (bf16 x, W, b, y): the casts of x and W into `scratch`
// (mx_linear_scratch bytes: x values, W values (bf16), x codes, W codes, x scales, W scales,
// each part 256-byte aligned), then the bf16 GEMM of the represented values.  K % 32 == 0.
size_t mx_linear_scratch(int M, int N, int K);
cudaError_t launch_mx_linear(int M, int N, int K, const __nv_bfloat16* x, const __nv_bfloat16* w,
                             const __nv_bfloat16* bias, __nv_bfloat16* y, void* scratch, uint32_t* status,
                             cudaStream_t stream);

struct AttnBwdProblem {
  int batch = 0, heads = 0, seq = 0, seq_pad = 0;
  const __half *q = nullptr, *k = nullptr, *v = nullptr, *dout = nullptr;  // [B, H, S, 128] fp16
  const float *lse = nullptr, *dsum = nullptr;  // [B, H, S_pad] (+ 64 floats of slack)
  float *dq = nullptr, *dk = nullptr, *dv = nullptr;  // [B, H, S, 128] fp32; dq zeroed by the launcher
};
cudaError_t launch_attention_bwd(const AttnBwdProblem& p, uint32_t* status, cudaStream_t stream);

// backward.cu: the row-wise steps of the block backward.
// QK-RMSNorm + RoPE backward of one stream.  q_pre, k_pre are columns [0, D) and [D, 2D) of
// qkv_pre [B, S_s, 3D] (the QKV linear's output with bias, before the norm); dq, dk, dv are the
// attention backward's fp32 [B, H, S_joint, 128] at joint rows seq_offset + s, scaled by the
// gradient scale of `amax` (null: 1); dqkv [B, S_s, 3D] receives dq_pre | dk_pre | dv unscaled.
struct QkBwdArgs {
  const void* qkv_pre = nullptr;
  const void* g_q = nullptr;  // [128] activation type
  const void* g_k = nullptr;
  const float* cos = nullptr;  // [B, S_joint, 64]
  const float* sin = nullptr;
  const void* dq = nullptr;
  const void* dk = nullptr;
  const void* dv = nullptr;
  void* dqkv = nullptr;
  float* part = nullptr;  // [qk_norm_rope_bwd_blocks(), 2, 128]
  const float* amax = nullptr;
  int batch = 0, seq_s = 0, seq_joint = 0, seq_offset = 0, heads = 0, hidden = 0, interleaved = 1;
  float eps = 1e-6f;
};
// h = LN(x)(1 + scale) + shift: dx (fp32) += the input gradient; dscale, dshift (per batch at
// b * mod_bstride; = or += with accumulate) through part (ln_modulate_bwd_part_bytes).
size_t ln_modulate_bwd_part_bytes(int batch, int rows_per_batch, int dim);
cudaError_t launch_ln_modulate_bwd(int act, int x_f32, const void* x, const void* dh, const float* scale,
                                   int64_t mod_bstride, int batch, int rows_per_batch, int dim, float eps,
                                   float* dx, float* dscale, float* dshift, int accumulate, float* part,
                                   cudaStream_t stream);
// y = x + gate f: df = dy gate (activation type), dgate (per batch, written) through part.
size_t gated_residual_bwd_part_bytes(int batch, int rows_per_batch, int dim);
cudaError_t launch_gated_residual_bwd(int act, const float* dy, const void* f, const float* gate,
                                      int64_t gate_bstride, int batch, int rows_per_batch, int dim,
                                      void* df, float* dgate, float* part, cudaStream_t stream);
// out = du GELU'(u_pre) (out may alias du).
cudaError_t launch_gelu_bwd(int act, const void* du, const void* u_pre, int64_t n, int tanh_form, void* out,
                            cudaStream_t stream);
int qk_norm_rope_bwd_blocks();
cudaError_t launch_qk_norm_rope_bwd(int act, const QkBwdArgs& a, float* dg_q, float* dg_k, cudaStream_t stream);
// amax[0] = max(amax[0], max |x|) (amax zeroed first when zero_first).
cudaError_t launch_grad_amax(const __nv_bfloat16* x, int64_t n, float* amax, bool zero_first, cudaStream_t stream);
// D[b, h, seq_offset + s] = g rowsum(dO O) and dOh = g dO head-major [B, H, S_joint, 128] (fp16), with g
// the gradient scale of amax(dO).
cudaError_t launch_attn_bwd_pre(const __nv_bfloat16* o, const __nv_bfloat16* dout, int batch, int seq_s,
                                int seq_joint, int seq_pad, int seq_offset, int heads, const float* amax,
                                float* Dsum, __half* doh, cudaStream_t stream);
// V [BH, S, 128] fp16 from V^T [BH, 128, S_pad] fp16.
cudaError_t launch_untranspose_vt(const __half* vt, int bh, int seq, int seq_pad, __half* v, cudaStream_t stream);
// q16 = q, k16 = k as fp16 (n elements each, n % 8 == 0; exact within fp16's range).
cudaError_t launch_qk_to_f16(const __nv_bfloat16* q, const __nv_bfloat16* k, int64_t n, __half* q16, __half* k16,
                             cudaStream_t stream);
// m = SiLU(vec) W^T + b: dW [rows, dim] and db [rows] fp32 (written; either may be null) and dvec
// [batch, dim] fp32 (= or += with accumulate) through part (modulation_dvec_chunks(rows) * batch *
// dim floats).  batch <= 8.
int modulation_dvec_chunks(int rows);
cudaError_t launch_modulation_bwd(int act, const void* vec, const void* w, const float* dm, int batch, int rows,
                                  int dim, float* dw, float* db, float* dvec, int accumulate, float* part,
                                  cudaStream_t stream);
// dst = src between the activation type and fp32 (to_f32 = 1: activation type -> fp32).
cudaError_t launch_convert(int act, int to_f32, const void* src, int64_t n, void* dst, cudaStream_t stream);

// elementwise.cu
cudaError_t launch_rope3d(const float* ids, int batch, int seq, const int axes[3], float theta,
                          float* cos_out, float* sin_out, cudaStream_t stream);
// m[b, n] = sum_k SiLU(vec[b, k]) w[n, k] + bias[n], n < rows, k < dim; m fp32 [B, rows].
cudaError_t launch_modulation(int act, const void* vec, const void* w, const void* bias, int batch,
                              int rows, int dim, float* m, cudaStream_t stream);
// The same for up to two weight sets sharing `vec`, in one launch.
struct ModulationJob {
  const void* w;
  const void* bias;
  void* out;  // [batch, rows]: fp32, or the activation type under kGemvOutAct
  int rows;
};
cudaError_t launch_modulation2(int act, const void* vec, const ModulationJob* jobs, int njobs,
                               int batch, int dim, cudaStream_t stream);
// The GEMV behind the modulation, for any number of weight matrices that read one input:
// out_j[b, :] (=, or +=) f(vec[b, :]) W_j^T + b_j, f = SiLU when silu != 0, else the identity.
// Jobs are grouped into launches of up to 80, batch rows into groups of up to 8.  vec is of the
// activation type, or fp32 when vec_f32 != 0 (the weights keep the activation type).
enum { kGemvOutF32 = 0, kGemvOutF32Add = 1, kGemvOutAct = 2 };
cudaError_t launch_gemv(int act, const void* vec, const ModulationJob* jobs, int njobs, int batch,
                        int dim, int silu, int mode, cudaStream_t stream, int vec_f32 = 0);
// Sinusoidal timestep features out[b, :] = [cos(tau f_k), sin(tau f_k)], tau = time_factor t[b],
// f_k = max_period^(-k / half), k < half = dim / 2 (dim even, half <= 256).
cudaError_t launch_timestep_features(int act, const float* t, int batch, int dim,
                                     double time_factor, double max_period, void* out,
                                     cudaStream_t stream);
// out [C, ld_out] = in [R, C] transposed (activation type), columns R .. ld_out - 1 zero.
cudaError_t launch_transpose_pad(int act, const void* in, int R, int C, int ld_out, void* out,
                                 cudaStream_t stream);
// out[c] = sum over rows of in [R, C] (fp32), fixed order: `chunks` row chunks into part
// [chunks, C], then summed in chunk order.
cudaError_t launch_colsum(int act, const void* in, int R, int C, float* part, int chunks, float* out,
                          cudaStream_t stream);
// vec = v32 (+ g[b] w_g + b_g when g != NULL), written in the activation type.
cudaError_t launch_vec_finish(int act, const float* v32, const float* g, const void* wg,
                              const void* bg, int batch, int dim, void* vec, cudaStream_t stream);
// out[r, :] = LN(x[r, :]) * (1 + scale[b]) + shift[b], b = r / rows_per_batch; x, out [R, D].
// x is fp32 when x_f32 != 0, else of the activation type; out is of the activation type.
cudaError_t launch_ln_modulate(int act, int x_f32, const void* x, const float* shift, const float* scale,
                               int64_t mod_bstride, int rows, int rows_per_batch, int dim, float eps,
                               void* out, cudaStream_t stream);
// The same for up to two row sets in one launch.
struct LnModJob {
  const void* x;
  const float* shift;
  const float* scale;
  int64_t mod_bstride;
  void* out;
  int rows;
  int rows_per_batch;
  // E4M3 output (out_e4m3 != 0 in the launch): out holds codes of the result * q_scale[0], and
  // q_amax[0] is raised to the largest |result|
  const float* q_scale = nullptr;
  float* q_amax = nullptr;
};
cudaError_t launch_ln_modulate2(int act, int x_f32, const LnModJob* jobs, int njobs, int dim, float eps,
                                cudaStream_t stream, int out_e4m3 = 0);
// z [B, C, HW] fp32 -> tokens [B, HW, C] of the activation type.  With z1 and t non-null the
// tokens are those of (1 - t[b]) z + t[b] z1 (the rectified-flow z_t, formed while reading), also
// written to z_t [B, C, HW] fp32 when z_t is non-null.
cudaError_t launch_patchify(int act, const float* z, int batch, int channels, int hw, void* out,
                            cudaStream_t stream, const float* z1 = nullptr, const float* t = nullptr,
                            float* z_t = nullptr);
// The output head's last stage with the flow-matching loss fused on: v = sum of the split-K
// partials [splits, M, N] + bias; pred[b, n, r] = v (m = b * hw + r; skipped if pred is null);
// with z0 non-null, loss = mean over M * N of (v - (z1 - z0))^2 (z0, z1 [B, N, hw] fp32), reduced
// in a fixed order through loss_partials [head_finish_blocks(M, N)] and a ticket counter that must
// be 0 on entry (the kernel leaves it 0).  N a multiple of 32.
int head_finish_blocks(int M, int N);
cudaError_t launch_head_finish(int act, const float* partials, int splits, int M, int N, const void* bias,
                               int hw, float* pred, const float* z0, const float* z1,
                               float* loss_partials, unsigned int* ticket, float* loss,
                               cudaStream_t stream);
// v [B, H, S, 128] bf16 -> vt [B, H, 128, seq_pad] fp16 (exact: bf16 values fit fp16 here)
cudaError_t launch_transpose_v(const __nv_bfloat16* v, int bh, int seq, int seq_pad, __half* vt,
                               cudaStream_t stream);
// Split-K finish: out[m, n] = sum_s partials[s][m][n] + bias[n] in the activation type, or, when
// unpatchify_rows > 0, pred[b, n, r] (fp32) with m = b * unpatchify_rows + r.
cudaError_t launch_splitk_reduce(int act, const float* partials, int splits, int M, int N,
                                 const void* bias, void* out, int unpatchify_rows,
                                 cudaStream_t stream);
// fp8.cu: E4M3 casts with delayed per-tensor scaling.
// dst[i] = E4M3(src[i] * scale[0]) (round to nearest even, saturating), and amax[0] is raised to
// max |src[i]|; n a multiple of 16, src and dst 16-byte aligned.
struct QuantJob {
  const __nv_bfloat16* src;
  uint8_t* dst;  // null: record max |src| into amax only
  int64_t n;
  const float* scale;
  float* amax;
  int e5m2 = 0;  // 1: E5M2 codes (the hybrid recipe's gradient format) instead of E4M3
};
constexpr int kQuantMaxJobs = 8;
cudaError_t launch_quantize_e4m3(const QuantJob* jobs, int njobs, cudaStream_t stream);
// out [C, ld_out] = in [R, C] transposed, for bytes (E4M3 / E5M2 codes); columns R .. ld_out - 1
// are zero.
cudaError_t launch_transpose_u8(const uint8_t* in, int R, int C, int ld_out, uint8_t* out, cudaStream_t stream);
// hist[i * hist_len + pos] = 0 for i < n.
cudaError_t launch_amax_reset(float* hist, int hist_len, int n, int pos, cudaStream_t stream);
// scale[i] = 448 / amax / 2^margin where amax, positive and finite, is hist[i * hist_len + pos]
// (algo 0, most_recent) or the largest of hist[i * hist_len + 0 .. hist_len) (algo 1, max).
cudaError_t launch_scale_update(const float* hist, float* scale, int hist_len, int n, int pos,
                                int margin, int algo, cudaStream_t stream);
// One Euler step with classifier-free guidance: z_out = z - dt (v_uncond + w (v_cond - v_uncond)),
// or z - dt v_cond when v_uncond is null; n a multiple of 8.
cudaError_t launch_euler_cfg(int dtype, int64_t n, const void* z, const void* v_cond,
                             const void* v_uncond, float guidance, float dt, void* z_out,
                             cudaStream_t stream);
// Rectified-flow noise and loss.  The loss kernel writes one partial sum per block, each block
// covering kFlowElemsPerPartial elements (fewer blocks, with a grid-stride loop, past
// kFlowMaxPartials); flow_partial_blocks gives that count, and launch_flow_match must be given it.
constexpr int64_t kFlowElemsPerPartial = 256 * 8 * 4;
constexpr int kFlowMaxPartials = 1024;
int flow_partial_blocks(int64_t n_total);
cudaError_t launch_flow_match(int dtype, const void* z0, const void* z1, const float* t, int batch,
                              int64_t n_per_sample, void* z_t, const void* pred, float* loss,
                              float* partials, int n_partials, cudaStream_t stream);

}  // namespace mmdit
