/*
 * mmdit.h -- C ABI of the GB300 (sm_103a) Flux MMDiT block-forward library (libmmdit.so).
 *
 * The library computes, with hand-written CUDA kernels for sm_103a, the forward pass of the
 * Flux double-stream (joint) block and single-stream block, their input embeddings and output
 * head, the 3D RoPE tables, and the rectified-flow noise / velocity target / MSE loss.
 *
 * Sources (page title, section):
 *   [API]  "Flux model API reference"
 *   [ARCH] "Flux architecture deep dive"
 *   [FP8]  "FP8 training for Flux models"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is DEVICE memory owned by the caller, except `dims`, the weight-set
 *    structs and `axes_dim`, which are host memory read during the call.  The library
 *    allocates no device memory and keeps no device state between calls, with one exception:
 *    flow_match_noise_and_loss_noalloc keeps its partial sums in a static device array of
 *    its own (described at its declaration).
 *  - Calls are asynchronous: kernels are enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and the call returns without synchronising.
 *  - Layouts are row-major.  Activations are token-major [B, S, features].  Linear weights are
 *    [out, in] (y = x W^T + b).  The QKV weight is [3D, D] as q|k|v blocks, each head-major
 *    (column h*head_dim + j is head h, element j).
 *  - Element types: `act` selects fp32 (MMDIT_F32: linears on tf32 tensor cores) or bf16
 *    (MMDIT_BF16).  Activations, weights, biases, gains and `vec` all use the `act` type.
 *    RoPE tables, modulation vectors, timesteps and the loss are fp32.
 *  - Every device pointer must be 16-byte aligned.  Row strides are the dense ones implied by
 *    the shapes; feature widths must be multiples of 8 elements so that rows fed to the
 *    tensor-memory-access (TMA) engine start on 16-byte boundaries.
 *  - Workspaces: entry points that take `workspace` need at least the bytes the matching
 *    *_workspace_size function returns, 256-byte aligned.  The first 256 bytes hold a device
 *    status word that the call clears on entry; kernels with bounded waits set bits there if a
 *    wait gives up (they then return early and the outputs are undefined).  Read it with
 *    mmdit_workspace_status after the stream has run.
 *  - Errors: argument problems return MMDIT_ERR_INVALID_ARG, shapes or modes the library does
 *    not implement return MMDIT_ERR_UNSUPPORTED, a short workspace returns
 *    MMDIT_ERR_WORKSPACE -- all before anything is enqueued.  A failed CUDA call or launch
 *    returns MMDIT_ERR_CUDA.  mmdit_last_error() gives a message for the calling thread's last
 *    failure.
 *  - Aliasing: outputs must not alias inputs unless an entry point says otherwise.
 */
#ifndef MMDIT_H_
#define MMDIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mmdit_status {
  MMDIT_OK = 0,
  MMDIT_ERR_INVALID_ARG = 1,
  MMDIT_ERR_UNSUPPORTED = 2,
  MMDIT_ERR_WORKSPACE = 3,
  MMDIT_ERR_CUDA = 4,
  MMDIT_ERR_NONFINITE = 5, /* reserved for a non-finite check of the outputs; no entry point returns it */
  MMDIT_ERR_DEVICE = 6 /* a kernel's bounded wait gave up; see mmdit_workspace_status */
} mmdit_status;

typedef enum mmdit_act_dtype { MMDIT_F32 = 0, MMDIT_BF16 = 1 } mmdit_act_dtype;

/* Linear-layer arithmetic: NATIVE = tf32 for MMDIT_F32, bf16 for MMDIT_BF16.
 * FP8_E4M3 = the four block linears (QKV, output projection, fc1, fc2) on E4M3 operands with
 * delayed per-tensor scaling ([FP8] §Configuration); needs act = MMDIT_BF16 and
 * mlp_hidden % 128 == 0.  The modulation, the attention (bf16, [FP8] §Configuration:
 * fp8_dot_product_attention false) and every other step keep the activation type. */
/* FP8_TENSORWISE = the same four linears on E4M3 operands with per-tensor CURRENT scaling ([FP8]
 * §Configuration, fp8_recipe "tensorwise"; §Training configuration, Aggressive): each operand's
 * scale comes from its own absolute maximum in the same call, scale = 448 / amax / 2^margin, so
 * every input is first written in bf16, its amax taken, then cast (weights likewise at every
 * call).  The state's history column `pos` records those amax and `scale` ends holding the scales
 * used; amax_compute_algo is not read. */
/* FP8_BLOCKWISE = the same four linears under the blockwise recipe ([FP8] §Configuration,
 * fp8_recipe "blockwise"; the arithmetic of mmdit_fp8_blockwise_linear_fwd): each input, written
 * in bf16, is cast per 1 x 128 tile of its rows and each weight per 128 x 128 tile, every tile
 * with its own scale 448 / amax, and the GEMMs rescale each 128-wide K slice's product before
 * their usual epilogues.  Nothing is kept between calls: the fp8 state argument must be NULL.
 * Needs hidden % 128 == 0 and mlp_hidden % 128 == 0; not for the parallel single block. */
/* FP8_MXFP8 = the same four linears under the MXFP8 recipe ([FP8] §Configuration, fp8_recipe
 * "mxfp8"; the arithmetic of mmdit_fp8_mxfp8_linear_fwd): each input, written in bf16, and each
 * weight are cast per 32 consecutive elements along K to E4M3 with a shared power-of-two scale,
 * and the linears multiply the values those casts represent (bf16 tensor cores, fp32 sums).
 * Nothing is kept between calls: the fp8 state argument must be NULL.  Needs
 * mlp_hidden % 128 == 0. */
typedef enum mmdit_gemm_mode {
  MMDIT_GEMM_NATIVE = 0,
  MMDIT_GEMM_FP8_E4M3 = 1,
  MMDIT_GEMM_FP8_TENSORWISE = 2,
  MMDIT_GEMM_FP8_BLOCKWISE = 3,
  MMDIT_GEMM_FP8_MXFP8 = 4
} mmdit_gemm_mode;

/* Shapes and options of one block call ([API] §Configuration, FluxConfig). */
typedef struct mmdit_dims {
  int32_t batch;      /* B */
  int32_t seq_img;    /* image tokens S_i */
  int32_t seq_txt;    /* text tokens S_t; the joint sequence is [image; text], S = S_i + S_t */
  int32_t hidden;     /* D = heads * head_dim; multiple of 128, at most 6144 */
  int32_t heads;      /* H */
  int32_t head_dim;   /* d; must be 128 */
  int32_t mlp_hidden; /* F; multiple of 64 */
  float ln_eps;       /* LayerNorm eps (1e-6, [API] §Configuration layernorm_epsilon) */
  float rms_eps;      /* QK-RMSNorm eps (1e-6) */
  int32_t rope_interleaved; /* 1: pairs (2j, 2j+1) ([API] rotary_interleaved); 0: (j, j+d/2) */
  int32_t gelu_tanh;  /* 0: exact erf GELU; 1: tanh approximation */
  int32_t act;        /* mmdit_act_dtype */
  int32_t gemm;       /* mmdit_gemm_mode */
} mmdit_dims;

/* One stream's weights ([ARCH] §Model components, 3. MMDiT layer).  All device pointers of
 * element type `act`.  Shapes: w_mod [6D, D], b_mod [6D] (AdaLN chunks in the order shift,
 * scale, gate, shift_mlp, scale_mlp, gate_mlp -- [API] §Normalization, AdaLN); w_qkv [3D, D],
 * b_qkv [3D]; g_q, g_k [d] (per-head QK-RMSNorm gains); w_o [D, D], b_o [D] (attention output
 * projection); w_1 [F, D], b_1 [F]; w_2 [D, F], b_2 [D] (GELU MLP).
 * mod: NULL, or this stream's modulation [B, 6D] fp32 (16-byte aligned) as mmdit_modulation_fwd
 * computes it from w_mod, b_mod and the call's vec -- for example on another stream, overlapped
 * with earlier work.  The block then reads it instead of recomputing it; the caller orders that
 * computation before the block call and keeps the buffer until the call has completed. */
typedef struct mmdit_stream_w {
  const void *w_mod, *b_mod;
  const void *w_qkv, *b_qkv;
  const void *g_q, *g_k;
  const void *w_o, *b_o;
  const void *w_1, *b_1;
  const void *w_2, *b_2;
  const float *mod;
} mmdit_stream_w;

/* FP8 delayed-scaling state of the block linears ([FP8] §Configuration, FP8 model
 * configuration: E4M3, amax_history_len 1024, amax_compute_algo most_recent, margin 0).
 * Caller-owned device memory; the struct itself is read on the host during the call.
 *   amax_history [n_tensors, hist_len] fp32 (row t is tensor t's history)
 *   scale        [n_tensors] fp32: the scale tensor t is cast with (E4M3(x * scale)); start
 *                with 1 (an empty history) and let the library update it
 *   pos          the history column this call records into, 0 <= pos < hist_len; the library
 *                does not advance it (the caller moves it between calls, e.g. pos + 1 mod
 *                hist_len; a replayed CUDA graph records into the column it was captured with)
 * Tensor t = 8 * slot + 2 * linear + operand, with slot 0 = image stream (or the single
 * block's one stream) and 1 = text stream; linear 0 = QKV, 1 = attention output projection,
 * 2 = fc1, 3 = fc2; operand 0 = the linear's input, 1 = its weight.  A double block needs
 * n_tensors >= 16, a single block >= 8.  A call zeroes column pos of those tensors, records
 * max |x| of every tensor it casts there, and, after its last linear, sets
 * scale[t] = 448 / amax / 2^margin for every such tensor whose amax is positive and finite (the
 * others keep their scale), where amax is amax_history[t, pos] with amax_compute_algo 0
 * (most_recent) or the largest entry of row t with amax_compute_algo 1 (max; [FP8]
 * §Troubleshooting and §Training configuration give it as the conservative choice).
 * margin: 0 to 16 ([FP8] §Configuration fp8_margin).  Calls sharing a state must be ordered on
 * one stream. */
typedef struct mmdit_fp8_state {
  float *amax_history; /* [n_tensors, hist_len] */
  float *scale;        /* [n_tensors] */
  int32_t hist_len;
  int32_t n_tensors;
  int32_t pos;
  int32_t amax_compute_algo; /* 0: most_recent, 1: max over the history */
  int32_t margin;            /* scale = 448 / amax / 2^margin */
} mmdit_fp8_state;

/* Message for the calling thread's most recent non-OK status (never NULL). */
const char *mmdit_last_error(void);

/* Synchronises `stream`, reads the status word of `workspace` and clears it.  Returns MMDIT_OK,
 * MMDIT_ERR_DEVICE if a kernel recorded a timed-out wait (bits in *bits_out if non-NULL), or
 * MMDIT_ERR_CUDA. */
mmdit_status mmdit_workspace_status(void *workspace, uint32_t *bits_out, void *stream);

/* Number of the library's own kernel launches enqueued by this thread since the last reset
 * (a diagnostic count used by benchmarks); mmdit_launch_count_reset() sets it to zero. */
uint64_t mmdit_launch_count(void);
void mmdit_launch_count_reset(void);

/* Per-step timing for diagnostics.  While enabled (on != 0) on the calling thread, every
 * library step (one named kernel, or a short fixed group such as the modulation GEMV) is
 * bracketed by two CUDA events recorded on the caller's stream.  mmdit_profile_collect
 * synchronises `stream`, writes up to max_entries records -- the step name (NUL-separated in
 * names_out, at most names_len bytes in total) and its duration in milliseconds (ms_out) --
 * clears the record and returns the number of records (or -1 on a CUDA error).  Enabling and
 * collecting must not overlap a stream capture. */
void mmdit_profile_enable(int32_t on);
int32_t mmdit_profile_collect(void *stream, char *names_out, size_t names_len, float *ms_out,
                              int32_t max_entries);

/* ---------------------------------------------------------------------------------------
 * 3D RoPE tables ([ARCH] §Model components, 2. Position embeddings (3D RoPE), and
 * §Mathematical formulation, 3D RoPE mathematics; [API] §Position embeddings, EmbedND).
 * For token ids p = ids[b, s, 0..2] and axis a of width axes_dim[a] (even), pair i < axes_dim[a]/2
 * gets angle p[a] * theta^(-2i/axes_dim[a]); the axes' angles are concatenated in axis order.
 *   ids      [batch, seq, 3] fp32 (device)
 *   axes_dim host int32[3], each even, sum <= 256 (Flux: 16, 56, 56)
 *   cos_out, sin_out [batch, seq, P] fp32 (device), P = sum(axes_dim)/2
 * No workspace.  batch*seq == 0 is a no-op. */
mmdit_status rope3d_freqs(const float *ids, int32_t batch, int32_t seq, const int32_t *axes_dim,
                          float theta, float *cos_out, float *sin_out, void *stream);

/* ---------------------------------------------------------------------------------------
 * AdaLN modulation ([API] §Normalization, AdaLN; [ARCH] §Implementation details, Adaptive
 * layer normalization): out[b, r] = sum_k SiLU(vec[b, k]) w[r, k] + bias[r], the linear of the
 * SiLU of the conditioning vector whose 6D rows a block splits into (shift, scale, gate) for the
 * attention and MLP branches (2D rows for the output head).
 *   vec [batch, dim], w [rows, dim], bias [rows] (may be NULL): element type `act`
 *   out [batch, rows] fp32.  dim a multiple of 8, at most 6144.  No workspace.
 * The result can be handed to a block through mmdit_stream_w.mod. */
mmdit_status mmdit_modulation_fwd(int32_t act, int32_t batch, int32_t rows, int32_t dim,
                                  const void *vec, const void *w, const void *bias, float *out,
                                  void *stream);

/* ---------------------------------------------------------------------------------------
 * Rectified flow ([ARCH] §Mathematical formulation, Flow matching objective; [API] §Training
 * utilities, apply_flow_matching_noise and compute_flow_matching_loss).
 *   z_t  = (1 - t[b]) * z0 + t[b] * z1                        (written if z_t != NULL)
 *   loss = mean over all batch*n elements of (pred - (z1 - z0))^2   (written if pred and
 *          loss are both non-NULL; one fp32 scalar; fixed-order, deterministic reduction)
 * z0, z1, z_t, pred: [batch, n_per_sample] of type `dtype` (MMDIT_F32 or MMDIT_BF16);
 * n_per_sample a multiple of 8.  t: [batch] fp32.
 * workspace >= flow_match_workspace_size(batch, n_per_sample) (per-block partial sums).
 * z_t may alias z0 or z1 only when no loss is requested. */
size_t flow_match_workspace_size(int32_t batch, int64_t n_per_sample);
mmdit_status flow_match_noise_and_loss(int32_t dtype, const void *z0, const void *z1,
                                       const float *t, int32_t batch, int64_t n_per_sample,
                                       void *z_t, const void *pred, float *loss,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* flow_match_noise_and_loss without a workspace, for callers that cannot allocate device
 * memory (a plug-in running under another framework's allocator, or a host whose memory is
 * fixed at start-up).  The pages have no counterpart; this is a packaging variant of the entry
 * point above with the same results.  The partial sums of the loss live in a static device
 * array of 256 floats (1 KiB) that every GPU loading the library keeps until the process exits,
 * so batch * n_per_sample may be at most 2,097,152; larger calls return MMDIT_ERR_UNSUPPORTED
 * (checked without forming the product).  Nothing is allocated.  The first call on each device
 * looks up the array's address (cudaGetSymbolAddress) and should precede any stream capture;
 * the address is kept for the life of the process, so after a cudaDeviceReset of a device this
 * entry point must not be called on it again.  All calls share the array: calls whose kernels
 * overlap on the GPU race, so order them on one stream. */
mmdit_status flow_match_noise_and_loss_noalloc(int32_t dtype, const void *z0, const void *z1,
                                               const float *t, int32_t batch,
                                               int64_t n_per_sample, void *z_t,
                                               const void *pred, float *loss, void *stream);

/* One sampling step ([ARCH] §Mathematical formulation, Sampling (inference): Euler integration
 * from t = 1 towards t = 0, and Classifier-free guidance):
 *   v     = v_uncond + guidance * (v_cond - v_uncond)   (v = v_cond when v_uncond is NULL)
 *   z_out = z - dt * v                                    (z_{t - dt} = z_t - dt v_t)
 * z, v_cond, v_uncond, z_out: [n] of type `dtype` (MMDIT_F32 or MMDIT_BF16), 16-byte aligned;
 * z_out may alias z.  n a multiple of 8; n == 0 is a no-op.  fp32 arithmetic.  No workspace. */
mmdit_status flow_match_euler_step(int32_t dtype, int64_t n, const void *z, const void *v_cond,
                                   const void *v_uncond, float guidance, float dt, void *z_out,
                                   void *stream);

/* ---------------------------------------------------------------------------------------
 * Plain linear layer y = x W^T + b on the tensor cores (the text embedding txt_in of [ARCH]
 * §Model components, 1. Input embeddings, and any other projection).
 *   x [M, K], w [N, K], b [N] (may be NULL), y [M, N]; element type `act`.
 *   N multiple of 32, K multiple of 8.  workspace >= mmdit_linear_workspace_size(act, M, N, K)
 *   (a narrow output with a long K is split along K; the fp32 partial sums live there). */
size_t mmdit_linear_workspace_size(int32_t act, int32_t M, int32_t N, int32_t K);
mmdit_status mmdit_linear_fwd(int32_t act, int32_t M, int32_t N, int32_t K, const void *x,
                              const void *w, const void *b, void *y, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Image embedding img_in ([ARCH] §Model components, 1. Input embeddings, and §Implementation
 * details, Memory layout): patchify latents [B, C, H, W] (fp32, patch size 1, token r*W + c)
 * into [B, H*W, C] and project with w [D, C], b [D] to out [B, H*W, D] (type `act`).
 * C multiple of 8. */
size_t mmdit_img_in_workspace_size(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                                   int32_t lat_w);
mmdit_status mmdit_img_in_fwd(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                              int32_t lat_w, int32_t hidden, const float *z, const void *w,
                              const void *b, void *out, void *workspace, size_t workspace_bytes,
                              void *stream);

/* img_in with the rectified-flow noise fused into its load ([ARCH] §Mathematical formulation,
 * Flow matching objective, and §Training data flow: the noised latents enter the image
 * embedding): the latents are z_t = (1 - t[b]) z0 + t[b] z1, formed while patchifying (the same
 * fp32 arithmetic as flow_match_noise_and_loss, so z_t is bit-equal), then projected as
 * mmdit_img_in_fwd projects z.
 *   z0, z1 [B, C, H, W] fp32; t [B] fp32; w, b, out as for mmdit_img_in_fwd;
 *   z_t: NULL, or [B, C, H, W] fp32 receiving the noised latents (may not alias z0 or z1).
 * workspace >= mmdit_img_in_workspace_size(act, batch, channels, lat_h, lat_w). */
mmdit_status mmdit_img_in_noise_fwd(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                                    int32_t lat_w, int32_t hidden, const float *z0, const float *z1,
                                    const float *t, const void *w, const void *b, void *out,
                                    float *z_t, void *workspace, size_t workspace_bytes, void *stream);

/* Output head ([ARCH] §Model components, 5. Output processing; [API] AdaLNContinuous):
 * (shift, scale) = SiLU(vec) w_ada^T + b_ada (w_ada [2D, D]); y = (LN(x_img) * (1 + scale) +
 * shift) w_out^T + b_out (w_out [C, D]); pred [B, C, H, W] fp32 with token r*W + c at [.., r, c].
 * Uses dims->batch, hidden, ln_eps, act; x_img is [B, lat_h*lat_w, D].  C multiple of 32. */
size_t mmdit_final_layer_workspace_size(const mmdit_dims *dims, int32_t channels);
mmdit_status mmdit_final_layer_fwd(const mmdit_dims *dims, int32_t channels, int32_t lat_h,
                                   int32_t lat_w, const void *x_img, const void *vec,
                                   const void *w_ada, const void *b_ada, const void *w_out,
                                   const void *b_out, float *pred, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Output head with the flow-matching loss fused onto its output stage ([ARCH] §Training data
 * flow: the prediction feeds the loss; §Mathematical formulation, Flow matching objective; [API]
 * §Training utilities, compute_flow_matching_loss): the head of mmdit_final_layer_fwd, whose last
 * kernel also forms
 *   loss = mean over all B * C * H * W elements of (pred - (z1 - z0))^2
 * from the prediction while it is in registers (one fp32 scalar; partial sums per block added
 * in a fixed order by the last block: deterministic).
 *   z0, z1 [B, C, H, W] fp32 (the latent pair of this step); loss: device fp32 scalar (4-byte
 *   aligned);
 *   pred: NULL, or [B, C, H, W] fp32 receiving the prediction (may not alias z0 or z1);
 *   mod: NULL, or the head's (shift, scale) [B, 2D] fp32 = SiLU(vec) w_ada^T + b_ada computed ahead
 *   (mmdit_modulation_fwd or the batched launch, which also takes the blocks' modulations);
 *   w_ada and b_ada are then not read.
 * Other arguments as mmdit_final_layer_fwd.
 * workspace >= mmdit_final_layer_loss_workspace_size(dims, channels). */
size_t mmdit_final_layer_loss_workspace_size(const mmdit_dims *dims, int32_t channels);
mmdit_status mmdit_final_layer_loss_fwd(const mmdit_dims *dims, int32_t channels, int32_t lat_h,
                                        int32_t lat_w, const void *x_img, const void *vec,
                                        const void *w_ada, const void *b_ada, const void *w_out,
                                        const void *b_out, const float *z0, const float *z1,
                                        float *pred, float *loss, const float *mod, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * LayerNorm + modulate on its own ([ARCH] §Implementation details, Adaptive layer normalization;
 * [API] §Normalization, AdaLN): the HBM pass the blocks run before their QKV and fc1 linears,
 *   out[b, r, :] = LN(x[b, r, :]) * (1 + scale[b * mod_bstride + :]) + shift[b * mod_bstride + :]
 * LN without affine, biased variance, fp32 statistics.  x [batch, rows_per_batch, dim] of type
 * `act` (fp32 when x_f32 != 0, as the blocks' fp32 residual), out of type `act` (may not alias x);
 * shift, scale fp32 (16-byte aligned; mod_bstride a multiple of 4 floats).  dim a multiple of 8, at
 * most 8192.  No workspace. */
mmdit_status mmdit_ln_modulate_fwd(int32_t act, int32_t x_f32, int32_t batch, int32_t rows_per_batch,
                                   int32_t dim, float eps, const void *x, const float *shift,
                                   const float *scale, int64_t mod_bstride, void *out, void *stream);

/* Strided row copy for callers that join or split the image and text streams themselves (the
 * single block reads [img; txt] per sample, the output head the image rows): for i < n_rows, copies
 * row_bytes bytes from src + i * src_stride to dst + i * dst_stride (device memory, through the copy
 * engine: cudaMemcpy2DAsync; no kernel).  Strides >= row_bytes; the ranges may not overlap.  Not a
 * step of the method: layout plumbing. */
mmdit_status mmdit_copy_rows(void *dst, int64_t dst_stride, const void *src, int64_t src_stride,
                             int64_t row_bytes, int32_t n_rows, void *stream);

/* ---------------------------------------------------------------------------------------
 * Joint softmax attention ([ARCH] §Implementation details, Attention implementation (no mask)
 * and Joint Attention Trick).  out[b, s, h*d + j] = sum_t softmax_t(q_s . k_t / sqrt(d)) v_t[j]
 * for each (b, h), over all S keys.  q, k, v [B, H, S, d] bf16; out [B, S, H*d] of type
 * `act`.  d must be 128.  workspace >= mmdit_attention_workspace_size(B, H, S).
 * Range: the PV product runs on fp16 operands (the probabilities and V, which fp16 holds exactly
 * for every bf16 value with 2^-14 <= |v| <= 65504).  A |v| above 65504 overflows to an infinite
 * output; a |v| below 2^-14 keeps fewer bits (an absolute error of at most 2^-25 per key weight).
 * The blocks' V, written by their QKV epilogue, is read the same way. */
size_t mmdit_attention_workspace_size(int32_t batch, int32_t heads, int32_t seq);
mmdit_status mmdit_attention_fwd(int32_t act, int32_t batch, int32_t heads, int32_t seq,
                                 int32_t head_dim, const void *q, const void *k, const void *v,
                                 void *out, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Joint attention on E4M3 operands, the opt-in fp8_dot_product_attention of [FP8]
 * §Configuration, FP8 model configuration (the blocks keep attention in bf16, its default):
 *   S  = E4M3(q scale_q) E4M3(k scale_k)^T / (scale_q scale_k sqrt(d))
 *   Pt = exp(S - rowmax S)  (fp32; the flash-style running maximum, so each tile's Pt <= 1)
 *   out = E4M3(Pt 448) E4M3(v scale_v) / (448 scale_v) / rowsum(Pt)   (row sum of the fp32 Pt)
 * Both products run on E4M3 tensor-core operands with fp32 accumulation.  q, k, v [B, H, S, d]
 * bf16; scale_q, scale_k, scale_v device fp32 scalars (e.g. delayed scaling's 448 / amax);
 * out [B, S, H*d] of type `act`.  d must be 128.
 * workspace >= mmdit_fp8_attention_workspace_size(B, H, S) (the casts). */
size_t mmdit_fp8_attention_workspace_size(int32_t batch, int32_t heads, int32_t seq);
mmdit_status mmdit_fp8_attention_fwd(int32_t act, int32_t batch, int32_t heads, int32_t seq,
                                     int32_t head_dim, const void *q, const void *k, const void *v,
                                     const float *scale_q, const float *scale_k, const float *scale_v,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* ---------------------------------------------------------------------------------------
 * Double-stream (joint) block forward ([ARCH] §Model components, 3. MMDiT layer (double
 * block); [API] §Layer specifications, MMDiTLayer).  Per stream s in {img, txt}, each with its
 * own weights:
 *   (shift1, scale1, gate1, shift2, scale2, gate2) = SiLU(vec) w_mod^T + b_mod;
 *   h = LN(x_s) * (1 + scale1) + shift1;   q|k|v = h w_qkv^T + b_qkv;
 *   q, k <- per-head RMSNorm (gains g_q, g_k), then RoPE with the joint-sequence tables;
 *   O = softmax(Q K^T / sqrt(d)) V over the joint sequence [img; txt];
 *   x1 = x_s + gate1 * (O_s w_o^T + b_o);
 *   y_s = x1 + gate2 * (GELU((LN(x1) * (1 + scale2) + shift2) w_1^T + b_1) w_2^T + b_2).
 * vec [B, D]; rope_cos, rope_sin [B, S_i + S_t, d/2] fp32 (rope3d_freqs of the joint ids);
 * x_img, y_img [B, S_i, D]; x_txt, y_txt [B, S_t, D]; y may alias x.
 * fp8: NULL with gemm = MMDIT_GEMM_NATIVE; the delayed-scaling state (n_tensors >= 16) with
 * gemm = MMDIT_GEMM_FP8_E4M3, where every weight is cast to E4M3 at each call (as training
 * does after each optimizer step) and the inputs of the four linears are cast where they are
 * produced (LayerNorm-modulate, the attention output, the fc1 GELU).
 * workspace >= mmdit_double_block_workspace_size(dims) (larger in FP8 mode: it holds the
 * E4M3 weights). */
size_t mmdit_double_block_workspace_size(const mmdit_dims *dims);
mmdit_status mmdit_double_block_fwd(const mmdit_dims *dims, const mmdit_stream_w *w_img,
                                    const mmdit_stream_w *w_txt, const void *vec,
                                    const float *rope_cos, const float *rope_sin,
                                    const void *x_img, const void *x_txt, void *y_img,
                                    void *y_txt, mmdit_fp8_state *fp8, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* Single-stream block forward ([ARCH] §Model components, 4. Flux single block; [API]
 * FluxSingleTransformerBlock): the same chain with one weight set over the whole concatenated
 * sequence x [B, S, D], S = S_i + S_t; returns all S rows in y (may alias x).
 * rope_cos, rope_sin [B, S, d/2].  fp8 as for the double block (n_tensors >= 8).
 * workspace >= mmdit_single_block_workspace_size(dims). */
size_t mmdit_single_block_workspace_size(const mmdit_dims *dims);
mmdit_status mmdit_single_block_fwd(const mmdit_dims *dims, const mmdit_stream_w *w,
                                    const void *vec, const float *rope_cos,
                                    const float *rope_sin, const void *x, void *y,
                                    mmdit_fp8_state *fp8, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* Byte offsets of named intermediates inside a block workspace, for inspection by tests:
 * out[0..16] = mod_img, mod_txt, Q, K, Vt, O_img, O_txt, x1_img, x1_txt, u_img, h_img, h_txt,
 * u_txt, O8_img, O8_txt, Wq_img, Wq_txt (a single block uses the *_img slots; unused slots are
 * -1).  Q, K are [B, H, S, d] bf16, Vt is [B, H, d, S_pad] fp16 (holding bf16-rounded values)
 * with S_pad = S rounded up to 8; h (LayerNorm-modulate output) and u (GELU output) are of the
 * activation type, or E4M3 codes in FP8 mode; O8 is the E4M3 attention output and Wq the E4M3
 * weights (QKV, output projection, fc1, fc2, back to back), FP8 mode only.  Writes
 * min(n, 17) entries and returns that count, or -1 on bad dims. */
int32_t mmdit_block_workspace_offsets(const mmdit_dims *dims, int32_t single, int64_t *out,
                                      int32_t n);

/* ---------------------------------------------------------------------------------------
 * E4M3 cast with delayed scaling ([FP8] §Configuration; the E4M3 format of "FP8 Formats for
 * Deep Learning", which the page selects): out[i] = E4M3(x[i] * scale[0]), rounded to nearest
 * even and saturated to +-448 (NaN stays NaN); amax[0] = max(amax[0], max_i |x[i]|).
 *   x [n] bf16, out [n] uint8 codes (device, 16-byte aligned); scale, amax: device fp32
 *   scalars (e.g. entries of an mmdit_fp8_state).  n a multiple of 16; n == 0 is a no-op.
 * No workspace. */
mmdit_status mmdit_fp8_quantize_e4m3(const void *x, int64_t n, const float *scale, float *amax,
                                     void *out, void *stream);

/* Linear layer on E4M3 operands ([FP8] §Configuration: the FP8 GEMM of a linear under delayed
 * scaling): y = (x_q w_q^T) / (scale_x[0] * scale_w[0]) + b, where x_q [M, K] and w_q [N, K]
 * hold E4M3 codes (as written by mmdit_fp8_quantize_e4m3 with those scales), b [N] bf16 (may
 * be NULL), y [M, N] bf16; fp32 accumulation on the tensor cores.  N % 128 == 0,
 * K % 16 == 0.  workspace >= mmdit_fp8_linear_workspace_size() (the status word). */
size_t mmdit_fp8_linear_workspace_size(void);
mmdit_status mmdit_fp8_linear_fwd(int32_t M, int32_t N, int32_t K, const void *x, const void *w,
                                  const float *scale_x, const float *scale_w, const void *b,
                                  void *y, void *workspace, size_t workspace_bytes, void *stream);

/* Blockwise FP8 linear ([FP8] §Configuration › FP8 model configuration, fp8_recipe "blockwise";
 * the page names the recipe only).  y = x W^T + b with every tile cast to E4M3 under its own
 * current scale s = 448 / amax(tile) (1 for a tile of zeros): x [M, K] in 1 x 128 tiles (one scale
 * per row and 128-wide K slice), W [N, K] in 128 x 128 tiles; the product sums, over the 128-wide
 * K slices j, Q_j(x) Q_j(W)^T / (s_x[m, j] s_w[n / 128, j]) in fp32 (tensor cores on the E4M3
 * codes, each slice rescaled as it is accumulated), then adds b.
 * x, W, b (NULL: none) and y are bf16, 16-byte aligned; N % 128 == 0, K % 128 == 0; M == 0 is a
 * no-op.  The casts are float32: s = 448 / amax is the IEEE quotient, each element's product x s
 * is rounded to float32 and then to E4M3 (nearest even, saturating).  The workspace (at least
 * mmdit_fp8_blockwise_linear_workspace_size bytes) holds after its 256-byte status word, each
 * part starting on a 256-byte boundary: the x codes [M, K], the W codes [N, K], s_x [K/128, M]
 * and s_w [N/128, K/128] (fp32), readable after the call. */
size_t mmdit_fp8_blockwise_linear_workspace_size(int32_t M, int32_t N, int32_t K);
mmdit_status mmdit_fp8_blockwise_linear_fwd(int32_t M, int32_t N, int32_t K, const void *x, const void *w,
                                            const void *b, void *y, void *workspace, size_t workspace_bytes,
                                            void *stream);

/* MXFP8 linear ([FP8] §Configuration › FP8 model configuration, fp8_recipe "mxfp8"; the page
 * names the recipe only, read as the OCP Microscaling formats v1.0 MXFP8 with E4M3 elements).
 * y = x W^T + b where x [M, K] and W [N, K] are each cast in blocks of 32 consecutive elements
 * along K: a block with largest magnitude amax gets the shared exponent
 * e = floor(log2 amax) - 8, clamped to [-127, 127] (-127 for a block of zeros), and each of its
 * elements v is stored as the E4M3 code P = E4M3(v / 2^e) (nearest even, saturating at 448),
 * standing for P * 2^e.  The product of those represented values accumulates in fp32 on the
 * tensor cores (exactly formed bf16 products; exact for every block whose amax is at least
 * 2^-116), then b is added.  x, W, b (NULL: none) and y are bf16, 16-byte aligned, finite;
 * N % 32 == 0, K % 32 == 0; M == 0 is a no-op.  The workspace (at least
 * mmdit_fp8_mxfp8_linear_workspace_size bytes) holds after its 256-byte status word, each part
 * starting on a 256-byte boundary: the represented values of x [M, K] and of W [N, K] (bf16),
 * the E4M3 codes of x [M, K] and of W [N, K], and the E8M0 scale codes e + 127 of x [M, K/32]
 * and of W [N, K/32] (one byte each), readable after the call. */
size_t mmdit_fp8_mxfp8_linear_workspace_size(int32_t M, int32_t N, int32_t K);
mmdit_status mmdit_fp8_mxfp8_linear_fwd(int32_t M, int32_t N, int32_t K, const void *x, const void *w,
                                        const void *b, void *y, void *workspace, size_t workspace_bytes,
                                        void *stream);

/* ---------------------------------------------------------------------------------------
 * Backward of the FP8 linear ([FP8] §Configuration, FP8 model configuration: fp8 "e4m3" or
 * "hybrid", fp8_wgrad; the chain rule of mmdit_fp8_linear_fwd), for a forward that ran on
 * x_q = E4M3(x scale_x) and w_q = E4M3(W scale_w):
 *   G  = Qg(dy * scale_dy[0])          Qg = E4M3 (recipe 0, "e4m3") or E5M2 (recipe 1, "hybrid";
 *                                      round to nearest even, saturating at 57344);
 *                                      amax_dy[0] = max(amax_dy[0], max |dy|)
 *   dx = G w_q / (scale_dy scale_w)    [M, K] bf16
 *   dW = G^T x_q / (scale_dy scale_x)  [N, K] fp32 with fp8_wgrad = 1; dy^T x on the bf16 tensors
 *                                      with fp8_wgrad = 0 (x read only then)
 *   db = column sums of dy             [N] fp32 (fixed order)
 * dy [M, N] bf16; x_q [M, K], w_q [N, K] uint8 codes; x [M, K] bf16; scales and amax_dy device
 * fp32 scalars; dw and db may be NULL.  K % 128 == 0, N % 16 == 0; both products run on the
 * tensor cores (kind::f8f6f4, E5M2 x E4M3 under "hybrid"), fp32 accumulation.
 * workspace >= mmdit_fp8_linear_bwd_workspace_size(M, N, K, fp8_wgrad). */
size_t mmdit_fp8_linear_bwd_workspace_size(int32_t M, int32_t N, int32_t K, int32_t fp8_wgrad);
mmdit_status mmdit_fp8_linear_bwd(int32_t M, int32_t N, int32_t K, int32_t recipe, int32_t fp8_wgrad,
                                  const void *dy, const void *x_q, const void *w_q, const void *x,
                                  const float *scale_x, const float *scale_w, const float *scale_dy,
                                  float *amax_dy, void *dx, float *dw, float *db, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Single-stream block with parallel branches (the whole-model row's shape option; [ARCH]
 * §Model components, 4. Flux single block draws the sequential form above).  One
 * LayerNorm-modulate h = LN(x)(1 + scale) + shift feeds both the attention (QKV, QK-RMSNorm,
 * RoPE, joint attention -> o) and the MLP (u = GELU(h W_1^T + b_1)); one gated residual adds both
 * through the output linear of the concatenation:
 *   y = x + gate ([o | u] [W_o | W_2]^T + b_o + b_2)
 * Modulation: three chunks (shift, scale, gate) = SiLU(vec) w_mod^T + b_mod with w_mod [3D, D],
 * b_mod [3D] (mod, if given, is [B, 3D] fp32); the other weights as mmdit_stream_w states.
 * Arguments, layouts and aliasing as mmdit_single_block_fwd; gemm must be MMDIT_GEMM_NATIVE.
 * workspace >= mmdit_single_block_workspace_size(dims). */
mmdit_status mmdit_single_block_parallel_fwd(const mmdit_dims *dims, const mmdit_stream_w *w,
                                             const void *vec, const float *rope_cos,
                                             const float *rope_sin, const void *x, void *y,
                                             void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Backward of a linear layer y = x W^T + b (the block backward's building block; the pages
 * train these blocks, [ARCH] §Training data flow, and print no backward: the chain rule):
 *   dx = dy W [M, K] (activation type), dW = dy^T x [N, K] fp32, db = column sums of dy [N] fp32.
 * dy [M, N], x [M, K], W [N, K] of type `act`.  Any of dx, dw, db may be NULL (not computed);
 * x is read only for dw and W only for dx.  bf16 operands with fp32 accumulation on the tensor
 * cores (tf32 for MMDIT_F32); db in a fixed order (deterministic).  K % 32 == 0, N % 8 == 0;
 * M == 0 zeroes dw and db.  workspace >= mmdit_linear_bwd_workspace_size(act, M, N, K). */
size_t mmdit_linear_bwd_workspace_size(int32_t act, int32_t M, int32_t N, int32_t K);
mmdit_status mmdit_linear_bwd(int32_t act, int32_t M, int32_t N, int32_t K, const void *dy, const void *x,
                              const void *w, void *dx, float *dw, float *db, void *workspace,
                              size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Block backward (the pages train these blocks: [ARCH] §Training data flow, and §Performance
 * optimizations, 5. Mixed precision, which calls loss.backward(); they print no backward, so
 * each gradient is the chain rule of the forward step it belongs to).
 * Given the block's inputs and dy (the gradient of the loss with respect to its outputs), a call
 * recomputes the forward (activation recomputation: nothing has to be kept from a forward call)
 * and writes
 *   dx   the gradient with respect to each input stream (type `act`; may not alias x or dy),
 *   dvec [B, D] fp32 (NULL: not computed) with respect to the conditioning vector,
 *   and, for each non-NULL member of a stream's mmdit_stream_grads, the fp32 gradient of that
 *   weight (same shape as the weight; written, not accumulated; NULL struct: none).
 * The attention backward recomputes its probabilities from the forward's row log-sum-exp
 * (flash style) and runs on the tensor cores with fp16 operands under a power-of-two gradient
 * scale; every reduction over rows (weight, bias, gain and modulation gradients) is a fixed-order
 * sum, so results are deterministic except dQ's atomic accumulation order in the attention
 * backward (fp32 additions).
 * Supported: act = MMDIT_BF16, gemm = MMDIT_GEMM_NATIVE, batch <= 8, mlp_hidden % 32 == 0; the
 * double block needs both streams non-empty.  A precomputed `mod` in the weights is ignored.
 * Arguments otherwise as for the forward entry points. */
typedef struct mmdit_stream_grads {
  float *w_mod, *b_mod;
  float *w_qkv, *b_qkv;
  float *g_q, *g_k;
  float *w_o, *b_o;
  float *w_1, *b_1;
  float *w_2, *b_2;
} mmdit_stream_grads;
size_t mmdit_double_block_bwd_workspace_size(const mmdit_dims *dims);
mmdit_status mmdit_double_block_bwd(const mmdit_dims *dims, const mmdit_stream_w *w_img,
                                    const mmdit_stream_w *w_txt, const void *vec,
                                    const float *rope_cos, const float *rope_sin,
                                    const void *x_img, const void *x_txt, const void *dy_img,
                                    const void *dy_txt, void *dx_img, void *dx_txt, float *dvec,
                                    const mmdit_stream_grads *g_img,
                                    const mmdit_stream_grads *g_txt, void *workspace,
                                    size_t workspace_bytes, void *stream);
size_t mmdit_single_block_bwd_workspace_size(const mmdit_dims *dims);
mmdit_status mmdit_single_block_bwd(const mmdit_dims *dims, const mmdit_stream_w *w,
                                    const void *vec, const float *rope_cos,
                                    const float *rope_sin, const void *x, const void *dy,
                                    void *dx, float *dvec, const mmdit_stream_grads *g,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* Training pair: the same backward split in two calls, so that a training step runs the forward
 * once.  mmdit_*_block_fwd_train computes the block's outputs y (as mmdit_*_block_fwd would, from
 * the same kernels) and leaves in `saved` (a buffer of mmdit_*_block_bwd_workspace_size bytes,
 * owned by the caller) everything the backward reads; mmdit_*_block_bwd_saved then writes the
 * gradients exactly as mmdit_*_block_bwd does, without recomputing the forward.  Between the two
 * calls `saved` must not be touched, and the dims, weights, vec, RoPE tables and inputs x must be
 * the same (the backward reads x again).  The backward consumes `saved`: a second backward needs
 * a new forward.  Checks and supported shapes as for mmdit_*_block_bwd; y is of type `act` with
 * the forward's layout. */
mmdit_status mmdit_double_block_fwd_train(const mmdit_dims *dims, const mmdit_stream_w *w_img,
                                          const mmdit_stream_w *w_txt, const void *vec,
                                          const float *rope_cos, const float *rope_sin,
                                          const void *x_img, const void *x_txt, void *y_img,
                                          void *y_txt, void *saved, size_t saved_bytes, void *stream);
mmdit_status mmdit_double_block_bwd_saved(const mmdit_dims *dims, const mmdit_stream_w *w_img,
                                          const mmdit_stream_w *w_txt, const void *vec,
                                          const float *rope_cos, const float *rope_sin,
                                          const void *x_img, const void *x_txt, const void *dy_img,
                                          const void *dy_txt, void *dx_img, void *dx_txt,
                                          float *dvec, const mmdit_stream_grads *g_img,
                                          const mmdit_stream_grads *g_txt, void *saved,
                                          size_t saved_bytes, void *stream);
mmdit_status mmdit_single_block_fwd_train(const mmdit_dims *dims, const mmdit_stream_w *w,
                                          const void *vec, const float *rope_cos,
                                          const float *rope_sin, const void *x, void *y, void *saved,
                                          size_t saved_bytes, void *stream);
mmdit_status mmdit_single_block_bwd_saved(const mmdit_dims *dims, const mmdit_stream_w *w,
                                          const void *vec, const float *rope_cos,
                                          const float *rope_sin, const void *x, const void *dy,
                                          void *dx, float *dvec, const mmdit_stream_grads *g,
                                          void *saved, size_t saved_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Many modulations in one launch: the AdaLN modulation of mmdit_modulation_fwd for every job
 * in `jobs` (every block of a model, which all read the same vec), out_j[b, r] =
 * sum_k SiLU(vec[b, k]) w_j[r, k] + b_j[r].  The weight traffic is the whole cost, so one
 * launch streams all of it at the HBM rate instead of one short launch per block.
 *   vec [batch, dim] of type `act`; each job: w [rows, dim], b [rows] (may be NULL) of type
 *   `act`, out [batch, rows] fp32 (16-byte aligned); jobs is a host array of n_jobs entries.
 * dim a multiple of 8, at most 6144.  No workspace. */
typedef struct mmdit_gemv_job {
  const void *w, *b;
  float *out;
  int32_t rows;
} mmdit_gemv_job;
mmdit_status mmdit_modulation_batched_fwd(int32_t act, int32_t batch, int32_t dim, const void *vec,
                                          int32_t n_jobs, const mmdit_gemv_job *jobs, void *stream);

/* ---------------------------------------------------------------------------------------
 * Conditioning vector ([ARCH] §Model components, 1. Input embeddings, Conditioning; [API]
 * §Components API, Embeddings, TimeStepEmbedder and MLPEmbedder):
 *   vec = MLP_t(sinusoid(1000 t)) + MLP_y(y) [+ g w_g + b_g]
 * sinusoid(tau)[b] = [cos(tau f_0 .. f_{h-1}), sin(tau f_0 .. f_{h-1})], f_k = 10000^(-k/h),
 * h = time_dim / 2 (the pages print no formula: a reading); MLP(x) = Linear2(SiLU(Linear1(x)));
 * the optional guidance term is a Linear of the scalar guidance scale.
 *   t [batch] fp32 in [0, 1]; y [batch, vec_in_dim] (pooled text vector) of type `act`;
 *   guidance [batch] fp32 or NULL (then w_guidance, b_guidance are not read);
 *   weights of type `act`: time_in.w1 [D, time_dim], vector_in.w1 [D, vec_in_dim],
 *   *.w2 [D, D], biases [D], w_guidance and b_guidance [D]; vec [batch, D] of type `act`.
 * time_dim even, at most 512; time_dim, vec_in_dim and D multiples of 8, at most 6144.
 * workspace >= mmdit_conditioning_workspace_size(). */
typedef struct mmdit_mlp_embedder_w {
  const void *w1, *b1; /* [D, in_dim], [D] */
  const void *w2, *b2; /* [D, D], [D] */
} mmdit_mlp_embedder_w;
typedef struct mmdit_cond_w {
  mmdit_mlp_embedder_w time_in;   /* in_dim = time_dim (256) */
  mmdit_mlp_embedder_w vector_in; /* in_dim = vec_in_dim (768) */
  const void *w_guidance, *b_guidance;
} mmdit_cond_w;
size_t mmdit_conditioning_workspace_size(int32_t act, int32_t batch, int32_t hidden, int32_t time_dim);
mmdit_status mmdit_conditioning_fwd(int32_t act, int32_t batch, int32_t hidden, int32_t time_dim,
                                    int32_t vec_in_dim, const mmdit_cond_w *w, const float *t,
                                    const void *y, const float *guidance, void *vec,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * The whole model forward ([ARCH] §Data flow, Complete forward pass; §Overview, Model
 * variants: Flux 12B has 19 double and 38 single blocks):
 *   vec = conditioning(t, y, guidance); x_img = img_in(z_t); x_txt = txt_in(txt);
 *   n_double double blocks on (x_img, x_txt); c = [x_img; x_txt];
 *   n_single single blocks on c; pred = output head on the image rows of c.
 * Every block's modulation is computed up front in one launch (they all read vec).
 *   cfg->block: the block dims (seq_img = lat_h * lat_w, gemm = MMDIT_GEMM_NATIVE);
 *   z_t [batch, channels, lat_h, lat_w] fp32; txt [batch, seq_txt, txt_dim] of type `act`;
 *   t, guidance, y as for mmdit_conditioning_fwd; rope_cos, rope_sin [batch, seq, 64] fp32 as
 *   rope3d_freqs writes them for the joint [image; text] ids; pred like z_t.
 *   w->double_img, double_txt: host arrays of n_double stream weights; w->single: host array
 *   of n_single (their `mod` fields are ignored: the call computes every modulation).
 * workspace >= mmdit_flux_workspace_size(cfg); a bounded-wait timeout in any step is reported
 * by mmdit_workspace_status on that workspace. */
typedef struct mmdit_flux_config {
  mmdit_dims block;
  int32_t n_double, n_single;
  int32_t lat_h, lat_w, channels; /* latent grid and channels (64) */
  int32_t txt_dim;                /* text embedding width (4096) */
  int32_t time_dim, vec_in_dim;   /* 256, 768 */
  int32_t single_parallel;        /* 0: sequential single blocks (six modulation chunks);
                                     1: parallel-branch single blocks as in
                                     mmdit_single_block_parallel_fwd (w_mod [3D, D]) */
} mmdit_flux_config;
typedef struct mmdit_flux_w {
  const void *w_img_in, *b_img_in; /* [D, channels], [D] */
  const void *w_txt_in, *b_txt_in; /* [D, txt_dim], [D] */
  mmdit_cond_w cond;
  const mmdit_stream_w *double_img, *double_txt, *single;
  const void *w_ada, *b_ada;       /* output head: [2D, D], [2D] */
  const void *w_out, *b_out;       /* [channels, D], [channels] */
} mmdit_flux_w;
size_t mmdit_flux_workspace_size(const mmdit_flux_config *cfg);
mmdit_status mmdit_flux_forward(const mmdit_flux_config *cfg, const mmdit_flux_w *w, const float *z_t,
                                const void *txt, const float *t, const void *y,
                                const float *guidance, const float *rope_cos, const float *rope_sin,
                                float *pred, void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MMDIT_H_ */
