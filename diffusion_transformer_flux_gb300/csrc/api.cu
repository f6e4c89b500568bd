// api.cu -- the C ABI of libmmdit.so (declared in include/mmdit.h): argument validation,
// workspace planning and the launch sequences of each entry point.  No device memory is
// allocated here; every buffer comes from the caller.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <array>
#include <initializer_list>
#include <vector>

#include "../../include/mmdit.h"
#include "internal.h"

namespace mmdit {

namespace {
thread_local char g_err[512] = "no error";
thread_local uint64_t g_launches = 0;

mmdit_status fail(mmdit_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

mmdit_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MMDIT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
constexpr int kColsumChunks = 128;  // row chunks of the bias-gradient column sums
size_t elt_bytes(int act) { return act == MMDIT_BF16 ? 2 : 4; }

// Sequential 256-byte-aligned carving of a workspace.
struct Carver {
  size_t off = kStatusBytes;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  }
};

}  // namespace

void count_launch(int n) { g_launches += static_cast<uint64_t>(n); }

namespace {
thread_local bool g_pdl_armed = false;
}
void pdl_begin_call() { g_pdl_armed = false; }
bool pdl_next_launch() {
  const bool armed = g_pdl_armed;
  g_pdl_armed = true;
  return armed;
}

int set_last_error(int status, const char* msg) {
  return static_cast<int>(fail(static_cast<mmdit_status>(status), "%s", msg));
}

// ----------------------------------------------------------------------------- step timing
namespace {
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
thread_local bool g_prof_on = false;
thread_local ProfRecord* g_prof = nullptr;
thread_local int g_prof_n = 0, g_prof_cap = 0;

// Brackets one library step with events on `stream` when profiling is enabled.
struct ProfScope {
  ProfRecord* rec = nullptr;
  cudaStream_t stream;
  ProfScope(const char* name, cudaStream_t s) : stream(s) {
    if (!g_prof_on) return;
    if (g_prof_n == g_prof_cap) {
      const int cap = g_prof_cap ? 2 * g_prof_cap : 256;
      ProfRecord* n = static_cast<ProfRecord*>(realloc(g_prof, cap * sizeof(ProfRecord)));
      if (!n) return;
      g_prof = n, g_prof_cap = cap;
    }
    ProfRecord r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess) return;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
      cudaEventDestroy(r.start);
      return;
    }
    g_prof[g_prof_n] = r;
    rec = &g_prof[g_prof_n++];
    cudaEventRecord(rec->start, stream);
  }
  ~ProfScope() {
    if (rec) cudaEventRecord(rec->stop, stream);
  }
};
}  // namespace

// SM count of the current device; without a device (size queries on a host-only machine) the
// GB300 count, so that workspace sizes do not depend on whether a GPU is visible.
constexpr int kDefaultSms = 152;
int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kDefaultSms;
  }
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return kDefaultSms;
    }
    cached[dev] = n > 0 ? n : kDefaultSms;
  }
  return cached[dev];
}

namespace {
// Per-thread cache of encoded tensor maps.  A map depends only on the arguments below, so a
// cached copy stays valid for as long as the same (address, shape) pair is passed again.
struct TmapKey {
  int32_t dtype, rank, swizzle, pad;
  const void* base;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box[5];
  uint32_t pad2;
};
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kTmapCache = 128;
thread_local TmapEntry g_tmap_cache[kTmapCache];
thread_local int g_tmap_next = 0;
}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  TmapKey key;
  memset(&key, 0, sizeof(key));
  key.dtype = static_cast<int32_t>(dtype), key.rank = rank, key.swizzle = static_cast<int32_t>(swizzle);
  key.base = base;
  for (int i = 0; i < rank && i < 5; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (int i = 0; i < rank - 1 && i < 4; ++i) key.strides[i] = strides_bytes[i];
  for (int i = 0; i < kTmapCache; ++i)
    if (g_tmap_cache[i].used && memcmp(&g_tmap_cache[i].key, &key, sizeof(key)) == 0) {
      *map = g_tmap_cache[i].map;
      return true;
    }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) d[i] = dims[i], b[i] = box[i], e[i] = 1;
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  if (fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, e,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmapEntry& slot = g_tmap_cache[g_tmap_next];
  g_tmap_next = (g_tmap_next + 1) % kTmapCache;
  slot.key = key, slot.map = *map, slot.used = true;
  return true;
}

// ----------------------------------------------------------------------------- block planning
struct BlockPlan {
  bool single;
  bool parallel = false;  // single block with parallel branches: one LayerNorm feeds QKV and fc1
  int mod_chunks = 6;     // modulation chunks per stream: 6, or 3 (shift, scale, gate) when parallel
  bool fp8;  // E4M3 linears: h, u hold E4M3 codes; o8 and wq hold the cast attention output
             // and weights
  bool fp8_current = false;  // tensorwise or blockwise (current) scaling: inputs staged in bf16 before their cast
  bool fp8_blockwise = false;  // blockwise: per-tile scales (bw_sx, bw_sw), the blockwise GEMM
  bool fp8_mx = false;  // MXFP8: bf16 operands holding the MX-represented values; wq holds the weights' (bf16)
  int B, Si, St, S, S_pad, D, H, F;
  size_t elt;
  size_t mod[2], h[2], q, k, vt, o[2], x1[2], u[2];
  size_t o8[2], wq[2], stage[2];
  size_t bw_sx[2], bw_sw[2];  // blockwise: the current input's s_x [K/128, rows]; the weights' s_w
  size_t total;
  // byte offsets of the four weights inside a stream's wq slot
  size_t wq_qkv() const { return 0; }
  size_t wq_o() const { return static_cast<size_t>(3) * D * D; }
  size_t wq_1() const { return static_cast<size_t>(4) * D * D; }
  size_t wq_2() const { return static_cast<size_t>(4) * D * D + static_cast<size_t>(F) * D; }
  size_t wq_bytes() const { return static_cast<size_t>(4) * D * D + static_cast<size_t>(2) * F * D; }
  // byte offsets of the four weights' s_w [N/128, K/128] inside a stream's bw_sw slot
  size_t sw_qkv() const { return 0; }
  size_t sw_o() const { return static_cast<size_t>(3 * D / 128) * (D / 128) * 4; }
  size_t sw_1() const { return sw_o() + static_cast<size_t>(D / 128) * (D / 128) * 4; }
  size_t sw_2() const { return sw_1() + static_cast<size_t>(F / 128) * (D / 128) * 4; }
  size_t sw_bytes() const { return sw_2() + static_cast<size_t>(D / 128) * (F / 128) * 4; }
};

static bool plan_block(const mmdit_dims* d, bool single, BlockPlan* p) {
  if (!d) return false;
  p->single = single;
  p->B = d->batch, p->Si = d->seq_img, p->St = d->seq_txt;
  p->S = d->seq_img + d->seq_txt;
  p->S_pad = static_cast<int>(round_up(static_cast<size_t>(p->S), 8));
  p->D = d->hidden, p->H = d->heads, p->F = d->mlp_hidden;
  p->elt = elt_bytes(d->act);
  p->fp8 = d->gemm == MMDIT_GEMM_FP8_E4M3 || d->gemm == MMDIT_GEMM_FP8_TENSORWISE ||
           d->gemm == MMDIT_GEMM_FP8_BLOCKWISE;
  p->fp8_blockwise = d->gemm == MMDIT_GEMM_FP8_BLOCKWISE;
  p->fp8_current = d->gemm == MMDIT_GEMM_FP8_TENSORWISE || p->fp8_blockwise;
  p->fp8_mx = d->gemm == MMDIT_GEMM_FP8_MXFP8;
  const size_t mm_elt = p->fp8 ? 1 : p->elt;  // inputs of the QKV and fc1/fc2 linears
  Carver c;
  const size_t B = p->B, D = p->D, F = p->F, S = p->S;
  const size_t rows[2] = {B * (single ? S : static_cast<size_t>(p->Si)),
                          single ? 0 : B * static_cast<size_t>(p->St)};
  const int ns = single ? 1 : 2;
  for (int s = 0; s < 2; ++s) p->mod[s] = s < ns ? c.take(B * 6 * D * 4) : 0;
  for (int s = 0; s < 2; ++s) p->h[s] = s < ns ? c.take(rows[s] * D * mm_elt) : 0;
  p->q = c.take(B * D * S * 2);
  p->k = c.take(B * D * S * 2);
  p->vt = c.take(B * D * static_cast<size_t>(p->S_pad) * 2);
  for (int s = 0; s < 2; ++s) p->o[s] = s < ns ? c.take(rows[s] * D * p->elt) : 0;
  // the in-block residual x1 stays fp32 so the output is rounded to the activation type once
  for (int s = 0; s < 2; ++s) p->x1[s] = s < ns ? c.take(rows[s] * D * 4) : 0;
  for (int s = 0; s < 2; ++s) p->u[s] = s < ns ? c.take(rows[s] * F * mm_elt) : 0;
  for (int s = 0; s < 2; ++s) p->o8[s] = p->fp8 && s < ns ? c.take(rows[s] * D) : 0;
  // E4M3 weight codes, or (MXFP8) the weights' represented values in bf16
  for (int s = 0; s < 2; ++s)
    p->wq[s] = (p->fp8 || p->fp8_mx) && s < ns ? c.take(p->wq_bytes() * (p->fp8_mx ? 2 : 1)) : 0;
  // tensorwise: a linear's bf16 input (LayerNorm-modulate output or GELU output) before its cast
  for (int s = 0; s < 2; ++s)
    p->stage[s] = p->fp8_current && s < ns ? c.take(rows[s] * (F > D ? F : D) * 2) : 0;
  for (int s = 0; s < 2; ++s) {
    p->bw_sx[s] = p->fp8_blockwise && s < ns ? c.take(rows[s] * ((F > D ? F : D) / 128) * 4) : 0;
    p->bw_sw[s] = p->fp8_blockwise && s < ns ? c.take(p->sw_bytes()) : 0;
  }
  p->total = c.off;
  return true;
}

static mmdit_status check_dims(const mmdit_dims* d) {
  if (!d) return fail(MMDIT_ERR_INVALID_ARG, "dims is NULL");
  if (d->batch < 1 || d->seq_img < 0 || d->seq_txt < 0 || d->seq_img + d->seq_txt < 1)
    return fail(MMDIT_ERR_INVALID_ARG, "bad batch/sequence sizes (B=%d, S_i=%d, S_t=%d)", d->batch,
                d->seq_img, d->seq_txt);
  if (d->act != MMDIT_F32 && d->act != MMDIT_BF16)
    return fail(MMDIT_ERR_INVALID_ARG, "act must be MMDIT_F32 or MMDIT_BF16 (got %d)", d->act);
  if (d->gemm != MMDIT_GEMM_NATIVE && d->gemm != MMDIT_GEMM_FP8_E4M3 && d->gemm != MMDIT_GEMM_FP8_TENSORWISE &&
      d->gemm != MMDIT_GEMM_FP8_BLOCKWISE && d->gemm != MMDIT_GEMM_FP8_MXFP8)
    return fail(MMDIT_ERR_INVALID_ARG, "unknown gemm mode %d", d->gemm);
  if (d->gemm != MMDIT_GEMM_NATIVE && d->act != MMDIT_BF16)
    return fail(MMDIT_ERR_UNSUPPORTED, "FP8 E4M3 linears need bf16 activations (act = MMDIT_BF16)");
  if (d->gemm != MMDIT_GEMM_NATIVE && d->mlp_hidden % 128 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "FP8 E4M3 linears need mlp_hidden %% 128 == 0 (got %d)",
                d->mlp_hidden);
  if (d->head_dim != 128)
    return fail(MMDIT_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", d->head_dim);
  if (d->hidden > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "hidden must be at most 6144 (got %d)", d->hidden);
  if (d->heads < 1 || d->heads * d->head_dim != d->hidden)
    return fail(MMDIT_ERR_INVALID_ARG, "heads * head_dim (%d * %d) != hidden (%d)", d->heads,
                d->head_dim, d->hidden);
  if (d->mlp_hidden < 64 || d->mlp_hidden % 64 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "mlp_hidden must be a positive multiple of 64 (got %d)",
                d->mlp_hidden);
  if (!(d->ln_eps >= 0.f) || !(d->rms_eps >= 0.f))
    return fail(MMDIT_ERR_INVALID_ARG, "eps must be non-negative");
  return MMDIT_OK;
}

static mmdit_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
  int i = 0;
  for (const void* p : ptrs) {
    if (!p) return fail(MMDIT_ERR_INVALID_ARG, "%s: pointer %d is NULL", what, i);
    if (!aligned16(p)) return fail(MMDIT_ERR_INVALID_ARG, "%s: pointer %d is not 16-byte aligned", what, i);
    ++i;
  }
  return MMDIT_OK;
}

static mmdit_status check_stream_w(const mmdit_stream_w* w, const char* what) {
  if (!w) return fail(MMDIT_ERR_INVALID_ARG, "%s: weight set is NULL", what);
  if (w->mod && !aligned16(w->mod))
    return fail(MMDIT_ERR_INVALID_ARG, "%s: precomputed modulation is not 16-byte aligned", what);
  return check_ptrs({w->w_mod, w->b_mod, w->w_qkv, w->b_qkv, w->g_q, w->g_k, w->w_o, w->b_o, w->w_1,
                     w->b_1, w->w_2, w->b_2},
                    what);
}

static mmdit_status check_workspace(void* ws, size_t have, size_t need) {
  if (!ws) return fail(MMDIT_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MMDIT_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (have < need)
    return fail(MMDIT_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", have, need);
  return MMDIT_OK;
}

// Tensors of the FP8 state a block uses: per stream slot (0 image / single, 1 text), linear g
// (0 QKV, 1 output projection, 2 fc1, 3 fc2) and operand (0 input, 1 weight), index
// 8 * slot + 2 * g + operand.
constexpr int kFp8TensorsPerStream = 8;
inline int fp8_tensor(int slot, int g, int operand) { return kFp8TensorsPerStream * slot + 2 * g + operand; }

static mmdit_status check_fp8(const mmdit_dims* d, const mmdit_fp8_state* f, int n_needed) {
  if (d->gemm == MMDIT_GEMM_NATIVE) {
    if (f) return fail(MMDIT_ERR_INVALID_ARG, "fp8 state given but the gemm mode is native");
    return MMDIT_OK;
  }
  if (d->gemm == MMDIT_GEMM_FP8_BLOCKWISE || d->gemm == MMDIT_GEMM_FP8_MXFP8) {
    // every scale is the call's own per-tile or per-block scale: there is no state to read or record
    if (f) return fail(MMDIT_ERR_INVALID_ARG, "fp8 state given but the %s recipe keeps none",
                       d->gemm == MMDIT_GEMM_FP8_MXFP8 ? "MXFP8" : "blockwise");
    return MMDIT_OK;
  }
  if (!f) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linears need an fp8 state (got NULL)");
  if (!f->amax_history || !f->scale)
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: NULL amax_history or scale");
  if ((reinterpret_cast<uintptr_t>(f->amax_history) & 3u) || (reinterpret_cast<uintptr_t>(f->scale) & 3u))
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: arrays must be 4-byte aligned");
  if (f->hist_len < 1 || f->pos < 0 || f->pos >= f->hist_len)
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: need hist_len >= 1 and 0 <= pos < hist_len (got %d, %d)",
                f->hist_len, f->pos);
  if (f->n_tensors < n_needed)
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: %d tensors given, this block records %d",
                f->n_tensors, n_needed);
  if (f->amax_compute_algo != 0 && f->amax_compute_algo != 1)
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: amax_compute_algo must be 0 (most_recent) or 1 (max), got %d",
                f->amax_compute_algo);
  if (f->margin < 0 || f->margin > 16)
    return fail(MMDIT_ERR_INVALID_ARG, "fp8 state: margin must be in [0, 16] (got %d)", f->margin);
  return MMDIT_OK;
}

#define MMDIT_CUDA(call, what)                       \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Split-K factor for a narrow GEMM (few output tiles, long K): enough work items to cover the
// SMs, at least 4 K slices per item, never an empty split.
static int choose_splits(int M, int N, int K, int elt_bytes) {
  const int bn = N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : (N % 64 == 0 ? 64 : 32));
  const int tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
  const int kb = (K * elt_bytes + 127) / 128;
  if (tiles * 2 > num_sms() || kb < 8) return 1;
  int s = num_sms() / tiles;
  if (s > kb / 4) s = kb / 4;
  if (s > 8) s = 8;
  if (s < 2) return 1;
  const int per = (kb + s - 1) / s;
  return (kb + per - 1) / per;  // every split gets at least one K slice
}

}  // namespace mmdit

using namespace mmdit;

namespace {

uint32_t* status_word(void* ws) { return static_cast<uint32_t*>(ws); }
template <typename T = uint8_t>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Launches the chain of one block over stream s (double block: s = 0 image, 1 text).
// The streams a block call runs: the image and text streams of a double block (each only if
// it has rows), or the single block's one stream over the joint sequence.  Each GEMM of the
// block is one launch over all of them (equal N and K, per-stream operands and epilogues).
struct Streams {
  int n = 0;
  int s[2] = {0, 0};  // plan slot: 0 image / single, 1 text
  const mmdit_stream_w* w[2] = {nullptr, nullptr};
  const void* x[2] = {nullptr, nullptr};
  void* y[2] = {nullptr, nullptr};
  int rpb[2] = {0, 0};  // rows per batch element
  const float* mod[2] = {nullptr, nullptr};  // [B, 6D] modulation (precomputed or in the workspace)
  // the backward's recomputation: where the linears' outputs before their norm, GELU or gate go
  // (null in the forward)
  void* pre_qkv[2] = {nullptr, nullptr};
  void* pre_o[2] = {nullptr, nullptr};
  void* pre_1[2] = {nullptr, nullptr};
  void* pre_2[2] = {nullptr, nullptr};
};

// The FP8 state of one block call (f == nullptr when the linears are not FP8): where each
// tensor's scale is read and where this call records its amax.
struct Fp8 {
  const mmdit_fp8_state* f = nullptr;
  bool current = false;  // tensorwise or blockwise: every scale from the tensor's own amax in this call
  bool blockwise = false;  // per-tile scales in the plan's bw_sx / bw_sw slots; no state (f == nullptr)
  bool mx = false;  // MXFP8: every linear input and weight replaced by its MX-represented values (bf16)
  int n_tensors = 0;     // tensors this block records (16 double, 8 single)
  bool on() const { return f != nullptr || blockwise; }  // the linears run on E4M3 codes
  const float* scale(int t) const { return f->scale + t; }
  float* amax(int t) const { return f->amax_history + static_cast<size_t>(t) * f->hist_len + f->pos; }
};

// Current (tensorwise) scaling of bf16 tensors about to be cast: record each one's amax (a first
// pass that casts nothing), turn the recorded amax into scales (448 / amax / 2^margin), then cast
// with them.  The cast records the same amax again.
mmdit_status fp8_cast_current(const Fp8& f8, const QuantJob* jobs, int n, cudaStream_t st, const char* what) {
  QuantJob amax_only[kQuantMaxJobs];
  for (int i = 0; i < n; ++i) amax_only[i] = jobs[i], amax_only[i].dst = nullptr;
  MMDIT_CUDA(launch_quantize_e4m3(amax_only, n, st), what);
  MMDIT_CUDA(launch_scale_update(f8.f->amax_history, f8.f->scale, f8.f->hist_len, f8.n_tensors, f8.f->pos,
                                 f8.f->margin, 0, st),
             what);
  MMDIT_CUDA(launch_quantize_e4m3(jobs, n, st), what);
  return MMDIT_OK;
}

// MXFP8: replace each stream's bf16 tensor [rows, K] at plan offset `off` by its MX-represented
// values, in place (one launch for the streams).
mmdit_status mx_in_place(const BlockPlan& p, const Streams& ss, const size_t* off, int K, void* ws, cudaStream_t st,
                         const char* what) {
  MxJob jobs[2];
  for (int i = 0; i < ss.n; ++i) {
    __nv_bfloat16* t = at<__nv_bfloat16>(ws, off[ss.s[i]]);
    jobs[i].src = t, jobs[i].deq = t, jobs[i].rows = static_cast<int64_t>(p.B) * ss.rpb[i], jobs[i].K = K;
  }
  MMDIT_CUDA(launch_mx_cast(jobs, ss.n, st), what);
  return MMDIT_OK;
}

void add_problem(GemmProblem& g, int i, int M, const void* A, const void* W, const EpiArgs& ep) {
  if (i == 0)
    g.M = M, g.A = A, g.W = W, g.ep = ep;
  else
    g.M1 = M, g.A1 = A, g.W1 = W, g.ep1 = ep;
}

mmdit_status run_qkv(const mmdit_dims* d, const BlockPlan& p, const Streams& ss, const float* cs,
                     const float* sn, const Fp8& f8, void* ws, cudaStream_t st) {
  {
    ProfScope ps_(p.single ? "single.ln1" : "double.ln1", st);
    LnModJob jobs[2];
    for (int i = 0; i < ss.n; ++i) {
      const float* mod = ss.mod[i];
      // tensorwise: the bf16 output is staged, then cast once its amax is known
      void* out = f8.current ? at(ws, p.stage[ss.s[i]]) : at(ws, p.h[ss.s[i]]);
      jobs[i] = {ss.x[i], mod, mod + p.D, static_cast<int64_t>(p.mod_chunks) * p.D, out,
                 p.B * ss.rpb[i], ss.rpb[i]};
      if (f8.on() && !f8.current) {
        const int t = fp8_tensor(ss.s[i], 0, 0);
        jobs[i].q_scale = f8.scale(t), jobs[i].q_amax = f8.amax(t);
      }
    }
    MMDIT_CUDA(launch_ln_modulate2(d->act, d->act == MMDIT_F32, jobs, ss.n, p.D, d->ln_eps, st,
                                   f8.on() && !f8.current ? 1 : 0),
               "LayerNorm-modulate (attention branch)");
  }
  if (f8.mx) {
    ProfScope ps_(p.single ? "single.fp8_cast_h1" : "double.fp8_cast_h1", st);
    mmdit_status s = mx_in_place(p, ss, p.h, p.D, ws, st, "MXFP8 cast of the QKV input");
    if (s != MMDIT_OK) return s;
  } else if (f8.blockwise) {
    ProfScope ps_(p.single ? "single.fp8_cast_h1" : "double.fp8_cast_h1", st);
    for (int i = 0; i < ss.n; ++i)
      MMDIT_CUDA(launch_blockwise_cast_act(at<__nv_bfloat16>(ws, p.stage[ss.s[i]]), p.B * ss.rpb[i], p.D,
                                           at<uint8_t>(ws, p.h[ss.s[i]]), at<float>(ws, p.bw_sx[ss.s[i]]), st),
                 "blockwise E4M3 cast of the QKV input");
  } else if (f8.current) {
    ProfScope ps_(p.single ? "single.fp8_cast_h1" : "double.fp8_cast_h1", st);
    QuantJob q[2];
    for (int i = 0; i < ss.n; ++i) {
      const int t = fp8_tensor(ss.s[i], 0, 0);
      q[i] = {at<__nv_bfloat16>(ws, p.stage[ss.s[i]]), at<uint8_t>(ws, p.h[ss.s[i]]),
              static_cast<int64_t>(p.B) * ss.rpb[i] * p.D, f8.scale(t), f8.amax(t)};
    }
    mmdit_status s = fp8_cast_current(f8, q, ss.n, st, "E4M3 cast of the QKV input (current scaling)");
    if (s != MMDIT_OK) return s;
  }
  GemmProblem g;
  g.act = f8.on() ? 2 : d->act, g.epi = kEpiQkv, g.N = 3 * p.D, g.K = p.D;
  for (int i = 0; i < ss.n; ++i) {
    const mmdit_stream_w* w = ss.w[i];
    EpiArgs e;
    const void* wmat = w->w_qkv;
    if (f8.mx) {
      wmat = at(ws, p.wq[ss.s[i]] + 2 * p.wq_qkv());
    } else if (f8.blockwise) {
      e.bw_sx = at<float>(ws, p.bw_sx[ss.s[i]]), e.bw_sw = at<float>(ws, p.bw_sw[ss.s[i]] + p.sw_qkv());
      wmat = at(ws, p.wq[ss.s[i]] + p.wq_qkv());
    } else if (f8.f) {
      e.scale_a = f8.scale(fp8_tensor(ss.s[i], 0, 0)), e.scale_w = f8.scale(fp8_tensor(ss.s[i], 0, 1));
      wmat = at(ws, p.wq[ss.s[i]] + p.wq_qkv());
    }
    e.bias = w->b_qkv, e.g_q = w->g_q, e.g_k = w->g_k;
    e.rope_cos = cs, e.rope_sin = sn;
    e.q = at<__nv_bfloat16>(ws, p.q), e.k = at<__nv_bfloat16>(ws, p.k);
    e.vt = at<__half>(ws, p.vt);
    e.rows_per_batch = ss.rpb[i];
    e.seq_offset = ss.s[i] == 0 ? 0 : p.Si;
    e.seq_joint = p.S, e.seq_pad = p.S_pad, e.heads = p.H, e.hidden = p.D;
    e.rms_eps = d->rms_eps, e.rope_interleaved = d->rope_interleaved ? 1 : 0;
    e.pre = ss.pre_qkv[i];
    add_problem(g, i, p.B * ss.rpb[i], at(ws, p.h[ss.s[i]]), wmat, e);
  }
  ProfScope ps_(p.single ? "single.qkv" : "double.qkv", st);
  MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "QKV projection");
  return MMDIT_OK;
}

mmdit_status run_post(const mmdit_dims* d, const BlockPlan& p, const Streams& ss, const Fp8& f8,
                      void* ws, cudaStream_t st) {
  // the linears' operand type, and each stream's weight matrices as the GEMMs read them
  const int mm = f8.on() ? 2 : d->act;
  auto weight = [&](int i, int g) -> const void* {
    const mmdit_stream_w* w = ss.w[i];
    if (!f8.on() && !f8.mx) return g == 1 ? w->w_o : (g == 2 ? w->w_1 : w->w_2);
    const size_t off = g == 1 ? p.wq_o() : (g == 2 ? p.wq_1() : p.wq_2());
    return at(ws, p.wq[ss.s[i]] + (f8.mx ? 2 : 1) * off);
  };
  auto dequant = [&](EpiArgs& e, int i, int g) {
    if (f8.blockwise) {
      const size_t off = g == 1 ? p.sw_o() : (g == 2 ? p.sw_1() : p.sw_2());
      e.bw_sx = at<float>(ws, p.bw_sx[ss.s[i]]), e.bw_sw = at<float>(ws, p.bw_sw[ss.s[i]] + off);
      return;
    }
    if (!f8.f) return;
    e.scale_a = f8.scale(fp8_tensor(ss.s[i], g, 0)), e.scale_w = f8.scale(fp8_tensor(ss.s[i], g, 1));
  };
  // blockwise: a bf16 input cast per 1 x 128 tile, its scales into the stream's bw_sx slot
  auto cast_blockwise = [&](int i, const void* src, size_t dst, int K, const char* what) -> mmdit_status {
    MMDIT_CUDA(launch_blockwise_cast_act(static_cast<const __nv_bfloat16*>(src), p.B * ss.rpb[i], K,
                                         at<uint8_t>(ws, dst), at<float>(ws, p.bw_sx[ss.s[i]]), st),
               what);
    return MMDIT_OK;
  };
  if (f8.mx) {
    ProfScope ps_(p.single ? "single.fp8_cast_o" : "double.fp8_cast_o", st);
    mmdit_status s = mx_in_place(p, ss, p.o, p.D, ws, st, "MXFP8 cast of the attention output");
    if (s != MMDIT_OK) return s;
  } else if (f8.blockwise) {
    ProfScope ps_(p.single ? "single.fp8_cast_o" : "double.fp8_cast_o", st);
    for (int i = 0; i < ss.n; ++i) {
      mmdit_status s = cast_blockwise(i, at(ws, p.o[ss.s[i]]), p.o8[ss.s[i]], p.D,
                                      "blockwise E4M3 cast of the attention output");
      if (s != MMDIT_OK) return s;
    }
  } else if (f8.f) {
    // the attention output (bf16) cast to E4M3 for the output projection
    ProfScope ps_(p.single ? "single.fp8_cast_o" : "double.fp8_cast_o", st);
    QuantJob jobs[2];
    for (int i = 0; i < ss.n; ++i) {
      const int t = fp8_tensor(ss.s[i], 1, 0);
      jobs[i] = {at<__nv_bfloat16>(ws, p.o[ss.s[i]]), at<uint8_t>(ws, p.o8[ss.s[i]]),
                 static_cast<int64_t>(p.B) * ss.rpb[i] * p.D, f8.scale(t), f8.amax(t)};
    }
    if (f8.current) {
      mmdit_status s = fp8_cast_current(f8, jobs, ss.n, st, "E4M3 cast of the attention output (current scaling)");
      if (s != MMDIT_OK) return s;
    } else {
      MMDIT_CUDA(launch_quantize_e4m3(jobs, ss.n, st), "E4M3 cast of the attention output");
    }
  }
  GemmProblem g;
  g.act = mm, g.epi = kEpiGateResid, g.N = p.D, g.K = p.D;
  for (int i = 0; i < ss.n; ++i) {
    const float* mod = ss.mod[i];
    EpiArgs e;
    e.bias = ss.w[i]->b_o, e.resid = ss.x[i], e.gate = mod + 2 * p.D,
    e.gate_bstride = static_cast<int64_t>(p.mod_chunks) * p.D;
    e.rows_per_batch = ss.rpb[i], e.out = at(ws, p.x1[ss.s[i]]), e.out_f32 = 1;
    e.pre = ss.pre_o[i];
    dequant(e, i, 1);
    add_problem(g, i, p.B * ss.rpb[i], at(ws, f8.on() ? p.o8[ss.s[i]] : p.o[ss.s[i]]), weight(i, 1), e);
  }
  {
    ProfScope ps_(p.single ? "single.out" : "double.out", st);
    MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "attention output projection");
  }
  if (!p.parallel) {
    // (the parallel block's fc1 reads the attention branch's LayerNorm output, still in h)
    ProfScope ps_(p.single ? "single.ln2" : "double.ln2", st);
    LnModJob jobs[2];
    for (int i = 0; i < ss.n; ++i) {
      const float* mod = ss.mod[i];
      void* out = f8.current ? at(ws, p.stage[ss.s[i]]) : at(ws, p.h[ss.s[i]]);
      jobs[i] = {at(ws, p.x1[ss.s[i]]), mod + 3 * p.D, mod + 4 * p.D, 6 * p.D, out,
                 p.B * ss.rpb[i], ss.rpb[i]};
      if (f8.on() && !f8.current) {
        const int t = fp8_tensor(ss.s[i], 2, 0);
        jobs[i].q_scale = f8.scale(t), jobs[i].q_amax = f8.amax(t);
      }
    }
    MMDIT_CUDA(launch_ln_modulate2(d->act, 1, jobs, ss.n, p.D, d->ln_eps, st, f8.on() && !f8.current ? 1 : 0),
               "LayerNorm-modulate (MLP branch)");
  }
  if (f8.mx && !p.parallel) {
    ProfScope ps_(p.single ? "single.fp8_cast_h2" : "double.fp8_cast_h2", st);
    mmdit_status s = mx_in_place(p, ss, p.h, p.D, ws, st, "MXFP8 cast of the fc1 input");
    if (s != MMDIT_OK) return s;
  } else if (f8.blockwise && !p.parallel) {
    ProfScope ps_(p.single ? "single.fp8_cast_h2" : "double.fp8_cast_h2", st);
    for (int i = 0; i < ss.n; ++i) {
      mmdit_status s = cast_blockwise(i, at(ws, p.stage[ss.s[i]]), p.h[ss.s[i]], p.D, "blockwise E4M3 cast of the fc1 input");
      if (s != MMDIT_OK) return s;
    }
  } else if (f8.current && !p.parallel) {
    ProfScope ps_(p.single ? "single.fp8_cast_h2" : "double.fp8_cast_h2", st);
    QuantJob q[2];
    for (int i = 0; i < ss.n; ++i) {
      const int t = fp8_tensor(ss.s[i], 2, 0);
      q[i] = {at<__nv_bfloat16>(ws, p.stage[ss.s[i]]), at<uint8_t>(ws, p.h[ss.s[i]]),
              static_cast<int64_t>(p.B) * ss.rpb[i] * p.D, f8.scale(t), f8.amax(t)};
    }
    mmdit_status s = fp8_cast_current(f8, q, ss.n, st, "E4M3 cast of the fc1 input (current scaling)");
    if (s != MMDIT_OK) return s;
  }
  GemmProblem f1;
  f1.act = mm, f1.epi = f8.on() && !f8.current ? kEpiGeluF8 : kEpiGelu, f1.N = p.F, f1.K = p.D;
  for (int i = 0; i < ss.n; ++i) {
    EpiArgs e;
    e.bias = ss.w[i]->b_1, e.gelu_tanh = d->gelu_tanh, e.pre = ss.pre_1[i];
    e.out = f8.current ? at(ws, p.stage[ss.s[i]]) : at(ws, p.u[ss.s[i]]);
    dequant(e, i, 2);
    if (f8.on() && !f8.current) {
      const int t = fp8_tensor(ss.s[i], 3, 0);  // GELU output = the input of fc2
      e.out_scale = f8.scale(t), e.out_amax = f8.amax(t);
    }
    add_problem(f1, i, p.B * ss.rpb[i], at(ws, p.h[ss.s[i]]), weight(i, 2), e);
  }
  {
    ProfScope ps_(p.single ? "single.fc1" : "double.fc1", st);
    MMDIT_CUDA(launch_gemm(f1, status_word(ws), st), "MLP fc1 + GELU");
  }
  if (f8.mx) {
    ProfScope ps_(p.single ? "single.fp8_cast_u" : "double.fp8_cast_u", st);
    mmdit_status s = mx_in_place(p, ss, p.u, p.F, ws, st, "MXFP8 cast of the fc2 input");
    if (s != MMDIT_OK) return s;
  } else if (f8.blockwise) {
    ProfScope ps_(p.single ? "single.fp8_cast_u" : "double.fp8_cast_u", st);
    for (int i = 0; i < ss.n; ++i) {
      mmdit_status s = cast_blockwise(i, at(ws, p.stage[ss.s[i]]), p.u[ss.s[i]], p.F, "blockwise E4M3 cast of the fc2 input");
      if (s != MMDIT_OK) return s;
    }
  } else if (f8.current) {
    ProfScope ps_(p.single ? "single.fp8_cast_u" : "double.fp8_cast_u", st);
    QuantJob q[2];
    for (int i = 0; i < ss.n; ++i) {
      const int t = fp8_tensor(ss.s[i], 3, 0);
      q[i] = {at<__nv_bfloat16>(ws, p.stage[ss.s[i]]), at<uint8_t>(ws, p.u[ss.s[i]]),
              static_cast<int64_t>(p.B) * ss.rpb[i] * p.F, f8.scale(t), f8.amax(t)};
    }
    mmdit_status s = fp8_cast_current(f8, q, ss.n, st, "E4M3 cast of the fc2 input (current scaling)");
    if (s != MMDIT_OK) return s;
  }
  GemmProblem f2;
  f2.act = mm, f2.epi = kEpiGateResid, f2.N = p.D, f2.K = p.F;
  for (int i = 0; i < ss.n; ++i) {
    const float* mod = ss.mod[i];
    EpiArgs e;
    // the parallel block adds both branches under its one gate: x1 + gate (u W_2^T + b_2) after
    // x1 = x + gate (o W_o^T + b_o) is x + gate ([o | u] [W_o | W_2]^T + b_o + b_2)
    e.bias = ss.w[i]->b_2, e.resid = at(ws, p.x1[ss.s[i]]), e.resid_f32 = 1;
    e.gate = mod + (p.parallel ? 2 : 5) * p.D;
    e.gate_bstride = static_cast<int64_t>(p.mod_chunks) * p.D, e.rows_per_batch = ss.rpb[i], e.out = ss.y[i];
    e.pre = ss.pre_2[i];
    dequant(e, i, 3);
    add_problem(f2, i, p.B * ss.rpb[i], at(ws, p.u[ss.s[i]]), weight(i, 3), e);
  }
  ProfScope ps_(p.single ? "single.fc2" : "double.fc2", st);
  MMDIT_CUDA(launch_gemm(f2, status_word(ws), st), "MLP fc2 + gated residual");
  return MMDIT_OK;
}

// FP8 calls: zero this call's amax slot of every tensor the block records, then cast all weights
// of the block's streams to E4M3 in one launch.
mmdit_status fp8_begin(const BlockPlan& p, const Streams& ss, const Fp8& f8, int n_tensors,
                       void* ws, cudaStream_t st) {
  ProfScope ps_(p.single ? "single.fp8_cast_w" : "double.fp8_cast_w", st);
  if (f8.mx) {
    // every weight's MX-represented values (bf16) into the stream's wq slot, one launch
    MxJob jobs[kMxMaxJobs];
    int n = 0;
    for (int i = 0; i < ss.n; ++i) {
      const mmdit_stream_w* w = ss.w[i];
      const void* src[4] = {w->w_qkv, w->w_o, w->w_1, w->w_2};
      const size_t off[4] = {p.wq_qkv(), p.wq_o(), p.wq_1(), p.wq_2()};
      const int nn[4] = {3 * p.D, p.D, p.F, p.D}, kk[4] = {p.D, p.D, p.D, p.F};
      for (int g = 0; g < 4; ++g, ++n) {
        jobs[n].src = static_cast<const __nv_bfloat16*>(src[g]);
        jobs[n].deq = at<__nv_bfloat16>(ws, p.wq[ss.s[i]] + 2 * off[g]);
        jobs[n].rows = nn[g], jobs[n].K = kk[g];
      }
    }
    MMDIT_CUDA(launch_mx_cast(jobs, n, st), "MXFP8 cast of the weights");
    return MMDIT_OK;
  }
  if (f8.blockwise) {
    // every weight cast per 128 x 128 tile, its scales into the stream's bw_sw slot
    for (int i = 0; i < ss.n; ++i) {
      const mmdit_stream_w* w = ss.w[i];
      const int slot = ss.s[i];
      const void* src[4] = {w->w_qkv, w->w_o, w->w_1, w->w_2};
      const size_t off[4] = {p.wq_qkv(), p.wq_o(), p.wq_1(), p.wq_2()};
      const size_t soff[4] = {p.sw_qkv(), p.sw_o(), p.sw_1(), p.sw_2()};
      const int nn[4] = {3 * p.D, p.D, p.F, p.D}, kk[4] = {p.D, p.D, p.D, p.F};
      for (int g = 0; g < 4; ++g)
        MMDIT_CUDA(launch_blockwise_cast_weight(static_cast<const __nv_bfloat16*>(src[g]), nn[g], kk[g],
                                                at<uint8_t>(ws, p.wq[slot] + off[g]),
                                                at<float>(ws, p.bw_sw[slot] + soff[g]), st),
                   "blockwise E4M3 cast of the weights");
    }
    return MMDIT_OK;
  }
  MMDIT_CUDA(launch_amax_reset(f8.f->amax_history, f8.f->hist_len, n_tensors, f8.f->pos, st),
             "FP8 amax slot reset");
  QuantJob jobs[kQuantMaxJobs];
  int n = 0;
  for (int i = 0; i < ss.n; ++i) {
    const mmdit_stream_w* w = ss.w[i];
    const int slot = ss.s[i];
    const void* src[4] = {w->w_qkv, w->w_o, w->w_1, w->w_2};
    const size_t off[4] = {p.wq_qkv(), p.wq_o(), p.wq_1(), p.wq_2()};
    const int64_t cnt[4] = {static_cast<int64_t>(3) * p.D * p.D, static_cast<int64_t>(p.D) * p.D,
                            static_cast<int64_t>(p.F) * p.D, static_cast<int64_t>(p.D) * p.F};
    for (int g = 0; g < 4; ++g) {
      const int t = fp8_tensor(slot, g, 1);
      jobs[n++] = {static_cast<const __nv_bfloat16*>(src[g]), at<uint8_t>(ws, p.wq[slot] + off[g]), cnt[g],
                   f8.scale(t), f8.amax(t)};
    }
  }
  if (f8.current) return fp8_cast_current(f8, jobs, n, st, "E4M3 cast of the weights (current scaling)");
  MMDIT_CUDA(launch_quantize_e4m3(jobs, n, st), "E4M3 cast of the weights");
  return MMDIT_OK;
}

// FP8 calls: the next call's scales from the recorded amax (most_recent or the history's max).
mmdit_status fp8_end(const BlockPlan& p, const Fp8& f8, int n_tensors, cudaStream_t st) {
  if (f8.blockwise) return MMDIT_OK;  // no state: every scale is this call's own
  ProfScope ps_(p.single ? "single.fp8_scale" : "double.fp8_scale", st);
  MMDIT_CUDA(launch_scale_update(f8.f->amax_history, f8.f->scale, f8.f->hist_len, n_tensors, f8.f->pos,
                                 f8.f->margin, f8.current ? 0 : f8.f->amax_compute_algo, st),
             "FP8 scale update");
  return MMDIT_OK;
}

mmdit_status run_attention(const BlockPlan& p, int act, void* ws, cudaStream_t st) {
  AttnProblem a;
  a.act = act, a.batch = p.B, a.heads = p.H, a.seq = p.S, a.seq_pad = p.S_pad;
  a.split = p.single ? p.S : p.Si;
  a.q = at<__nv_bfloat16>(ws, p.q), a.k = at<__nv_bfloat16>(ws, p.k);
  a.vt = at<__half>(ws, p.vt);
  a.out0 = at(ws, p.o[0]);
  a.out1 = p.single ? nullptr : at(ws, p.o[1]);
  { ProfScope ps_(p.single ? "single.attention" : "double.attention", st);
  MMDIT_CUDA(launch_attention(a, status_word(ws), st), "joint attention"); }
  return MMDIT_OK;
}

// ----------------------------------------------------------------------------- step bodies
// The work of an entry point after its checks, on a workspace whose first word is the status
// word the caller cleared: the whole-model forward runs them back to back on one workspace, so
// a timeout in any step stays visible.

mmdit_status double_block_body(const mmdit_dims* d, const BlockPlan& p, const mmdit_stream_w* w_img,
                               const mmdit_stream_w* w_txt, const void* vec, const float* rope_cos,
                               const float* rope_sin, const void* x_img, const void* x_txt,
                               void* y_img, void* y_txt, mmdit_fp8_state* fp8, void* workspace,
                               cudaStream_t st) {
  mmdit_status s = MMDIT_OK;
  {
    // both streams' AdaLN modulation in one launch (they share vec), unless precomputed
    ModulationJob jobs[2];
    int nj = 0;
    if (!w_img->mod) jobs[nj++] = {w_img->w_mod, w_img->b_mod, at<float>(workspace, p.mod[0]), 6 * p.D};
    if (!w_txt->mod) jobs[nj++] = {w_txt->w_mod, w_txt->b_mod, at<float>(workspace, p.mod[1]), 6 * p.D};
    if (nj) {
      ProfScope ps_("double.modulation", st);
      MMDIT_CUDA(launch_modulation2(d->act, vec, jobs, nj, p.B, p.D, st), "modulation");
    }
  }
  Streams ss;
  const mmdit_stream_w* wsets[2] = {w_img, w_txt};
  const void* xs[2] = {x_img, x_txt};
  void* ys[2] = {y_img, y_txt};
  const int rpb[2] = {p.Si, p.St};
  for (int i = 0; i < 2; ++i)
    if (rpb[i] > 0) {
      ss.s[ss.n] = i, ss.w[ss.n] = wsets[i], ss.x[ss.n] = xs[i], ss.y[ss.n] = ys[i];
      ss.rpb[ss.n] = rpb[i];
      ss.mod[ss.n] = wsets[i]->mod ? wsets[i]->mod : at<float>(workspace, p.mod[i]);
      ++ss.n;
    }
  Fp8 f8;
  f8.f = fp8;
  const int n_tensors = 2 * kFp8TensorsPerStream;
  f8.current = p.fp8_current, f8.blockwise = p.fp8_blockwise, f8.mx = p.fp8_mx, f8.n_tensors = n_tensors;
  if ((f8.on() || f8.mx) && (s = fp8_begin(p, ss, f8, n_tensors, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_qkv(d, p, ss, rope_cos, rope_sin, f8, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_attention(p, d->act, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_post(d, p, ss, f8, workspace, st)) != MMDIT_OK) return s;
  return f8.on() ? fp8_end(p, f8, n_tensors, st) : MMDIT_OK;
}

mmdit_status single_block_body(const mmdit_dims* d, const BlockPlan& p, const mmdit_stream_w* w,
                               const void* vec, const float* rope_cos, const float* rope_sin,
                               const void* x, void* y, mmdit_fp8_state* fp8, void* workspace,
                               cudaStream_t st) {
  mmdit_status s = MMDIT_OK;
  if (!w->mod) {
    ProfScope ps_("single.modulation", st);
    MMDIT_CUDA(launch_modulation(d->act, vec, w->w_mod, w->b_mod, p.B, p.mod_chunks * p.D, p.D,
                                 at<float>(workspace, p.mod[0]), st),
               "modulation");
  }
  Streams ss;
  ss.n = 1, ss.s[0] = 0, ss.w[0] = w, ss.x[0] = x, ss.y[0] = y, ss.rpb[0] = p.S;
  ss.mod[0] = w->mod ? w->mod : at<float>(workspace, p.mod[0]);
  Fp8 f8;
  f8.f = fp8;
  f8.current = p.fp8_current, f8.blockwise = p.fp8_blockwise, f8.mx = p.fp8_mx, f8.n_tensors = kFp8TensorsPerStream;
  if ((f8.on() || f8.mx) && (s = fp8_begin(p, ss, f8, kFp8TensorsPerStream, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_qkv(d, p, ss, rope_cos, rope_sin, f8, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_attention(p, d->act, workspace, st)) != MMDIT_OK) return s;
  if ((s = run_post(d, p, ss, f8, workspace, st)) != MMDIT_OK) return s;
  return f8.on() ? fp8_end(p, f8, kFp8TensorsPerStream, st) : MMDIT_OK;
}

// Output-head workspace: the head's modulation, its LayerNorm-modulate output, the split-K
// partials, and (loss variant) one partial sum per finishing block.  The loss variant's ticket
// counter sits inside the status region (kHeadTicketOffset), cleared with the status word.
constexpr size_t kHeadTicketOffset = 128;
struct HeadPlan {
  size_t mod, h, partials, loss_partials, total;
  int splits;
};
HeadPlan plan_head(const mmdit_dims* d, int channels, bool with_loss) {
  HeadPlan p;
  Carver c;
  const int M = d->batch * d->seq_img;
  p.mod = c.take(static_cast<size_t>(d->batch) * 2 * d->hidden * 4);
  p.h = c.take(static_cast<size_t>(M) * d->hidden * elt_bytes(d->act));
  p.splits = choose_splits(M, channels, d->hidden, static_cast<int>(elt_bytes(d->act)));
  // the loss variant always takes the partials path: its finishing kernel forms pred and the loss
  p.partials = p.splits > 1 || with_loss ? c.take(static_cast<size_t>(p.splits) * M * channels * sizeof(float)) : 0;
  p.loss_partials = with_loss ? c.take(static_cast<size_t>(head_finish_blocks(M, channels)) * sizeof(float)) : 0;
  p.total = c.off;
  return p;
}

mmdit_status final_layer_body(const mmdit_dims* d, int channels, const void* x_img, const void* vec,
                              const void* w_ada, const void* b_ada, const void* w_out,
                              const void* b_out, float* pred, void* workspace, cudaStream_t st,
                              const float* z0 = nullptr, const float* z1 = nullptr,
                              float* loss = nullptr, const float* mod_in = nullptr) {
  const bool with_loss = loss != nullptr;
  const HeadPlan hp = plan_head(d, channels, with_loss);
  // the head's (shift, scale): precomputed by the caller, or computed here
  const float* mod = mod_in ? mod_in : at<float>(workspace, hp.mod);
  void* h = at(workspace, hp.h);
  const int D = d->hidden, rows = d->batch * d->seq_img;
  ProfScope ps_(with_loss ? "final_layer_loss" : "final_layer", st);
  if (!mod_in)
    MMDIT_CUDA(launch_modulation(d->act, vec, w_ada, b_ada, d->batch, 2 * D, D, at<float>(workspace, hp.mod), st),
               "final modulation");
  MMDIT_CUDA(launch_ln_modulate(d->act, d->act == MMDIT_F32, x_img, mod, mod + D, 2 * D, rows, d->seq_img, D, d->ln_eps, h, st),
             "final LayerNorm-modulate");
  GemmProblem g;
  g.act = d->act, g.M = rows, g.N = channels, g.K = D, g.A = h, g.W = w_out;
  const int splits = hp.splits;
  if (with_loss) {
    // the projection's fp32 partials, then one kernel forming pred and the fused loss
    float* partials = at<float>(workspace, hp.partials);
    g.epi = kEpiPartial, g.splits = splits, g.ep.out = partials;
    MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "final projection (partials)");
    MMDIT_CUDA(launch_head_finish(d->act, partials, splits, rows, channels, b_out, d->seq_img, pred, z0, z1,
                                  at<float>(workspace, hp.loss_partials),
                                  at<unsigned int>(workspace, kHeadTicketOffset), loss, st),
               "final projection sum + flow-matching loss");
  } else if (splits > 1) {
    float* partials = at<float>(workspace, hp.partials);
    g.epi = kEpiPartial, g.splits = splits, g.ep.out = partials;
    MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "final projection (split K)");
    MMDIT_CUDA(launch_splitk_reduce(d->act, partials, splits, rows, channels, b_out, pred,
                                    d->seq_img, st),
               "final projection (split-K sum)");
  } else {
    g.epi = kEpiUnpatchify, g.ep.bias = b_out, g.ep.out = pred, g.ep.rows_per_batch = d->seq_img;
    MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "final projection");
  }
  return MMDIT_OK;
}

mmdit_status img_in_body(int act, int batch, int channels, int lat_h, int lat_w, int hidden,
                         const float* z, const void* w, const void* b, void* out, void* workspace,
                         cudaStream_t st, const float* z1 = nullptr, const float* t = nullptr,
                         float* z_t = nullptr) {
  void* tokens = at(workspace, kStatusBytes);
  const int hw = lat_h * lat_w;
  ProfScope ps_(z1 ? "img_in_noise" : "img_in", st);
  MMDIT_CUDA(launch_patchify(act, z, batch, channels, hw, tokens, st, z1, t, z_t),
             z1 ? "patchify of z_t" : "patchify");
  GemmProblem g;
  g.act = act, g.epi = kEpiBias, g.M = batch * hw, g.N = hidden, g.K = channels;
  g.A = tokens, g.W = w, g.ep.bias = b, g.ep.out = out;
  MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "img_in linear");
  return MMDIT_OK;
}

mmdit_status linear_body(int act, int M, int N, int K, const void* x, const void* w, const void* b,
                         void* y, void* workspace, cudaStream_t st) {
  if (M == 0) return MMDIT_OK;
  const int splits = choose_splits(M, N, K, static_cast<int>(elt_bytes(act)));
  GemmProblem g;
  g.act = act, g.M = M, g.N = N, g.K = K, g.A = x, g.W = w;
  ProfScope ps_("linear", st);
  if (splits > 1) {
    // narrow GEMM: K split across work items, fp32 partials, then a fixed-order finish
    float* partials = at<float>(workspace, kStatusBytes);
    g.epi = kEpiPartial, g.splits = splits, g.ep.out = partials;
    MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "linear (split K)");
    MMDIT_CUDA(launch_splitk_reduce(act, partials, splits, M, N, b, y, 0, st), "linear (split-K sum)");
  } else {
    g.epi = kEpiBias, g.ep.bias = b, g.ep.out = y;
    MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "linear");
  }
  return MMDIT_OK;
}

size_t conditioning_workspace(int act, int batch, int hidden, int time_dim) {
  Carver c;
  const size_t e = elt_bytes(act);
  c.take(static_cast<size_t>(batch) * time_dim * e);  // sinusoidal features
  c.take(static_cast<size_t>(batch) * hidden * 4);    // timestep MLP hidden layer (fp32)
  c.take(static_cast<size_t>(batch) * hidden * 4);    // vector MLP hidden layer (fp32)
  c.take(static_cast<size_t>(batch) * hidden * 4);    // fp32 sum of the embeddings
  return c.off;
}

mmdit_status conditioning_body(int act, int B, int D, int time_dim, int vec_in_dim, const mmdit_cond_w* w,
                               const float* t, const void* y, const float* g, void* vec, void* workspace,
                               cudaStream_t st) {
  Carver c;
  const size_t e = elt_bytes(act);
  void* feat = at(workspace, c.take(static_cast<size_t>(B) * time_dim * e));
  float* ht = at<float>(workspace, c.take(static_cast<size_t>(B) * D * 4));
  float* hy = at<float>(workspace, c.take(static_cast<size_t>(B) * D * 4));
  float* v32 = at<float>(workspace, c.take(static_cast<size_t>(B) * D * 4));
  ProfScope ps_("conditioning", st);
  MMDIT_CUDA(launch_timestep_features(act, t, B, time_dim, 1000.0, 10000.0, feat, st), "timestep features");
  // first layers (no activation on their inputs); the hidden layers stay fp32, so the second
  // layers' operand SiLU(h) is rounded once, where it enters the linear
  const ModulationJob l1t{w->time_in.w1, w->time_in.b1, ht, D};
  MMDIT_CUDA(launch_gemv(act, feat, &l1t, 1, B, time_dim, 0, kGemvOutF32, st), "timestep MLP layer 1");
  const ModulationJob l1y{w->vector_in.w1, w->vector_in.b1, hy, D};
  MMDIT_CUDA(launch_gemv(act, y, &l1y, 1, B, vec_in_dim, 0, kGemvOutF32, st), "vector MLP layer 1");
  // second layers read SiLU of the hidden layers; the vector MLP adds onto the timestep's
  const ModulationJob l2t{w->time_in.w2, w->time_in.b2, v32, D};
  MMDIT_CUDA(launch_gemv(act, ht, &l2t, 1, B, D, 1, kGemvOutF32, st, 1), "timestep MLP layer 2");
  const ModulationJob l2y{w->vector_in.w2, w->vector_in.b2, v32, D};
  MMDIT_CUDA(launch_gemv(act, hy, &l2y, 1, B, D, 1, kGemvOutF32Add, st, 1), "vector MLP layer 2");
  MMDIT_CUDA(launch_vec_finish(act, v32, g, w->w_guidance, w->b_guidance, B, D, vec, st), "conditioning vector");
  return MMDIT_OK;
}

// ----------------------------------------------------------------------------- block backward
// Scratch of one linear backward (the weight transpose, the transposed operands of dW, the bias
// gradient's partial column sums).
size_t linear_bwd_scratch(size_t e, size_t M, size_t N, size_t K) {
  const size_t Mp = round_up(M, 8);
  Carver c;
  c.off = 0;
  c.take(K * N * e);
  c.take(N * Mp * e);
  c.take(K * Mp * e);
  c.take(static_cast<size_t>(kColsumChunks) * N * 4);
  return c.off;
}

// dx = dy W [M, K] (activation type), dW = dy^T x [N, K] fp32, db = column sums of dy [N] fp32, each
// skipped when its pointer is null; `scratch` holds linear_bwd_scratch bytes, `ws` the status word.
// With gelu_pre ([M, K], the input of a GELU whose output is x), dx is multiplied by GELU'(gelu_pre):
// the gradient of that GELU's input.
mmdit_status linear_bwd_body(int act, int M, int N, int K, const void* dy, const void* x, const void* w, void* dx,
                             float* dw, float* db, void* scratch, void* ws, cudaStream_t st,
                             const void* gelu_pre = nullptr, int gelu_tanh = 0) {
  const size_t e = elt_bytes(act);
  const int Mp = static_cast<int>(round_up(static_cast<size_t>(M), 8));
  Carver c;
  c.off = 0;
  void* wt = at(scratch, c.take(static_cast<size_t>(K) * N * e));
  void* dyt = at(scratch, c.take(static_cast<size_t>(N) * Mp * e));
  void* xt = at(scratch, c.take(static_cast<size_t>(K) * Mp * e));
  float* part = at<float>(scratch, c.take(static_cast<size_t>(kColsumChunks) * N * 4));
  // bf16 with K % 256 == 0: the tensor cores read W, dy and x as stored (MN-major operands);
  // otherwise the operands are transposed into K-major copies first
  const bool mn = act == 1 && K % 256 == 0 && N % 8 == 0;
  if (dx) {
    // dx [M, K] = dy [M, N] W [N, K]: A = dy (K-major), B = W read as W^T's MN-major form
    GemmProblem g;
    g.act = act, g.epi = kEpiBias, g.M = M, g.N = K, g.K = N, g.A = dy, g.W = w, g.ep.out = dx;
    if (mn) {
      g.b_mn = 1;
      if (gelu_pre) g.epi = kEpiDGelu, g.ep.aux = gelu_pre, g.ep.gelu_tanh = gelu_tanh;
    } else {
      MMDIT_CUDA(launch_transpose_pad(act, w, N, K, N, wt, st), "W transpose");
      g.W = wt;
    }
    MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "dx GEMM");
    if (gelu_pre && !mn)
      MMDIT_CUDA(launch_gelu_bwd(act, dx, gelu_pre, static_cast<int64_t>(M) * K, gelu_tanh, dx, st), "GELU backward");
  }
  if (dw) {
    // dW [N, K] = dy^T x, contracted over the M rows
    GemmProblem g;
    g.act = act, g.epi = kEpiBias, g.M = N, g.N = K, g.ep.out = dw;
    g.ep.out_f32 = 1;
    if (mn) {
      // dy [M, N] and x [M, K] are dy^T's and x^T's MN-major forms; rows past M read as zeros
      g.K = M, g.A = dy, g.W = x, g.a_mn = 1, g.b_mn = 1;
    } else {
      // K-major copies dy^T [N, Mp] and x^T [K, Mp], zero-padded to Mp
      MMDIT_CUDA(launch_transpose_pad(act, dy, M, N, Mp, dyt, st), "dy transpose");
      MMDIT_CUDA(launch_transpose_pad(act, x, M, K, Mp, xt, st), "x transpose");
      g.K = Mp, g.A = dyt, g.W = xt;
    }
    MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "dW GEMM");
  }
  if (db) MMDIT_CUDA(launch_colsum(act, dy, M, N, part, kColsumChunks, db, st), "db column sums");
  return MMDIT_OK;
}

// The linear backward of a block's two streams (same N and K; M[0] and M[1] rows): in bf16 with
// MN-major operands, both streams' dx run in one GEMM launch and both dW in another (the text
// stream's short contraction interleaved with the image stream's tiles, so its epilogue-heavy
// tiles do not form a wave of their own); otherwise, or when the streams ask for different
// outputs, one linear_bwd_body per stream.
mmdit_status linear_bwd_streams(int act, int ns, const int* M, int N, int K, const void* const* dy,
                                const void* const* x, const void* const* w, void* const* dx, float* const* dw,
                                float* const* db, void* scratch, void* ws, cudaStream_t st,
                                const void* const* gelu_pre = nullptr, int gelu_tanh = 0) {
  const bool joint = ns == 2 && M[0] > 0 && M[1] > 0 && act == 1 && K % 256 == 0 && N % 8 == 0 &&
                     (dx[0] == nullptr) == (dx[1] == nullptr) && (dw[0] == nullptr) == (dw[1] == nullptr) &&
                     (gelu_pre == nullptr || (gelu_pre[0] == nullptr) == (gelu_pre[1] == nullptr));
  if (!joint) {
    for (int i = 0; i < ns; ++i) {
      if (M[i] == 0) continue;
      mmdit_status s = linear_bwd_body(act, M[i], N, K, dy[i], x[i], w[i], dx[i], dw[i], db[i], scratch, ws, st,
                                       gelu_pre ? gelu_pre[i] : nullptr, gelu_tanh);
      if (s != MMDIT_OK) return s;
    }
    return MMDIT_OK;
  }
  const bool dgelu = gelu_pre && gelu_pre[0];
  if (dx[0]) {
    GemmProblem g;
    g.act = act, g.epi = dgelu ? kEpiDGelu : kEpiBias, g.N = K, g.K = N, g.b_mn = 1;
    g.M = M[0], g.A = dy[0], g.W = w[0], g.ep.out = dx[0];
    g.M1 = M[1], g.A1 = dy[1], g.W1 = w[1], g.ep1.out = dx[1];
    if (dgelu) {
      g.ep.aux = gelu_pre[0], g.ep1.aux = gelu_pre[1];
      g.ep.gelu_tanh = g.ep1.gelu_tanh = gelu_tanh;
    }
    MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "dx GEMM (both streams)");
  }
  if (dw[0]) {
    GemmProblem g;
    g.act = act, g.epi = kEpiBias, g.N = K, g.a_mn = 1, g.b_mn = 1, g.interleave = 1;
    g.M = N, g.K = M[0], g.A = dy[0], g.W = x[0], g.ep.out = dw[0], g.ep.out_f32 = 1;
    g.M1 = N, g.K1 = M[1], g.A1 = dy[1], g.W1 = x[1], g.ep1.out = dw[1], g.ep1.out_f32 = 1;
    MMDIT_CUDA(launch_gemm(g, status_word(ws), st), "dW GEMM (both streams)");
  }
  // (no transposed copies on this path: the column-sum partials take the scratch's start)
  float* part = at<float>(scratch, 0);
  for (int i = 0; i < 2; ++i)
    if (db[i]) MMDIT_CUDA(launch_colsum(act, dy[i], M[i], N, part, kColsumChunks, db[i], st), "db column sums");
  return MMDIT_OK;
}

// Workspace of a block backward: the forward's own slots first (the backward recomputes the
// forward into them), then what the backward reads of the forward and its own gradients.
struct BwdPlan {
  BlockPlan f;
  size_t h1[2], qkv_pre[2], a[2], u_pre[2], fo[2], ytmp[2];
  size_t dx1[2], df[2], du[2], dh[2], dO[2], dqkv[2], dm[2];
  size_t lse, dsum, doh, q16, k16, v, dq, dk, dv, amax;
  size_t part, lin;
  size_t total;
};

bool plan_block_bwd(const mmdit_dims* d, bool single, BwdPlan* p) {
  if (!plan_block(d, single, &p->f)) return false;
  const BlockPlan& f = p->f;
  const size_t B = f.B, D = f.D, F = f.F, e = f.elt, H = f.H, S = f.S, Sp = f.S_pad;
  const int ns = single ? 1 : 2;
  const size_t rows[2] = {B * (single ? S : static_cast<size_t>(f.Si)), single ? 0 : B * static_cast<size_t>(f.St)};
  Carver c;
  c.off = round_up(f.total, 256);
  for (int s = 0; s < 2; ++s) {
    const size_t R = s < ns ? rows[s] : 0;
    p->h1[s] = c.take(R * D * e), p->qkv_pre[s] = c.take(R * 3 * D * e), p->a[s] = c.take(R * D * e);
    p->u_pre[s] = c.take(R * F * e), p->fo[s] = c.take(R * D * e), p->ytmp[s] = c.take(R * D * e);
    p->dx1[s] = c.take(R * D * 4), p->df[s] = c.take(R * D * e), p->du[s] = c.take(R * F * e);
    p->dh[s] = c.take(R * D * e), p->dO[s] = c.take(R * D * e), p->dqkv[s] = c.take(R * 3 * D * e);
    p->dm[s] = c.take(s < ns ? B * 6 * D * 4 : 0);
  }
  // L and D are read in 64-row tiles by bulk copies: 64 floats of slack past the end
  p->lse = c.take((B * H * Sp + 64) * 4), p->dsum = c.take((B * H * Sp + 64) * 4);
  // the attention backward's fp16 operands, [B, H, S, 128] each
  p->doh = c.take(B * H * S * 128 * 2), p->q16 = c.take(B * H * S * 128 * 2), p->k16 = c.take(B * H * S * 128 * 2);
  p->v = c.take(B * H * S * 128 * 2);
  p->dq = c.take(B * H * S * 128 * 4), p->dk = c.take(B * H * S * 128 * 4), p->dv = c.take(B * H * S * 128 * 4);
  p->amax = c.take(256);
  size_t part = static_cast<size_t>(qk_norm_rope_bwd_blocks()) * 2 * 128 * 4;
  part = std::max(part, static_cast<size_t>(modulation_dvec_chunks(6 * f.D)) * B * D * 4);
  size_t lin = 0;
  for (int s = 0; s < ns; ++s) {
    const int rpb = single ? f.S : (s ? f.St : f.Si);
    part = std::max(part, ln_modulate_bwd_part_bytes(f.B, rpb, f.D));
    part = std::max(part, gated_residual_bwd_part_bytes(f.B, rpb, f.D));
    lin = std::max(lin, linear_bwd_scratch(e, rows[s], D, F));      // fc2
    lin = std::max(lin, linear_bwd_scratch(e, rows[s], F, D));      // fc1
    lin = std::max(lin, linear_bwd_scratch(e, rows[s], 3 * D, D));  // QKV
    lin = std::max(lin, linear_bwd_scratch(e, rows[s], D, D));      // attention output projection
  }
  p->part = c.take(part);
  p->lin = c.take(lin);
  p->total = c.off;
  return true;
}

// The backward of a double block (ns = 2: image and text streams) or a single block (ns = 1, one
// stream over the joint rows).  The forward is recomputed into the workspace first (activation
// recomputation: the call needs only the block's inputs), keeping what the backward reads: the
// attention branch's LayerNorm output h1, the QKV linear before its norm, the attention output
// and its log-sum-exp, the output projection a, the fp32 residual x1, the MLP's LayerNorm output,
// its pre-GELU u_pre, GELU output and fc2 output (the linears' pre-norm, pre-GELU and pre-gate
// outputs are written by the fused GEMMs' epilogues alongside their usual outputs).  Then, per stream, the MLP branch and the
// attention projection backward; the joint attention backward; per stream the QK-RMSNorm + RoPE,
// QKV and LayerNorm backward and the modulation backward.
//
// `phases` selects the parts: kBwdForward (the recomputation, into the workspace; with Y the block's
// outputs also go there) and kBwdGradients (everything after it, reading what the forward left in
// the workspace).  The training pair mmdit_*_block_fwd_train / mmdit_*_block_bwd_saved runs them
// in two calls around the caller's own work.
constexpr int kBwdForward = 1, kBwdGradients = 2;
mmdit_status block_bwd_body(const mmdit_dims* d, const BwdPlan& bp, int ns, const mmdit_stream_w* const* W,
                            const void* vec, const float* rope_cos, const float* rope_sin, const void* const* X,
                            const void* const* DY, void* const* DX, float* dvec,
                            const mmdit_stream_grads* const* G, void* ws, cudaStream_t st,
                            int phases = kBwdForward | kBwdGradients, void* const* Y = nullptr) {
  const BlockPlan& p = bp.f;
  const int act = d->act, B = p.B, D = p.D, F = p.F, H = p.H, S = p.S;
  const size_t e = p.elt;
  const int rpb[2] = {ns == 1 ? p.S : p.Si, p.St};
  const int off[2] = {0, p.Si};
  const mmdit_stream_grads none = {};
  mmdit_status s = MMDIT_OK;
  // ---------------- forward, keeping what the backward reads
  if (phases & kBwdForward) {
  {
    ModulationJob jobs[2];
    for (int i = 0; i < ns; ++i) jobs[i] = {W[i]->w_mod, W[i]->b_mod, at<float>(ws, p.mod[i]), 6 * D};
    ProfScope ps_("bwd.recompute.modulation", st);
    MMDIT_CUDA(launch_modulation2(act, vec, jobs, ns, B, D, st), "modulation");
  }
  Streams ss;
  ss.n = 0;
  for (int i = 0; i < ns; ++i) {
    if (rpb[i] == 0) continue;
    ss.s[ss.n] = i, ss.w[ss.n] = W[i], ss.x[ss.n] = X[i], ss.rpb[ss.n] = rpb[i];
    ss.y[ss.n] = Y ? Y[i] : at(ws, bp.ytmp[i]);
    ss.mod[ss.n] = at<float>(ws, p.mod[i]);
    // the linears' outputs before their norm, GELU or gate come out of the same GEMMs
    ss.pre_qkv[ss.n] = at(ws, bp.qkv_pre[i]), ss.pre_o[ss.n] = at(ws, bp.a[i]);
    ss.pre_1[ss.n] = at(ws, bp.u_pre[i]), ss.pre_2[ss.n] = at(ws, bp.fo[i]);
    ++ss.n;
  }
  Fp8 no_fp8;
  if ((s = run_qkv(d, p, ss, rope_cos, rope_sin, no_fp8, ws, st)) != MMDIT_OK) return s;
  for (int i = 0; i < ns; ++i) {
    const size_t R = static_cast<size_t>(B) * rpb[i];
    if (R == 0) continue;
    ProfScope ps_("bwd.recompute.keep_h1", st);
    MMDIT_CUDA(cudaMemcpyAsync(at(ws, bp.h1[i]), at(ws, p.h[i]), R * D * e, cudaMemcpyDeviceToDevice, st), "keep h1");
    pdl_begin_call();  // the next kernel follows a copy
  }
  {
    AttnProblem a;
    a.act = act, a.batch = B, a.heads = H, a.seq = S, a.seq_pad = p.S_pad, a.split = ns == 1 ? S : p.Si;
    a.q = at<__nv_bfloat16>(ws, p.q), a.k = at<__nv_bfloat16>(ws, p.k), a.vt = at<__half>(ws, p.vt);
    a.out0 = at(ws, p.o[0]), a.out1 = ns == 1 ? nullptr : at(ws, p.o[1]);
    a.lse = at<float>(ws, bp.lse);
    ProfScope ps_("bwd.recompute.attention", st);
    MMDIT_CUDA(launch_attention(a, status_word(ws), st), "joint attention (with log-sum-exp)");
  }
  // x1, the MLP's h (in h), u, and the linears' pre-gate / pre-GELU outputs
  if ((s = run_post(d, p, ss, no_fp8, ws, st)) != MMDIT_OK) return s;
  }
  if (!(phases & kBwdGradients)) return MMDIT_OK;
  // ---------------- backward: MLP branch and the attention projection, both streams step by step
  // (each linear's backward runs for both streams in shared launches)
  float* part = at<float>(ws, bp.part);
  void* lin = at(ws, bp.lin);
  const int64_t bstr = 6 * static_cast<int64_t>(D);
  int R[2] = {0, 0};
  const mmdit_stream_grads* Gs[2] = {&none, &none};
  for (int i = 0; i < ns; ++i) R[i] = B * rpb[i], Gs[i] = G[i] ? G[i] : &none;
  auto ptrs = [&](auto f) {  // a per-stream pointer pair
    using T = decltype(f(0));
    std::array<T, 2> a{};
    for (int i = 0; i < ns; ++i) a[i] = f(i);
    return a;
  };
  {
    ProfScope ps_("bwd.mlp_and_out_proj", st);
    for (int i = 0; i < ns; ++i) {
      if (R[i] == 0) continue;  // (the entry points reject streams without rows)
      const float* mod = at<float>(ws, p.mod[i]);
      float* dx1 = at<float>(ws, bp.dx1[i]);
      MMDIT_CUDA(launch_convert(act, 1, DY[i], static_cast<int64_t>(R[i]) * D, dx1, st), "dy to fp32");
      MMDIT_CUDA(launch_gated_residual_bwd(act, dx1, at(ws, bp.fo[i]), mod + 5 * D, bstr, B, rpb[i], D,
                                           at(ws, bp.df[i]), at<float>(ws, bp.dm[i]) + 5 * D, part, st),
                 "gate2 backward");
    }
    // fc2's input gradient times GELU'(u_pre): the gradient of fc1's output
    {
      const auto dy = ptrs([&](int i) -> const void* { return at(ws, bp.df[i]); });
      const auto xx = ptrs([&](int i) -> const void* { return at(ws, p.u[i]); });
      const auto ww = ptrs([&](int i) -> const void* { return W[i]->w_2; });
      const auto dx = ptrs([&](int i) -> void* { return at(ws, bp.du[i]); });
      const auto dw = ptrs([&](int i) -> float* { return Gs[i]->w_2; });
      const auto db = ptrs([&](int i) -> float* { return Gs[i]->b_2; });
      const auto gp = ptrs([&](int i) -> const void* { return at(ws, bp.u_pre[i]); });
      if ((s = linear_bwd_streams(act, ns, R, D, F, dy.data(), xx.data(), ww.data(), dx.data(), dw.data(), db.data(),
                                  lin, ws, st, gp.data(), d->gelu_tanh)) != MMDIT_OK)
        return s;
    }
    {
      const auto dy = ptrs([&](int i) -> const void* { return at(ws, bp.du[i]); });
      const auto xx = ptrs([&](int i) -> const void* { return at(ws, p.h[i]); });
      const auto ww = ptrs([&](int i) -> const void* { return W[i]->w_1; });
      const auto dx = ptrs([&](int i) -> void* { return at(ws, bp.dh[i]); });
      const auto dw = ptrs([&](int i) -> float* { return Gs[i]->w_1; });
      const auto db = ptrs([&](int i) -> float* { return Gs[i]->b_1; });
      if ((s = linear_bwd_streams(act, ns, R, F, D, dy.data(), xx.data(), ww.data(), dx.data(), dw.data(), db.data(),
                                  lin, ws, st)) != MMDIT_OK)
        return s;
    }
    for (int i = 0; i < ns; ++i) {
      if (R[i] == 0) continue;
      const float* mod = at<float>(ws, p.mod[i]);
      float* dx1 = at<float>(ws, bp.dx1[i]);
      float* dm = at<float>(ws, bp.dm[i]);
      MMDIT_CUDA(launch_ln_modulate_bwd(act, 1, at(ws, p.x1[i]), at(ws, bp.dh[i]), mod + 4 * D, bstr, B, rpb[i], D,
                                        d->ln_eps, dx1, dm + 4 * D, dm + 3 * D, 0, part, st), "LN2 backward");
      MMDIT_CUDA(launch_gated_residual_bwd(act, dx1, at(ws, bp.a[i]), mod + 2 * D, bstr, B, rpb[i], D,
                                           at(ws, bp.df[i]), dm + 2 * D, part, st), "gate1 backward");
    }
    {
      const auto dy = ptrs([&](int i) -> const void* { return at(ws, bp.df[i]); });
      const auto xx = ptrs([&](int i) -> const void* { return at(ws, p.o[i]); });
      const auto ww = ptrs([&](int i) -> const void* { return W[i]->w_o; });
      const auto dx = ptrs([&](int i) -> void* { return at(ws, bp.dO[i]); });
      const auto dw = ptrs([&](int i) -> float* { return Gs[i]->w_o; });
      const auto db = ptrs([&](int i) -> float* { return Gs[i]->b_o; });
      if ((s = linear_bwd_streams(act, ns, R, D, D, dy.data(), xx.data(), ww.data(), dx.data(), dw.data(), db.data(),
                                  lin, ws, st)) != MMDIT_OK)
        return s;
    }
  }
  // ---------------- the joint attention backward
  const int bh = B * H;
  float* amax = at<float>(ws, bp.amax);
  {
    ProfScope ps_("bwd.attention_prepass", st);
    bool first = true;
    for (int i = 0; i < ns; ++i) {
      if (rpb[i] == 0) continue;
      MMDIT_CUDA(launch_grad_amax(at<__nv_bfloat16>(ws, bp.dO[i]), static_cast<int64_t>(B) * rpb[i] * D, amax,
                                  first, st), "dO amax");
      first = false;
    }
    for (int i = 0; i < ns; ++i)
      MMDIT_CUDA(launch_attn_bwd_pre(at<__nv_bfloat16>(ws, p.o[i]), at<__nv_bfloat16>(ws, bp.dO[i]), B, rpb[i], S,
                                     p.S_pad, off[i], H, amax, at<float>(ws, bp.dsum),
                                     at<__half>(ws, bp.doh), st), "attention pre-pass");
    MMDIT_CUDA(launch_qk_to_f16(at<__nv_bfloat16>(ws, p.q), at<__nv_bfloat16>(ws, p.k),
                                static_cast<int64_t>(bh) * S * 128, at<__half>(ws, bp.q16), at<__half>(ws, bp.k16), st),
               "Q, K to fp16");
    MMDIT_CUDA(launch_untranspose_vt(at<__half>(ws, p.vt), bh, S, p.S_pad, at<__half>(ws, bp.v), st), "V");
  }
  {
    AttnBwdProblem a;
    a.batch = B, a.heads = H, a.seq = S, a.seq_pad = p.S_pad;
    a.q = at<__half>(ws, bp.q16), a.k = at<__half>(ws, bp.k16), a.v = at<__half>(ws, bp.v);
    a.dout = at<__half>(ws, bp.doh);
    a.lse = at<float>(ws, bp.lse), a.dsum = at<float>(ws, bp.dsum);
    a.dq = at<float>(ws, bp.dq), a.dk = at<float>(ws, bp.dk), a.dv = at<float>(ws, bp.dv);
    ProfScope ps_("bwd.attention", st);
    MMDIT_CUDA(launch_attention_bwd(a, status_word(ws), st), "attention backward");
  }
  // ---------------- QK-RMSNorm + RoPE, QKV (both streams' linear backward in shared launches) and
  // LayerNorm backward, the modulation
  {
    ProfScope ps_("bwd.qkv_and_ln1", st);
    for (int i = 0; i < ns; ++i) {
      if (R[i] == 0) continue;
      QkBwdArgs q;
      q.qkv_pre = at(ws, bp.qkv_pre[i]), q.g_q = W[i]->g_q, q.g_k = W[i]->g_k;
      q.cos = rope_cos, q.sin = rope_sin;
      q.dq = at(ws, bp.dq), q.dk = at(ws, bp.dk), q.dv = at(ws, bp.dv), q.dqkv = at(ws, bp.dqkv[i]);
      q.part = part, q.amax = amax;
      q.batch = B, q.seq_s = rpb[i], q.seq_joint = S, q.seq_offset = off[i], q.heads = H, q.hidden = D;
      q.interleaved = d->rope_interleaved ? 1 : 0, q.eps = d->rms_eps;
      MMDIT_CUDA(launch_qk_norm_rope_bwd(act, q, Gs[i]->g_q, Gs[i]->g_k, st), "QK-RMSNorm + RoPE backward");
    }
    {
      const auto dy = ptrs([&](int i) -> const void* { return at(ws, bp.dqkv[i]); });
      const auto xx = ptrs([&](int i) -> const void* { return at(ws, bp.h1[i]); });
      const auto ww = ptrs([&](int i) -> const void* { return W[i]->w_qkv; });
      const auto dx = ptrs([&](int i) -> void* { return at(ws, bp.dh[i]); });
      const auto dw = ptrs([&](int i) -> float* { return Gs[i]->w_qkv; });
      const auto db = ptrs([&](int i) -> float* { return Gs[i]->b_qkv; });
      if ((s = linear_bwd_streams(act, ns, R, 3 * D, D, dy.data(), xx.data(), ww.data(), dx.data(), dw.data(),
                                  db.data(), lin, ws, st)) != MMDIT_OK)
        return s;
    }
    bool dvec_written = false;
    for (int i = 0; i < ns; ++i) {
      const mmdit_stream_grads* g = Gs[i];
      float* dm = at<float>(ws, bp.dm[i]);
      const float* mod = at<float>(ws, p.mod[i]);
      float* dx1 = at<float>(ws, bp.dx1[i]);
      if (R[i] > 0)
        MMDIT_CUDA(launch_ln_modulate_bwd(act, 0, X[i], at(ws, bp.dh[i]), mod + D, bstr, B, rpb[i], D, d->ln_eps,
                                          dx1, dm + D, dm, 0, part, st),
                   "LN1 backward");
      MMDIT_CUDA(launch_modulation_bwd(act, vec, W[i]->w_mod, dm, B, 6 * D, D, g->w_mod, g->b_mod, dvec,
                                       dvec_written ? 1 : 0, part, st),
                 "modulation backward");
      dvec_written = dvec_written || dvec != nullptr;
      if (R[i] > 0)
        MMDIT_CUDA(launch_convert(act, 0, dx1, static_cast<int64_t>(R[i]) * D, DX[i], st), "dx to the activation type");
    }
  }
  return MMDIT_OK;
}

// Workspace of the whole-model forward: one region that every step in turn uses from its start
// (status word first), then the model's own tensors.
struct FluxPlan {
  BlockPlan dbl, sgl;
  size_t vec, mods, x_img, x_txt, c, total;
  int n_mod;
};

bool plan_flux(const mmdit_flux_config* cfg, FluxPlan* f) {
  const mmdit_dims* d = &cfg->block;
  const int B = d->batch, D = d->hidden, Si = d->seq_img, St = d->seq_txt, S = Si + St;
  const size_t e = elt_bytes(d->act);
  size_t region = conditioning_workspace(d->act, B, D, cfg->time_dim);
  auto grow = [&](size_t x) { region = x > region ? x : region; };
  if (!plan_block(d, false, &f->dbl) || !plan_block(d, true, &f->sgl)) return false;
  if (cfg->single_parallel) f->sgl.parallel = true, f->sgl.mod_chunks = 3;
  if (cfg->n_double > 0) grow(f->dbl.total);
  if (cfg->n_single > 0) grow(f->sgl.total);
  grow(mmdit_final_layer_workspace_size(d, cfg->channels));
  grow(mmdit_img_in_workspace_size(d->act, B, cfg->channels, cfg->lat_h, cfg->lat_w));
  grow(mmdit_linear_workspace_size(d->act, B * St, D, cfg->txt_dim));
  Carver c;
  c.off = round_up(region, 256);
  f->n_mod = 2 * cfg->n_double + cfg->n_single;
  f->vec = c.take(static_cast<size_t>(B) * D * e);
  f->mods = c.take(static_cast<size_t>(f->n_mod) * B * 6 * D * 4);
  f->c = c.take(static_cast<size_t>(B) * S * D * e);
  if (B == 1) {
    // one sample: the streams sit back to back inside [img; txt], so joining them is free
    f->x_img = f->c;
    f->x_txt = f->c + static_cast<size_t>(Si) * D * e;
  } else {
    f->x_img = c.take(static_cast<size_t>(B) * Si * D * e);
    f->x_txt = c.take(static_cast<size_t>(B) * St * D * e);
  }
  f->total = c.off;
  return true;
}

mmdit_status check_flux(const mmdit_flux_config* cfg) {
  if (!cfg) return fail(MMDIT_ERR_INVALID_ARG, "flux config is NULL");
  const mmdit_dims* d = &cfg->block;
  mmdit_status s = check_dims(d);
  if (s != MMDIT_OK) return s;
  if (d->gemm != MMDIT_GEMM_NATIVE)
    return fail(MMDIT_ERR_UNSUPPORTED, "whole-model forward: native GEMMs only (FP8 runs per block)");
  if (d->batch < 1 || d->seq_img < 1) return fail(MMDIT_ERR_INVALID_ARG, "whole-model forward: empty batch or image");
  if (cfg->n_double < 0 || cfg->n_single < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative block count");
  if (cfg->single_parallel != 0 && cfg->single_parallel != 1)
    return fail(MMDIT_ERR_INVALID_ARG, "single_parallel must be 0 or 1");
  if (cfg->lat_h < 1 || cfg->lat_w < 1 || d->seq_img != cfg->lat_h * cfg->lat_w)
    return fail(MMDIT_ERR_INVALID_ARG, "seq_img must equal lat_h * lat_w");
  if (cfg->channels < 32 || cfg->channels % 32 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "channels must be a multiple of 32");
  if (d->hidden % 256 != 0) return fail(MMDIT_ERR_UNSUPPORTED, "whole-model forward: hidden must be a multiple of 256");
  if (d->seq_txt > 0 && (cfg->txt_dim < 8 || cfg->txt_dim % 8 != 0))
    return fail(MMDIT_ERR_UNSUPPORTED, "txt_dim must be a positive multiple of 8");
  if (cfg->time_dim < 8 || cfg->time_dim % 8 != 0 || cfg->time_dim > 512)
    return fail(MMDIT_ERR_UNSUPPORTED, "time_dim must be a multiple of 8 in [8, 512]");
  if (cfg->vec_in_dim < 8 || cfg->vec_in_dim % 8 != 0 || cfg->vec_in_dim > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "vec_in_dim must be a multiple of 8 in [8, 6144]");
  if (static_cast<int64_t>(d->batch) * d->heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "batch * heads must be <= 65535");
  return MMDIT_OK;
}

mmdit_status check_cond_w(const mmdit_cond_w* w, bool guided) {
  if (!w) return fail(MMDIT_ERR_INVALID_ARG, "conditioning weights are NULL");
  mmdit_status s = check_ptrs({w->time_in.w1, w->time_in.b1, w->time_in.w2, w->time_in.b2},
                              "timestep embedder weights");
  if (s != MMDIT_OK) return s;
  if ((s = check_ptrs({w->vector_in.w1, w->vector_in.b1, w->vector_in.w2, w->vector_in.b2},
                      "vector embedder weights")) != MMDIT_OK)
    return s;
  if (guided && (s = check_ptrs({w->w_guidance, w->b_guidance}, "guidance weights")) != MMDIT_OK) return s;
  return MMDIT_OK;
}

}  // namespace

extern "C" {

const char* mmdit_last_error(void) { return g_err; }

uint64_t mmdit_launch_count(void) { return g_launches; }
void mmdit_launch_count_reset(void) { g_launches = 0; }

void mmdit_profile_enable(int32_t on) { g_prof_on = on != 0; }

int32_t mmdit_profile_collect(void* stream, char* names_out, size_t names_len, float* ms_out,
                              int32_t max_entries) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  int32_t n = 0;
  size_t used = 0;
  bool ok = true;
  for (int i = 0; i < g_prof_n; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof[i].start, g_prof[i].stop) != cudaSuccess) ok = false;
    const size_t len = strlen(g_prof[i].name) + 1;
    if (n < max_entries && ms_out && names_out && used + len <= names_len) {
      memcpy(names_out + used, g_prof[i].name, len);
      used += len;
      ms_out[n++] = ms;
    }
    cudaEventDestroy(g_prof[i].start);
    cudaEventDestroy(g_prof[i].stop);
  }
  g_prof_n = 0;
  return ok ? n : -1;
}

mmdit_status mmdit_workspace_status(void* workspace, uint32_t* bits_out, void* stream) {
  if (!workspace) return fail(MMDIT_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  MMDIT_CUDA(cudaStreamSynchronize(st), "stream synchronize");
  MMDIT_CUDA(cudaMemcpy(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost), "status read");
  MMDIT_CUDA(cudaMemset(workspace, 0, sizeof(bits)), "status clear");
  if (bits_out) *bits_out = bits;
  if (bits) return fail(MMDIT_ERR_DEVICE, "a kernel gave up a bounded wait (status bits 0x%x)", bits);
  return MMDIT_OK;
}

mmdit_status rope3d_freqs(const float* ids, int32_t batch, int32_t seq, const int32_t* axes_dim,
                          float theta, float* cos_out, float* sin_out, void* stream) {
  if (!axes_dim) return fail(MMDIT_ERR_INVALID_ARG, "axes_dim is NULL");
  if (batch < 0 || seq < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative batch or seq");
  int sum = 0;
  for (int a = 0; a < 3; ++a) {
    if (axes_dim[a] < 0 || axes_dim[a] % 2 != 0)
      return fail(MMDIT_ERR_INVALID_ARG, "axes_dim[%d] = %d must be even and >= 0", a, axes_dim[a]);
    sum += axes_dim[a];
  }
  if (sum > 256) return fail(MMDIT_ERR_UNSUPPORTED, "sum(axes_dim) = %d exceeds 256", sum);
  if (!(theta > 0.f)) return fail(MMDIT_ERR_INVALID_ARG, "theta must be positive");
  if (static_cast<int64_t>(batch) * seq == 0) return MMDIT_OK;
  if (!ids || !cos_out || !sin_out) return fail(MMDIT_ERR_INVALID_ARG, "NULL ids or output");
  const int axes[3] = {axes_dim[0], axes_dim[1], axes_dim[2]};
  pdl_begin_call();
  ProfScope ps_("rope3d_freqs", static_cast<cudaStream_t>(stream));
  MMDIT_CUDA(launch_rope3d(ids, batch, seq, axes, theta, cos_out, sin_out,
                           static_cast<cudaStream_t>(stream)),
             "rope3d_freqs");
  return MMDIT_OK;
}

mmdit_status mmdit_modulation_fwd(int32_t act, int32_t batch, int32_t rows, int32_t dim, const void* vec,
                                  const void* w, const void* bias, float* out, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 0 || rows < 0 || dim < 1) return fail(MMDIT_ERR_INVALID_ARG, "bad modulation shape");
  if (dim % 8 != 0 || dim > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "modulation: dim must be a multiple of 8, at most 6144 (got %d)", dim);
  if (static_cast<int64_t>(batch) * rows == 0) return MMDIT_OK;
  mmdit_status s = check_ptrs({vec, w, out}, "modulation");
  if (s != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pdl_begin_call();
  ProfScope ps_("modulation", st);
  MMDIT_CUDA(launch_modulation(act, vec, w, bias, batch, rows, dim, out, st), "modulation");
  return MMDIT_OK;
}

size_t flow_match_workspace_size(int32_t batch, int64_t n_per_sample) {
  // the partial-sum count saturates at kFlowMaxPartials, so a product that would overflow
  // needs the same workspace as any other large call
  const int64_t b = batch > 0 ? batch : 0, n1 = n_per_sample > 0 ? n_per_sample : 0;
  const int64_t n = b > 0 && n1 > INT64_MAX / b ? INT64_MAX : b * n1;
  return kStatusBytes + round_up(static_cast<size_t>(flow_partial_blocks(n)) * sizeof(float), 256);
}

mmdit_status flow_match_noise_and_loss(int32_t dtype, const void* z0, const void* z1, const float* t,
                                       int32_t batch, int64_t n_per_sample, void* z_t,
                                       const void* pred, float* loss, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (dtype != MMDIT_F32 && dtype != MMDIT_BF16)
    return fail(MMDIT_ERR_INVALID_ARG, "dtype must be MMDIT_F32 or MMDIT_BF16");
  if (batch < 0 || n_per_sample < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative size");
  if (n_per_sample % 8 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "n_per_sample must be a multiple of 8 (got %lld)",
                static_cast<long long>(n_per_sample));
  if (batch > 0 && n_per_sample > INT64_MAX / batch)
    return fail(MMDIT_ERR_INVALID_ARG, "batch * n_per_sample overflows a 64-bit count");
  if ((pred == nullptr) != (loss == nullptr))
    return fail(MMDIT_ERR_INVALID_ARG, "pred and loss must both be given or both be NULL");
  mmdit_status s = check_ptrs({z0, z1}, "flow_match latents");
  if (s != MMDIT_OK) return s;
  if (z_t && (s = check_ptrs({z_t, t}, "flow_match z_t/t")) != MMDIT_OK) return s;
  if (pred && (s = check_ptrs({pred, loss}, "flow_match pred/loss")) != MMDIT_OK) return s;
  if (pred && z_t && (z_t == z0 || z_t == z1))
    return fail(MMDIT_ERR_INVALID_ARG, "z_t may not alias z0/z1 when the loss is requested");
  if ((s = check_workspace(workspace, workspace_bytes,
                           flow_match_workspace_size(batch, n_per_sample))) != MMDIT_OK)
    return s;
  const int64_t n = static_cast<int64_t>(batch) * n_per_sample;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  ProfScope ps_(pred ? (z_t ? "flow_match.noise_loss" : "flow_match.loss") : "flow_match.noise", st);
  MMDIT_CUDA(launch_flow_match(dtype, z0, z1, t, batch, n_per_sample, z_t, pred, loss,
                               at<float>(workspace, kStatusBytes), flow_partial_blocks(n), st),
             "flow_match_noise_and_loss");
  return MMDIT_OK;
}

mmdit_status flow_match_euler_step(int32_t dtype, int64_t n, const void* z, const void* v_cond,
                                   const void* v_uncond, float guidance, float dt, void* z_out,
                                   void* stream) {
  if (dtype != MMDIT_F32 && dtype != MMDIT_BF16)
    return fail(MMDIT_ERR_INVALID_ARG, "dtype must be MMDIT_F32 or MMDIT_BF16");
  if (n < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative element count");
  if (n % 8 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "n must be a multiple of 8 (got %lld)", static_cast<long long>(n));
  if (n == 0) return MMDIT_OK;
  mmdit_status s = check_ptrs({z, v_cond, z_out}, "Euler step");
  if (s != MMDIT_OK) return s;
  if (v_uncond && !aligned16(v_uncond))
    return fail(MMDIT_ERR_INVALID_ARG, "Euler step: v_uncond is not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pdl_begin_call();
  ProfScope ps_("flow_match.euler_step", st);
  MMDIT_CUDA(launch_euler_cfg(dtype, n, z, v_cond, v_uncond, guidance, dt, z_out, st), "Euler step");
  return MMDIT_OK;
}

size_t mmdit_linear_workspace_size(int32_t act, int32_t M, int32_t N, int32_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return kStatusBytes;
  const int splits = choose_splits(M, N, K, static_cast<int>(elt_bytes(act)));
  if (splits <= 1) return kStatusBytes;
  Carver c;
  c.take(static_cast<size_t>(splits) * M * N * sizeof(float));
  return c.off;
}

mmdit_status mmdit_linear_fwd(int32_t act, int32_t M, int32_t N, int32_t K, const void* x,
                              const void* w, const void* b, void* y, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (M < 0 || N <= 0 || K <= 0) return fail(MMDIT_ERR_INVALID_ARG, "bad shape M=%d N=%d K=%d", M, N, K);
  if (N % 32 != 0 || K % 8 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "N must be a multiple of 32 and K of 8 (N=%d, K=%d)", N, K);
  mmdit_status s = check_ptrs({x, w, y}, "linear");
  if (s != MMDIT_OK) return s;
  if (b && !aligned16(b)) return fail(MMDIT_ERR_INVALID_ARG, "linear: bias not 16-byte aligned");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_linear_workspace_size(act, M, N, K))) !=
      MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return linear_body(act, M, N, K, x, w, b, y, workspace, st);
}

size_t mmdit_img_in_workspace_size(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                                   int32_t lat_w) {
  Carver c;
  c.take(static_cast<size_t>(batch > 0 ? batch : 0) * (lat_h > 0 ? lat_h : 0) *
         (lat_w > 0 ? lat_w : 0) * (channels > 0 ? channels : 0) * elt_bytes(act));
  return c.off;
}

mmdit_status mmdit_img_in_fwd(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                              int32_t lat_w, int32_t hidden, const float* z, const void* w,
                              const void* b, void* out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 1 || channels < 1 || lat_h < 1 || lat_w < 1 || hidden < 1)
    return fail(MMDIT_ERR_INVALID_ARG, "bad img_in shape");
  if (channels % 8 != 0 || hidden % 32 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "channels must be a multiple of 8 and hidden of 32");
  mmdit_status s = check_ptrs({z, w, b, out}, "img_in");
  if (s != MMDIT_OK) return s;
  if ((s = check_workspace(workspace, workspace_bytes,
                           mmdit_img_in_workspace_size(act, batch, channels, lat_h, lat_w))) != MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return img_in_body(act, batch, channels, lat_h, lat_w, hidden, z, w, b, out, workspace, st);
}

mmdit_status mmdit_img_in_noise_fwd(int32_t act, int32_t batch, int32_t channels, int32_t lat_h,
                                    int32_t lat_w, int32_t hidden, const float* z0, const float* z1,
                                    const float* t, const void* w, const void* b, void* out,
                                    float* z_t, void* workspace, size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 1 || channels < 1 || lat_h < 1 || lat_w < 1 || hidden < 1)
    return fail(MMDIT_ERR_INVALID_ARG, "bad img_in shape");
  if (channels % 8 != 0 || hidden % 32 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "channels must be a multiple of 8 and hidden of 32");
  mmdit_status s = check_ptrs({z0, z1, t, w, b, out}, "img_in + noise");
  if (s != MMDIT_OK) return s;
  if (z_t && (s = check_ptrs({z_t}, "img_in + noise: z_t")) != MMDIT_OK) return s;
  if (z_t && (z_t == z0 || z_t == z1))
    return fail(MMDIT_ERR_INVALID_ARG, "img_in + noise: z_t may not alias z0 or z1");
  if ((s = check_workspace(workspace, workspace_bytes,
                           mmdit_img_in_workspace_size(act, batch, channels, lat_h, lat_w))) != MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return img_in_body(act, batch, channels, lat_h, lat_w, hidden, z0, w, b, out, workspace, st, z1, t, z_t);
}

size_t mmdit_final_layer_workspace_size(const mmdit_dims* d, int32_t channels) {
  if (!d || d->batch < 1 || d->hidden < 1 || d->seq_img < 0 || channels < 1) return 0;
  return plan_head(d, channels, false).total;
}

size_t mmdit_final_layer_loss_workspace_size(const mmdit_dims* d, int32_t channels) {
  if (!d || d->batch < 1 || d->hidden < 1 || d->seq_img < 0 || channels < 1) return 0;
  return plan_head(d, channels, true).total;
}

mmdit_status mmdit_final_layer_fwd(const mmdit_dims* d, int32_t channels, int32_t lat_h,
                                   int32_t lat_w, const void* x_img, const void* vec,
                                   const void* w_ada, const void* b_ada, const void* w_out,
                                   const void* b_out, float* pred, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!d) return fail(MMDIT_ERR_INVALID_ARG, "dims is NULL");
  if (d->act != MMDIT_F32 && d->act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act");
  if (d->batch < 1 || lat_h < 1 || lat_w < 1 || d->seq_img != lat_h * lat_w)
    return fail(MMDIT_ERR_INVALID_ARG, "final layer: seq_img must equal lat_h * lat_w");
  if (channels < 32 || channels % 32 != 0 || d->hidden % 256 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "final layer: channels multiple of 32, hidden of 256");
  mmdit_status s = check_ptrs({x_img, vec, w_ada, b_ada, w_out, b_out, pred}, "final layer");
  if (s != MMDIT_OK) return s;
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_final_layer_workspace_size(d, channels))) !=
      MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return final_layer_body(d, channels, x_img, vec, w_ada, b_ada, w_out, b_out, pred, workspace, st);
}

mmdit_status mmdit_final_layer_loss_fwd(const mmdit_dims* d, int32_t channels, int32_t lat_h,
                                        int32_t lat_w, const void* x_img, const void* vec,
                                        const void* w_ada, const void* b_ada, const void* w_out,
                                        const void* b_out, const float* z0, const float* z1,
                                        float* pred, float* loss, const float* mod, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!d) return fail(MMDIT_ERR_INVALID_ARG, "dims is NULL");
  if (d->act != MMDIT_F32 && d->act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act");
  if (d->batch < 1 || lat_h < 1 || lat_w < 1 || d->seq_img != lat_h * lat_w)
    return fail(MMDIT_ERR_INVALID_ARG, "final layer + loss: seq_img must equal lat_h * lat_w");
  if (channels < 32 || channels % 32 != 0 || d->hidden % 256 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "final layer + loss: channels multiple of 32, hidden of 256");
  mmdit_status s = check_ptrs({x_img, vec, w_ada, b_ada, w_out, b_out, z0, z1}, "final layer + loss");
  if (s != MMDIT_OK) return s;
  // the loss is one fp32 scalar: its own alignment is enough
  if (!loss || (reinterpret_cast<uintptr_t>(loss) & 3u))
    return fail(MMDIT_ERR_INVALID_ARG, "final layer + loss: loss is NULL or not 4-byte aligned");
  if (pred && (s = check_ptrs({pred}, "final layer + loss: pred")) != MMDIT_OK) return s;
  if (pred && (pred == z0 || pred == z1))
    return fail(MMDIT_ERR_INVALID_ARG, "final layer + loss: pred may not alias z0 or z1");
  if (mod && !aligned16(mod)) return fail(MMDIT_ERR_INVALID_ARG, "final layer + loss: mod is not 16-byte aligned");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_final_layer_loss_workspace_size(d, channels))) !=
      MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word and the loss ticket counter (both inside the status region)
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, kStatusBytes, st), "status clear");
  pdl_begin_call();
  return final_layer_body(d, channels, x_img, vec, w_ada, b_ada, w_out, b_out, pred, workspace, st, z0,
                          z1, loss, mod);
}


mmdit_status mmdit_ln_modulate_fwd(int32_t act, int32_t x_f32, int32_t batch, int32_t rows_per_batch,
                                   int32_t dim, float eps, const void* x, const float* shift,
                                   const float* scale, int64_t mod_bstride, void* out, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 0 || rows_per_batch < 0 || dim < 1 || mod_bstride < 0 || !(eps >= 0.f))
    return fail(MMDIT_ERR_INVALID_ARG, "LayerNorm-modulate: bad shape or eps");
  if (dim % 8 != 0 || dim > 8192)
    return fail(MMDIT_ERR_UNSUPPORTED, "LayerNorm-modulate: dim must be a multiple of 8, at most 8192 (got %d)", dim);
  const int64_t rows = static_cast<int64_t>(batch) * rows_per_batch;
  if (rows > INT32_MAX) return fail(MMDIT_ERR_UNSUPPORTED, "LayerNorm-modulate: more than 2^31 - 1 rows");
  if (rows == 0) return MMDIT_OK;
  if (mod_bstride % 4 != 0)
    return fail(MMDIT_ERR_INVALID_ARG, "LayerNorm-modulate: mod_bstride must be a multiple of 4 (16-byte rows)");
  mmdit_status s = check_ptrs({x, shift, scale, out}, "LayerNorm-modulate");
  if (s != MMDIT_OK) return s;
  if (out == x) return fail(MMDIT_ERR_INVALID_ARG, "LayerNorm-modulate: out may not alias x");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pdl_begin_call();
  ProfScope ps_("ln_modulate", st);
  MMDIT_CUDA(launch_ln_modulate(act, x_f32 ? 1 : 0, x, shift, scale, mod_bstride, static_cast<int>(rows),
                                rows_per_batch, dim, eps, out, st),
             "LayerNorm-modulate");
  return MMDIT_OK;
}

mmdit_status mmdit_copy_rows(void* dst, int64_t dst_stride, const void* src, int64_t src_stride,
                             int64_t row_bytes, int32_t n_rows, void* stream) {
  if (n_rows < 0 || row_bytes < 0 || dst_stride < row_bytes || src_stride < row_bytes)
    return fail(MMDIT_ERR_INVALID_ARG, "copy_rows: bad sizes or strides");
  if (n_rows == 0 || row_bytes == 0) return MMDIT_OK;
  if (!dst || !src) return fail(MMDIT_ERR_INVALID_ARG, "copy_rows: NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemcpy2DAsync(dst, static_cast<size_t>(dst_stride), src, static_cast<size_t>(src_stride),
                               static_cast<size_t>(row_bytes), static_cast<size_t>(n_rows),
                               cudaMemcpyDeviceToDevice, st),
             "copy_rows");
  pdl_begin_call();  // a later kernel of this thread follows a copy, not a kernel
  return MMDIT_OK;
}

size_t mmdit_attention_workspace_size(int32_t batch, int32_t heads, int32_t seq) {
  if (batch < 1 || heads < 1 || seq < 1) return kStatusBytes;
  Carver c;
  c.take(static_cast<size_t>(batch) * heads * 128 * round_up(static_cast<size_t>(seq), 8) * 2);
  return c.off;
}

mmdit_status mmdit_attention_fwd(int32_t act, int32_t batch, int32_t heads, int32_t seq,
                                 int32_t head_dim, const void* q, const void* k, const void* v,
                                 void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (head_dim != 128) return fail(MMDIT_ERR_UNSUPPORTED, "head_dim must be 128");
  if (batch < 1 || heads < 1 || seq < 1) return fail(MMDIT_ERR_INVALID_ARG, "bad attention shape");
  if (static_cast<int64_t>(batch) * heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "batch * heads must be <= 65535");
  mmdit_status s = check_ptrs({q, k, v, out}, "attention");
  if (s != MMDIT_OK) return s;
  if ((s = check_workspace(workspace, workspace_bytes,
                           mmdit_attention_workspace_size(batch, heads, seq))) != MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  const int seq_pad = static_cast<int>(round_up(static_cast<size_t>(seq), 8));
  __half* vt = at<__half>(workspace, kStatusBytes);
  ProfScope ps_("attention", st);
  MMDIT_CUDA(launch_transpose_v(static_cast<const __nv_bfloat16*>(v), batch * heads, seq, seq_pad, vt, st),
             "V transpose");
  AttnProblem a;
  a.act = act, a.batch = batch, a.heads = heads, a.seq = seq, a.seq_pad = seq_pad, a.split = seq;
  a.q = static_cast<const __nv_bfloat16*>(q), a.k = static_cast<const __nv_bfloat16*>(k), a.vt = vt;
  a.out0 = out, a.out1 = nullptr;
  MMDIT_CUDA(launch_attention(a, status_word(workspace), st), "attention");
  return MMDIT_OK;
}

size_t mmdit_double_block_workspace_size(const mmdit_dims* d) {
  BlockPlan p;
  if (check_dims(d) != MMDIT_OK || !plan_block(d, false, &p)) return 0;
  return p.total;
}

size_t mmdit_single_block_workspace_size(const mmdit_dims* d) {
  BlockPlan p;
  if (check_dims(d) != MMDIT_OK || !plan_block(d, true, &p)) return 0;
  return p.total;
}

int32_t mmdit_block_workspace_offsets(const mmdit_dims* d, int32_t single, int64_t* out, int32_t n) {
  BlockPlan p;
  if (!out || check_dims(d) != MMDIT_OK || !plan_block(d, single != 0, &p)) return -1;
  const int64_t none = -1;
  auto two = [&](size_t off, int s) { return (single && s == 1) ? none : static_cast<int64_t>(off); };
  auto f8 = [&](size_t off, int s) { return p.fp8 ? two(off, s) : none; };
  const int64_t v[17] = {two(p.mod[0], 0), two(p.mod[1], 1), static_cast<int64_t>(p.q),
                         static_cast<int64_t>(p.k), static_cast<int64_t>(p.vt), two(p.o[0], 0),
                         two(p.o[1], 1), two(p.x1[0], 0), two(p.x1[1], 1), two(p.u[0], 0),
                         two(p.h[0], 0), two(p.h[1], 1), two(p.u[1], 1), f8(p.o8[0], 0),
                         f8(p.o8[1], 1), f8(p.wq[0], 0), f8(p.wq[1], 1)};
  const int m = n < 17 ? n : 17;
  for (int i = 0; i < m; ++i) out[i] = v[i];
  return m;
}

mmdit_status mmdit_double_block_fwd(const mmdit_dims* d, const mmdit_stream_w* w_img,
                                    const mmdit_stream_w* w_txt, const void* vec,
                                    const float* rope_cos, const float* rope_sin, const void* x_img,
                                    const void* x_txt, void* y_img, void* y_txt, mmdit_fp8_state* fp8,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  mmdit_status s = check_dims(d);
  if (s != MMDIT_OK) return s;
  if ((s = check_fp8(d, fp8, 2 * kFp8TensorsPerStream)) != MMDIT_OK) return s;
  if ((s = check_stream_w(w_img, "image weights")) != MMDIT_OK) return s;
  if ((s = check_stream_w(w_txt, "text weights")) != MMDIT_OK) return s;
  if ((s = check_ptrs({vec, rope_cos, rope_sin}, "double block conditioning")) != MMDIT_OK) return s;
  if (d->seq_img > 0 && (s = check_ptrs({x_img, y_img}, "image stream")) != MMDIT_OK) return s;
  if (d->seq_txt > 0 && (s = check_ptrs({x_txt, y_txt}, "text stream")) != MMDIT_OK) return s;
  if (static_cast<int64_t>(d->batch) * d->heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "batch * heads must be <= 65535");
  BlockPlan p;
  plan_block(d, false, &p);
  if ((s = check_workspace(workspace, workspace_bytes, p.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return double_block_body(d, p, w_img, w_txt, vec, rope_cos, rope_sin, x_img, x_txt, y_img, y_txt, fp8,
                           workspace, st);
}

mmdit_status mmdit_single_block_fwd(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec,
                                    const float* rope_cos, const float* rope_sin, const void* x,
                                    void* y, mmdit_fp8_state* fp8, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  mmdit_status s = check_dims(d);
  if (s != MMDIT_OK) return s;
  if ((s = check_fp8(d, fp8, kFp8TensorsPerStream)) != MMDIT_OK) return s;
  if ((s = check_stream_w(w, "single-block weights")) != MMDIT_OK) return s;
  if ((s = check_ptrs({vec, rope_cos, rope_sin, x, y}, "single block")) != MMDIT_OK) return s;
  if (static_cast<int64_t>(d->batch) * d->heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "batch * heads must be <= 65535");
  BlockPlan p;
  plan_block(d, true, &p);
  if ((s = check_workspace(workspace, workspace_bytes, p.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return single_block_body(d, p, w, vec, rope_cos, rope_sin, x, y, fp8, workspace, st);
}

mmdit_status mmdit_fp8_quantize_e4m3(const void* x, int64_t n, const float* scale, float* amax,
                                     void* out, void* stream) {
  if (n < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative element count");
  if (n % 16 != 0) return fail(MMDIT_ERR_UNSUPPORTED, "n must be a multiple of 16 (got %lld)",
                               static_cast<long long>(n));
  if (n == 0) return MMDIT_OK;
  mmdit_status s = check_ptrs({x, out}, "E4M3 cast");
  if (s != MMDIT_OK) return s;
  if (!scale || !amax) return fail(MMDIT_ERR_INVALID_ARG, "E4M3 cast: NULL scale or amax");
  if ((reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return fail(MMDIT_ERR_INVALID_ARG, "E4M3 cast: scale and amax must be 4-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const QuantJob job{static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(out), n, scale, amax};
  pdl_begin_call();
  ProfScope ps_("fp8_quantize", st);
  MMDIT_CUDA(launch_quantize_e4m3(&job, 1, st), "E4M3 cast");
  return MMDIT_OK;
}

size_t mmdit_fp8_linear_workspace_size(void) { return kStatusBytes; }

mmdit_status mmdit_fp8_linear_fwd(int32_t M, int32_t N, int32_t K, const void* x, const void* w,
                                  const float* scale_x, const float* scale_w, const void* b, void* y,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 1 || K < 1) return fail(MMDIT_ERR_INVALID_ARG, "bad FP8 linear shape");
  if (N % 128 != 0 || K % 16 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "FP8 linear needs N %% 128 == 0 and K %% 16 == 0 (got %d, %d)", N, K);
  mmdit_status s = check_ptrs({x, w, y}, "FP8 linear");
  if (s != MMDIT_OK) return s;
  if (b && !aligned16(b)) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear: bias is not 16-byte aligned");
  if (!scale_x || !scale_w) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear: NULL scale");
  if ((s = check_workspace(workspace, workspace_bytes, kStatusBytes)) != MMDIT_OK) return s;
  if (M == 0) return MMDIT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  GemmProblem g;
  g.act = 2, g.epi = kEpiBias, g.M = M, g.N = N, g.K = K, g.A = x, g.W = w;
  g.ep.bias = b, g.ep.out = y, g.ep.scale_a = scale_x, g.ep.scale_w = scale_w;
  ProfScope ps_("fp8_linear", st);
  MMDIT_CUDA(launch_gemm(g, status_word(workspace), st), "FP8 linear");
  return MMDIT_OK;
}

size_t mmdit_fp8_blockwise_linear_workspace_size(int32_t M, int32_t N, int32_t K) {
  if (M < 0 || N < 1 || K < 1) return kStatusBytes;
  return kStatusBytes + blockwise_linear_scratch(M, N, K);
}

mmdit_status mmdit_fp8_blockwise_linear_fwd(int32_t M, int32_t N, int32_t K, const void* x, const void* w,
                                            const void* b, void* y, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  if (M < 0 || N < 1 || K < 1) return fail(MMDIT_ERR_INVALID_ARG, "bad blockwise FP8 linear shape");
  if (N % 128 != 0 || K % 128 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "blockwise FP8 linear needs N %% 128 == 0 and K %% 128 == 0 (got %d, %d)", N, K);
  if (M > 65535 * 128) return fail(MMDIT_ERR_UNSUPPORTED, "blockwise FP8 linear: M must be <= %d", 65535 * 128);
  mmdit_status s = check_ptrs({x, w, y}, "blockwise FP8 linear");
  if (s != MMDIT_OK) return s;
  if (b && !aligned16(b)) return fail(MMDIT_ERR_INVALID_ARG, "blockwise FP8 linear: bias is not 16-byte aligned");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_fp8_blockwise_linear_workspace_size(M, N, K))) != MMDIT_OK)
    return s;
  if (M == 0) return MMDIT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  ProfScope ps_("fp8_blockwise_linear", st);
  MMDIT_CUDA(launch_blockwise_linear(M, N, K, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w),
                                     static_cast<const __nv_bfloat16*>(b), static_cast<__nv_bfloat16*>(y),
                                     at(workspace, kStatusBytes), status_word(workspace), st),
             "blockwise FP8 linear");
  return MMDIT_OK;
}

size_t mmdit_fp8_mxfp8_linear_workspace_size(int32_t M, int32_t N, int32_t K) {
  if (M < 0 || N < 1 || K < 1) return kStatusBytes;
  return kStatusBytes + mx_linear_scratch(M, N, K);
}

mmdit_status mmdit_fp8_mxfp8_linear_fwd(int32_t M, int32_t N, int32_t K, const void* x, const void* w, const void* b,
                                        void* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 1 || K < 1) return fail(MMDIT_ERR_INVALID_ARG, "bad MXFP8 linear shape");
  if (N % 32 != 0 || K % 32 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "MXFP8 linear needs N %% 32 == 0 and K %% 32 == 0 (got %d, %d)", N, K);
  mmdit_status s = check_ptrs({x, w, y}, "MXFP8 linear");
  if (s != MMDIT_OK) return s;
  if (b && !aligned16(b)) return fail(MMDIT_ERR_INVALID_ARG, "MXFP8 linear: bias is not 16-byte aligned");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_fp8_mxfp8_linear_workspace_size(M, N, K))) != MMDIT_OK)
    return s;
  if (M == 0) return MMDIT_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  ProfScope ps_("fp8_mxfp8_linear", st);
  MMDIT_CUDA(launch_mx_linear(M, N, K, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w),
                              static_cast<const __nv_bfloat16*>(b), static_cast<__nv_bfloat16*>(y),
                              at(workspace, kStatusBytes), status_word(workspace), st),
             "MXFP8 linear");
  return MMDIT_OK;
}

mmdit_status mmdit_single_block_parallel_fwd(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec,
                                             const float* rope_cos, const float* rope_sin, const void* x,
                                             void* y, void* workspace, size_t workspace_bytes, void* stream) {
  mmdit_status s = check_dims(d);
  if (s != MMDIT_OK) return s;
  if (d->gemm != MMDIT_GEMM_NATIVE)
    return fail(MMDIT_ERR_UNSUPPORTED, "parallel single block: native GEMMs only");
  if ((s = check_stream_w(w, "parallel single-block weights")) != MMDIT_OK) return s;
  if ((s = check_ptrs({vec, rope_cos, rope_sin, x, y}, "parallel single block")) != MMDIT_OK) return s;
  if (static_cast<int64_t>(d->batch) * d->heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "batch * heads must be <= 65535");
  BlockPlan p;
  plan_block(d, true, &p);
  p.parallel = true, p.mod_chunks = 3;
  if ((s = check_workspace(workspace, workspace_bytes, p.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return single_block_body(d, p, w, vec, rope_cos, rope_sin, x, y, nullptr, workspace, st);
}

size_t mmdit_linear_bwd_workspace_size(int32_t act, int32_t M, int32_t N, int32_t K) {
  if (M < 0 || N <= 0 || K <= 0) return kStatusBytes;
  const size_t e = elt_bytes(act), Mp = round_up(static_cast<size_t>(M), 8);
  Carver c;
  c.take(static_cast<size_t>(K) * N * e);   // W^T
  c.take(static_cast<size_t>(N) * Mp * e);  // dy^T (rows padded with zeros to a multiple of 8)
  c.take(static_cast<size_t>(K) * Mp * e);  // x^T
  c.take(static_cast<size_t>(kColsumChunks) * N * 4);  // partial column sums of dy
  return c.off;
}

mmdit_status mmdit_linear_bwd(int32_t act, int32_t M, int32_t N, int32_t K, const void* dy, const void* x,
                              const void* w, void* dx, float* dw, float* db, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (M < 0 || N <= 0 || K <= 0) return fail(MMDIT_ERR_INVALID_ARG, "bad shape M=%d N=%d K=%d", M, N, K);
  if (K % 32 != 0 || N % 8 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "linear backward: K must be a multiple of 32 and N of 8 (K=%d, N=%d)", K, N);
  mmdit_status s = MMDIT_OK;
  if (M > 0 && (dx || dw || db) && (s = check_ptrs({dy}, "linear backward dy")) != MMDIT_OK) return s;
  if (dx && ((s = check_ptrs({w, dx}, "linear backward dx")) != MMDIT_OK)) return s;
  if (dw && ((s = check_ptrs({dw}, "linear backward dW")) != MMDIT_OK)) return s;
  if (dw && M > 0 && ((s = check_ptrs({x}, "linear backward x")) != MMDIT_OK)) return s;
  if (db && !aligned16(db)) return fail(MMDIT_ERR_INVALID_ARG, "linear backward: db not 16-byte aligned");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_linear_bwd_workspace_size(act, M, N, K))) != MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  if (M == 0) {  // an empty batch: zero weight and bias gradients, nothing else
    if (dw) MMDIT_CUDA(cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * K * 4, st), "dW clear");
    if (db) MMDIT_CUDA(cudaMemsetAsync(db, 0, static_cast<size_t>(N) * 4, st), "db clear");
    return MMDIT_OK;
  }
  pdl_begin_call();
  ProfScope ps_("linear_bwd", st);
  return linear_bwd_body(act, M, N, K, dy, x, w, dx, dw, db, at(workspace, kStatusBytes), workspace, st);
}

size_t mmdit_conditioning_workspace_size(int32_t act, int32_t batch, int32_t hidden, int32_t time_dim) {
  if (batch < 1 || hidden < 1 || time_dim < 1) return kStatusBytes;
  return conditioning_workspace(act, batch, hidden, time_dim);
}

mmdit_status mmdit_conditioning_fwd(int32_t act, int32_t batch, int32_t hidden, int32_t time_dim,
                                    int32_t vec_in_dim, const mmdit_cond_w* w, const float* t,
                                    const void* y, const float* guidance, void* vec, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 0) return fail(MMDIT_ERR_INVALID_ARG, "negative batch");
  if (hidden < 8 || hidden % 8 != 0 || hidden > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "hidden must be a multiple of 8 in [8, 6144] (got %d)", hidden);
  if (time_dim < 8 || time_dim % 8 != 0 || time_dim > 512)
    return fail(MMDIT_ERR_UNSUPPORTED, "time_dim must be a multiple of 8 in [8, 512] (got %d)", time_dim);
  if (vec_in_dim < 8 || vec_in_dim % 8 != 0 || vec_in_dim > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "vec_in_dim must be a multiple of 8 in [8, 6144] (got %d)", vec_in_dim);
  mmdit_status s = check_cond_w(w, guidance != nullptr);
  if (s != MMDIT_OK) return s;
  if (batch == 0) return MMDIT_OK;
  if ((s = check_ptrs({t, y, vec}, "conditioning")) != MMDIT_OK) return s;
  if ((s = check_workspace(workspace, workspace_bytes,
                           mmdit_conditioning_workspace_size(act, batch, hidden, time_dim))) != MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  return conditioning_body(act, batch, hidden, time_dim, vec_in_dim, w, t, y, guidance, vec, workspace, st);
}

static mmdit_status check_block_bwd(const mmdit_dims* d, bool single) {
  mmdit_status s = check_dims(d);
  if (s != MMDIT_OK) return s;
  if (d->act != MMDIT_BF16) return fail(MMDIT_ERR_UNSUPPORTED, "block backward: bf16 activations only");
  if (d->gemm != MMDIT_GEMM_NATIVE) return fail(MMDIT_ERR_UNSUPPORTED, "block backward: native (bf16) linears only");
  if (d->batch > 8) return fail(MMDIT_ERR_UNSUPPORTED, "block backward: batch must be at most 8 (got %d)", d->batch);
  if (!single && (d->seq_img < 1 || d->seq_txt < 1))
    return fail(MMDIT_ERR_UNSUPPORTED, "double block backward: both streams need rows (S_i=%d, S_t=%d)", d->seq_img,
                d->seq_txt);
  if (d->mlp_hidden % 32 != 0) return fail(MMDIT_ERR_UNSUPPORTED, "block backward: mlp_hidden must be a multiple of 32");
  return MMDIT_OK;
}

static mmdit_status check_grads(const mmdit_stream_grads* g, const char* what) {
  if (!g) return MMDIT_OK;
  const float* p[12] = {g->w_mod, g->b_mod, g->w_qkv, g->b_qkv, g->g_q, g->g_k, g->w_o, g->b_o, g->w_1, g->b_1,
                        g->w_2, g->b_2};
  for (int i = 0; i < 12; ++i)
    if (p[i] && !aligned16(p[i])) return fail(MMDIT_ERR_INVALID_ARG, "%s: gradient %d is not 16-byte aligned", what, i);
  return MMDIT_OK;
}

// FP8 linear backward workspace: the gradient's codes G [M, N], W^T codes [K, N], and for the FP8
// weight gradient G^T [N, Mp] and x^T codes [K, Mp] (Mp = M rounded up to 16, zero columns), or
// the bf16 linear-backward scratch for the unquantised weight gradient; the bias gradient's
// partial column sums.
struct Fp8BwdPlan {
  size_t g, wt, gt, xt, lin, part, total;
  int Mp;
};
Fp8BwdPlan plan_fp8_bwd(int M, int N, int K, int fp8_wgrad) {
  Fp8BwdPlan p;
  Carver c;
  p.Mp = static_cast<int>(round_up(static_cast<size_t>(M > 0 ? M : 0), 16));
  p.g = c.take(static_cast<size_t>(M) * N);
  p.wt = c.take(static_cast<size_t>(K) * N);
  p.gt = fp8_wgrad ? c.take(static_cast<size_t>(N) * p.Mp) : 0;
  p.xt = fp8_wgrad ? c.take(static_cast<size_t>(K) * p.Mp) : 0;
  p.lin = fp8_wgrad ? 0 : c.take(linear_bwd_scratch(2, static_cast<size_t>(M), N, K));
  p.part = c.take(static_cast<size_t>(kColsumChunks) * N * 4);
  p.total = c.off;
  return p;
}

size_t mmdit_fp8_linear_bwd_workspace_size(int32_t M, int32_t N, int32_t K, int32_t fp8_wgrad) {
  if (M < 0 || N <= 0 || K <= 0) return kStatusBytes;
  return plan_fp8_bwd(M, N, K, fp8_wgrad).total;
}

mmdit_status mmdit_fp8_linear_bwd(int32_t M, int32_t N, int32_t K, int32_t recipe, int32_t fp8_wgrad,
                                  const void* dy, const void* x_q, const void* w_q, const void* x,
                                  const float* scale_x, const float* scale_w, const float* scale_dy,
                                  float* amax_dy, void* dx, float* dw, float* db, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear backward: bad shape M=%d N=%d K=%d", M, N, K);
  if (recipe != 0 && recipe != 1)
    return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear backward: recipe must be 0 (e4m3) or 1 (hybrid), got %d", recipe);
  if (fp8_wgrad != 0 && fp8_wgrad != 1) return fail(MMDIT_ERR_INVALID_ARG, "fp8_wgrad must be 0 or 1");
  if (K % 128 != 0 || N % 16 != 0)
    return fail(MMDIT_ERR_UNSUPPORTED, "FP8 linear backward: K must be a multiple of 128 and N of 16 (K=%d, N=%d)", K, N);
  mmdit_status s = check_ptrs({dy, w_q, dx}, "FP8 linear backward");
  if (s != MMDIT_OK) return s;
  if (!scale_x || !scale_w || !scale_dy || !amax_dy)
    return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear backward: NULL scale or amax");
  if (dw && !aligned16(dw)) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear backward: dW not 16-byte aligned");
  if (db && !aligned16(db)) return fail(MMDIT_ERR_INVALID_ARG, "FP8 linear backward: db not 16-byte aligned");
  if (dw && fp8_wgrad && (s = check_ptrs({x_q}, "FP8 linear backward x_q")) != MMDIT_OK) return s;
  if (dw && !fp8_wgrad && (s = check_ptrs({x}, "FP8 linear backward x")) != MMDIT_OK) return s;
  const Fp8BwdPlan fp = plan_fp8_bwd(M, N, K, fp8_wgrad);
  if ((s = check_workspace(workspace, workspace_bytes, fp.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  if (M == 0) {
    if (dw) MMDIT_CUDA(cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * K * 4, st), "dW clear");
    if (db) MMDIT_CUDA(cudaMemsetAsync(db, 0, static_cast<size_t>(N) * 4, st), "db clear");
    return MMDIT_OK;
  }
  pdl_begin_call();
  ProfScope ps_("fp8_linear_bwd", st);
  uint8_t* g = at<uint8_t>(workspace, fp.g);
  // G = Qg(dy scale_dy): E4M3 or, under the hybrid recipe, E5M2; amax_dy records max |dy|
  QuantJob q{static_cast<const __nv_bfloat16*>(dy), g, static_cast<int64_t>(M) * N, scale_dy, amax_dy, recipe};
  MMDIT_CUDA(launch_quantize_e4m3(&q, 1, st), "gradient cast");
  const int kind = recipe ? 3 : 2;
  {
    // dx [M, K] = G W_q / (s_dy s_w): K-major operands G [M, N] and W_q^T [K, N]
    MMDIT_CUDA(launch_transpose_u8(static_cast<const uint8_t*>(w_q), N, K, N, at<uint8_t>(workspace, fp.wt), st),
               "W codes transpose");
    GemmProblem gp;
    gp.act = kind, gp.epi = kEpiBias, gp.M = M, gp.N = K, gp.K = N, gp.A = g, gp.W = at(workspace, fp.wt);
    gp.ep.out = dx, gp.ep.scale_a = scale_dy, gp.ep.scale_w = scale_w;
    MMDIT_CUDA(launch_gemm(gp, status_word(workspace), st), "FP8 dgrad GEMM");
  }
  if (dw && fp8_wgrad) {
    // dW [N, K] = G^T X_q / (s_dy s_x), contracted over the M rows (zero-padded to Mp)
    MMDIT_CUDA(launch_transpose_u8(g, M, N, fp.Mp, at<uint8_t>(workspace, fp.gt), st), "G transpose");
    MMDIT_CUDA(launch_transpose_u8(static_cast<const uint8_t*>(x_q), M, K, fp.Mp, at<uint8_t>(workspace, fp.xt), st),
               "x codes transpose");
    GemmProblem gp;
    gp.act = kind, gp.epi = kEpiBias, gp.M = N, gp.N = K, gp.K = fp.Mp, gp.A = at(workspace, fp.gt);
    gp.W = at(workspace, fp.xt), gp.ep.out = dw, gp.ep.out_f32 = 1, gp.ep.scale_a = scale_dy, gp.ep.scale_w = scale_x;
    MMDIT_CUDA(launch_gemm(gp, status_word(workspace), st), "FP8 wgrad GEMM");
  } else if (dw) {
    // without fp8_wgrad the weight gradient is dy^T x on the unquantised bf16 tensors
    mmdit_status r = linear_bwd_body(MMDIT_BF16, M, N, K, dy, x, nullptr, nullptr, dw, nullptr,
                                     at(workspace, fp.lin), workspace, st);
    if (r != MMDIT_OK) return r;
  }
  if (db) MMDIT_CUDA(launch_colsum(MMDIT_BF16, dy, M, N, at<float>(workspace, fp.part), kColsumChunks, db, st),
                     "db column sums");
  return MMDIT_OK;
}

size_t mmdit_fp8_attention_workspace_size(int32_t batch, int32_t heads, int32_t seq) {
  if (batch < 1 || heads < 1 || seq < 1) return kStatusBytes;
  const size_t bh = static_cast<size_t>(batch) * heads, sp = round_up(static_cast<size_t>(seq), 16);
  Carver c;
  c.take(bh * seq * 128);  // q8
  c.take(bh * seq * 128);  // k8
  c.take(bh * 128 * sp);   // vt8
  c.take(2 * sizeof(float));
  return c.off;
}

mmdit_status mmdit_fp8_attention_fwd(int32_t act, int32_t batch, int32_t heads, int32_t seq, int32_t head_dim,
                                     const void* q, const void* k, const void* v, const float* scale_q,
                                     const float* scale_k, const float* scale_v, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 1 || heads < 1 || seq < 0) return fail(MMDIT_ERR_INVALID_ARG, "FP8 attention: bad shape");
  if (head_dim != 128) return fail(MMDIT_ERR_UNSUPPORTED, "FP8 attention: head_dim must be 128");
  if (static_cast<int64_t>(batch) * heads > 65535)
    return fail(MMDIT_ERR_UNSUPPORTED, "FP8 attention: batch * heads must be <= 65535");
  mmdit_status s = check_ptrs({q, k, v, out}, "FP8 attention");
  if (s != MMDIT_OK) return s;
  if (!scale_q || !scale_k || !scale_v) return fail(MMDIT_ERR_INVALID_ARG, "FP8 attention: NULL scale");
  if ((s = check_workspace(workspace, workspace_bytes, mmdit_fp8_attention_workspace_size(batch, heads, seq))) !=
      MMDIT_OK)
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  if (seq == 0) return MMDIT_OK;
  pdl_begin_call();
  const size_t bh = static_cast<size_t>(batch) * heads;
  Carver c;
  AttnFp8Problem a;
  a.act = act, a.batch = batch, a.heads = heads, a.seq = seq, a.seq_pad = static_cast<int>(round_up(seq, 16));
  a.split = seq;
  a.q = static_cast<const __nv_bfloat16*>(q), a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q8 = at<uint8_t>(workspace, c.take(bh * seq * 128));
  a.k8 = at<uint8_t>(workspace, c.take(bh * seq * 128));
  a.vt8 = at<uint8_t>(workspace, c.take(bh * 128 * a.seq_pad));
  a.amax = at<float>(workspace, c.take(2 * sizeof(float)));
  a.scale_q = scale_q, a.scale_k = scale_k, a.scale_v = scale_v;
  a.out0 = out;
  ProfScope ps_("fp8_attention", st);
  MMDIT_CUDA(launch_attention_fp8(a, status_word(workspace), st), "FP8 joint attention");
  return MMDIT_OK;
}

size_t mmdit_double_block_bwd_workspace_size(const mmdit_dims* d) {
  BwdPlan p;
  if (check_dims(d) != MMDIT_OK || !plan_block_bwd(d, false, &p)) return 0;
  return p.total;
}

size_t mmdit_single_block_bwd_workspace_size(const mmdit_dims* d) {
  BwdPlan p;
  if (check_dims(d) != MMDIT_OK || !plan_block_bwd(d, true, &p)) return 0;
  return p.total;
}

namespace {

// The checks and set-up every double-block backward call shares; `dy`, `dx` may be NULL for the
// forward half of the training pair.
mmdit_status double_bwd_call(const mmdit_dims* d, const mmdit_stream_w* w_img, const mmdit_stream_w* w_txt,
                             const void* vec, const float* rope_cos, const float* rope_sin, const void* x_img,
                             const void* x_txt, const void* dy_img, const void* dy_txt, void* dx_img, void* dx_txt,
                             float* dvec, const mmdit_stream_grads* g_img, const mmdit_stream_grads* g_txt,
                             void* y_img, void* y_txt, void* workspace, size_t workspace_bytes, void* stream,
                             int phases, const char* what) {
  mmdit_status s = check_block_bwd(d, false);
  if (s != MMDIT_OK) return s;
  if ((s = check_stream_w(w_img, "image weights")) != MMDIT_OK || (s = check_stream_w(w_txt, "text weights")) != MMDIT_OK)
    return s;
  if ((s = check_ptrs({vec, rope_cos, rope_sin, x_img, x_txt}, what)) != MMDIT_OK) return s;
  if ((phases & kBwdGradients) && (s = check_ptrs({dy_img, dy_txt, dx_img, dx_txt}, what)) != MMDIT_OK) return s;
  if (!(phases & kBwdGradients) && (s = check_ptrs({y_img, y_txt}, what)) != MMDIT_OK) return s;
  if (dvec && !aligned16(dvec)) return fail(MMDIT_ERR_INVALID_ARG, "dvec is not 16-byte aligned");
  if ((s = check_grads(g_img, "image gradients")) != MMDIT_OK || (s = check_grads(g_txt, "text gradients")) != MMDIT_OK)
    return s;
  BwdPlan p;
  plan_block_bwd(d, false, &p);
  if ((s = check_workspace(workspace, workspace_bytes, p.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  // the forward's modulation is recomputed from the weights (a precomputed `mod` is not used)
  mmdit_stream_w wi = *w_img, wt = *w_txt;
  wi.mod = nullptr, wt.mod = nullptr;
  const mmdit_stream_w* W[2] = {&wi, &wt};
  const void* X[2] = {x_img, x_txt};
  const void* DY[2] = {dy_img, dy_txt};
  void* DX[2] = {dx_img, dx_txt};
  void* Y[2] = {y_img, y_txt};
  const mmdit_stream_grads* G[2] = {g_img, g_txt};
  return block_bwd_body(d, p, 2, W, vec, rope_cos, rope_sin, X, DY, DX, dvec, G, workspace, st, phases,
                        (phases & kBwdGradients) ? nullptr : Y);
}

mmdit_status single_bwd_call(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec, const float* rope_cos,
                             const float* rope_sin, const void* x, const void* dy, void* dx, float* dvec,
                             const mmdit_stream_grads* g, void* y, void* workspace, size_t workspace_bytes,
                             void* stream, int phases, const char* what) {
  mmdit_status s = check_block_bwd(d, true);
  if (s != MMDIT_OK) return s;
  if ((s = check_stream_w(w, "single block weights")) != MMDIT_OK) return s;
  if ((s = check_ptrs({vec, rope_cos, rope_sin, x}, what)) != MMDIT_OK) return s;
  if ((phases & kBwdGradients) && (s = check_ptrs({dy, dx}, what)) != MMDIT_OK) return s;
  if (!(phases & kBwdGradients) && (s = check_ptrs({y}, what)) != MMDIT_OK) return s;
  if (dvec && !aligned16(dvec)) return fail(MMDIT_ERR_INVALID_ARG, "dvec is not 16-byte aligned");
  if ((s = check_grads(g, "single block gradients")) != MMDIT_OK) return s;
  BwdPlan p;
  plan_block_bwd(d, true, &p);
  if ((s = check_workspace(workspace, workspace_bytes, p.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  mmdit_stream_w w1 = *w;
  w1.mod = nullptr;
  const mmdit_stream_w* W[1] = {&w1};
  const void* X[1] = {x};
  const void* DY[1] = {dy};
  void* DX[1] = {dx};
  void* Y[1] = {y};
  const mmdit_stream_grads* G[1] = {g};
  return block_bwd_body(d, p, 1, W, vec, rope_cos, rope_sin, X, DY, DX, dvec, G, workspace, st, phases,
                        (phases & kBwdGradients) ? nullptr : Y);
}

}  // namespace

mmdit_status mmdit_double_block_bwd(const mmdit_dims* d, const mmdit_stream_w* w_img, const mmdit_stream_w* w_txt,
                                    const void* vec, const float* rope_cos, const float* rope_sin, const void* x_img,
                                    const void* x_txt, const void* dy_img, const void* dy_txt, void* dx_img,
                                    void* dx_txt, float* dvec, const mmdit_stream_grads* g_img,
                                    const mmdit_stream_grads* g_txt, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return double_bwd_call(d, w_img, w_txt, vec, rope_cos, rope_sin, x_img, x_txt, dy_img, dy_txt, dx_img, dx_txt,
                         dvec, g_img, g_txt, nullptr, nullptr, workspace, workspace_bytes, stream,
                         kBwdForward | kBwdGradients, "double block backward");
}

mmdit_status mmdit_double_block_fwd_train(const mmdit_dims* d, const mmdit_stream_w* w_img,
                                          const mmdit_stream_w* w_txt, const void* vec, const float* rope_cos,
                                          const float* rope_sin, const void* x_img, const void* x_txt, void* y_img,
                                          void* y_txt, void* saved, size_t saved_bytes, void* stream) {
  return double_bwd_call(d, w_img, w_txt, vec, rope_cos, rope_sin, x_img, x_txt, nullptr, nullptr, nullptr, nullptr,
                         nullptr, nullptr, nullptr, y_img, y_txt, saved, saved_bytes, stream, kBwdForward,
                         "double block training forward");
}

mmdit_status mmdit_double_block_bwd_saved(const mmdit_dims* d, const mmdit_stream_w* w_img,
                                          const mmdit_stream_w* w_txt, const void* vec, const float* rope_cos,
                                          const float* rope_sin, const void* x_img, const void* x_txt,
                                          const void* dy_img, const void* dy_txt, void* dx_img, void* dx_txt,
                                          float* dvec, const mmdit_stream_grads* g_img,
                                          const mmdit_stream_grads* g_txt, void* saved, size_t saved_bytes,
                                          void* stream) {
  return double_bwd_call(d, w_img, w_txt, vec, rope_cos, rope_sin, x_img, x_txt, dy_img, dy_txt, dx_img, dx_txt,
                         dvec, g_img, g_txt, nullptr, nullptr, saved, saved_bytes, stream, kBwdGradients,
                         "double block backward (saved forward)");
}

mmdit_status mmdit_single_block_bwd(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec,
                                    const float* rope_cos, const float* rope_sin, const void* x, const void* dy,
                                    void* dx, float* dvec, const mmdit_stream_grads* g, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return single_bwd_call(d, w, vec, rope_cos, rope_sin, x, dy, dx, dvec, g, nullptr, workspace, workspace_bytes,
                         stream, kBwdForward | kBwdGradients, "single block backward");
}

mmdit_status mmdit_single_block_fwd_train(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec,
                                          const float* rope_cos, const float* rope_sin, const void* x, void* y,
                                          void* saved, size_t saved_bytes, void* stream) {
  return single_bwd_call(d, w, vec, rope_cos, rope_sin, x, nullptr, nullptr, nullptr, nullptr, y, saved, saved_bytes,
                         stream, kBwdForward, "single block training forward");
}

mmdit_status mmdit_single_block_bwd_saved(const mmdit_dims* d, const mmdit_stream_w* w, const void* vec,
                                          const float* rope_cos, const float* rope_sin, const void* x, const void* dy,
                                          void* dx, float* dvec, const mmdit_stream_grads* g, void* saved,
                                          size_t saved_bytes, void* stream) {
  return single_bwd_call(d, w, vec, rope_cos, rope_sin, x, dy, dx, dvec, g, nullptr, saved, saved_bytes, stream,
                         kBwdGradients, "single block backward (saved forward)");
}

mmdit_status mmdit_modulation_batched_fwd(int32_t act, int32_t batch, int32_t dim, const void* vec,
                                          int32_t n_jobs, const mmdit_gemv_job* jobs, void* stream) {
  if (act != MMDIT_F32 && act != MMDIT_BF16) return fail(MMDIT_ERR_INVALID_ARG, "bad act %d", act);
  if (batch < 0 || dim < 1 || n_jobs < 0) return fail(MMDIT_ERR_INVALID_ARG, "bad batched modulation shape");
  if (dim % 8 != 0 || dim > 6144)
    return fail(MMDIT_ERR_UNSUPPORTED, "modulation: dim must be a multiple of 8, at most 6144 (got %d)", dim);
  if (n_jobs > 0 && !jobs) return fail(MMDIT_ERR_INVALID_ARG, "jobs is NULL");
  if (batch == 0 || n_jobs == 0) return MMDIT_OK;
  mmdit_status s = check_ptrs({vec}, "batched modulation input");
  if (s != MMDIT_OK) return s;
  std::vector<ModulationJob> mj(static_cast<size_t>(n_jobs));
  for (int i = 0; i < n_jobs; ++i) {
    if (jobs[i].rows < 0) return fail(MMDIT_ERR_INVALID_ARG, "job %d: negative rows", i);
    if (jobs[i].rows > 0 && (s = check_ptrs({jobs[i].w, jobs[i].out}, "batched modulation job")) != MMDIT_OK)
      return s;
    mj[i] = {jobs[i].w, jobs[i].b, jobs[i].out, jobs[i].rows};
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pdl_begin_call();
  ProfScope ps_("modulation.batched", st);
  MMDIT_CUDA(launch_gemv(act, vec, mj.data(), n_jobs, batch, dim, 1, kGemvOutF32, st), "batched modulation");
  return MMDIT_OK;
}

size_t mmdit_flux_workspace_size(const mmdit_flux_config* cfg) {
  FluxPlan f;
  if (check_flux(cfg) != MMDIT_OK || !plan_flux(cfg, &f)) return 0;
  return f.total;
}

mmdit_status mmdit_flux_forward(const mmdit_flux_config* cfg, const mmdit_flux_w* w, const float* z_t,
                                const void* txt, const float* t, const void* y, const float* guidance,
                                const float* rope_cos, const float* rope_sin, float* pred, void* workspace,
                                size_t workspace_bytes, void* stream) {
  mmdit_status s = check_flux(cfg);
  if (s != MMDIT_OK) return s;
  if (!w) return fail(MMDIT_ERR_INVALID_ARG, "model weights are NULL");
  const mmdit_dims* d = &cfg->block;
  const int B = d->batch, D = d->hidden, Si = d->seq_img, St = d->seq_txt, S = Si + St;
  if ((s = check_cond_w(&w->cond, guidance != nullptr)) != MMDIT_OK) return s;
  if ((s = check_ptrs({z_t, t, y, rope_cos, rope_sin, pred}, "whole-model inputs")) != MMDIT_OK) return s;
  if ((s = check_ptrs({w->w_img_in, w->b_img_in, w->w_ada, w->b_ada, w->w_out, w->b_out},
                      "embedding and head weights")) != MMDIT_OK)
    return s;
  if (St > 0 && (s = check_ptrs({txt, w->w_txt_in, w->b_txt_in}, "text input")) != MMDIT_OK) return s;
  if (cfg->n_double > 0 && (!w->double_img || !w->double_txt))
    return fail(MMDIT_ERR_INVALID_ARG, "double-block weight arrays are NULL");
  if (cfg->n_single > 0 && !w->single) return fail(MMDIT_ERR_INVALID_ARG, "single-block weight array is NULL");
  for (int i = 0; i < cfg->n_double; ++i) {
    if ((s = check_stream_w(&w->double_img[i], "double block image weights")) != MMDIT_OK) return s;
    if ((s = check_stream_w(&w->double_txt[i], "double block text weights")) != MMDIT_OK) return s;
  }
  for (int i = 0; i < cfg->n_single; ++i)
    if ((s = check_stream_w(&w->single[i], "single block weights")) != MMDIT_OK) return s;
  FluxPlan f;
  if (!plan_flux(cfg, &f)) return fail(MMDIT_ERR_INVALID_ARG, "bad whole-model dims");
  if ((s = check_workspace(workspace, workspace_bytes, f.total)) != MMDIT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elt_bytes(d->act);
  void* vec = at(workspace, f.vec);
  float* mods = at<float>(workspace, f.mods);
  void* x_img = at(workspace, f.x_img);
  void* x_txt = at(workspace, f.x_txt);
  void* c = at(workspace, f.c);
  MMDIT_CUDA(cudaMemsetAsync(workspace, 0, 4, st), "status clear");
  pdl_begin_call();
  if ((s = conditioning_body(d->act, B, D, cfg->time_dim, cfg->vec_in_dim, &w->cond, t, y, guidance, vec,
                             workspace, st)) != MMDIT_OK)
    return s;
  // every block's modulation in one launch: they all read vec
  std::vector<mmdit_stream_w> wd(2 * static_cast<size_t>(cfg->n_double)), ws1(static_cast<size_t>(cfg->n_single));
  std::vector<ModulationJob> jobs;
  jobs.reserve(static_cast<size_t>(f.n_mod));
  const size_t mod_stride = static_cast<size_t>(B) * 6 * D;
  for (int i = 0; i < cfg->n_double; ++i)
    for (int k = 0; k < 2; ++k) {
      mmdit_stream_w& sw = wd[2 * i + k];
      sw = k ? w->double_txt[i] : w->double_img[i];
      float* m = mods + (2 * static_cast<size_t>(i) + k) * mod_stride;
      sw.mod = m;
      jobs.push_back({sw.w_mod, sw.b_mod, m, 6 * D});
    }
  for (int i = 0; i < cfg->n_single; ++i) {
    ws1[i] = w->single[i];
    float* m = mods + (2 * static_cast<size_t>(cfg->n_double) + i) * mod_stride;
    ws1[i].mod = m;
    jobs.push_back({ws1[i].w_mod, ws1[i].b_mod, m, (cfg->single_parallel ? 3 : 6) * D});
  }
  if (!jobs.empty()) {
    ProfScope ps_("modulation.batched", st);
    MMDIT_CUDA(launch_gemv(d->act, vec, jobs.data(), static_cast<int>(jobs.size()), B, D, 1, kGemvOutF32, st),
               "every block's modulation");
  }
  if ((s = img_in_body(d->act, B, cfg->channels, cfg->lat_h, cfg->lat_w, D, z_t, w->w_img_in, w->b_img_in,
                       x_img, workspace, st)) != MMDIT_OK)
    return s;
  if (St > 0 && (s = linear_body(d->act, B * St, D, cfg->txt_dim, txt, w->w_txt_in, w->b_txt_in, x_txt,
                                 workspace, st)) != MMDIT_OK)
    return s;
  for (int i = 0; i < cfg->n_double; ++i)
    if ((s = double_block_body(d, f.dbl, &wd[2 * i], &wd[2 * i + 1], vec, rope_cos, rope_sin, x_img, x_txt,
                               x_img, x_txt, nullptr, workspace, st)) != MMDIT_OK)
      return s;
  const void* img_rows = x_img;
  if (cfg->n_single > 0) {
    if (B > 1) {
      // [img; txt] per sample (strided copies), then the next kernel launches normally
      MMDIT_CUDA(cudaMemcpy2DAsync(c, S * D * e, x_img, Si * D * e, Si * D * e, B, cudaMemcpyDeviceToDevice, st),
                 "join image rows");
      if (St > 0)
        MMDIT_CUDA(cudaMemcpy2DAsync(static_cast<uint8_t*>(c) + Si * D * e, S * D * e, x_txt, St * D * e,
                                     St * D * e, B, cudaMemcpyDeviceToDevice, st),
                   "join text rows");
      pdl_begin_call();
    }
    for (int i = 0; i < cfg->n_single; ++i)
      if ((s = single_block_body(d, f.sgl, &ws1[i], vec, rope_cos, rope_sin, c, c, nullptr, workspace, st)) !=
          MMDIT_OK)
        return s;
    if (B > 1) {
      MMDIT_CUDA(cudaMemcpy2DAsync(x_img, Si * D * e, c, S * D * e, Si * D * e, B, cudaMemcpyDeviceToDevice, st),
                 "image rows of the last block");
      pdl_begin_call();
    } else {
      img_rows = c;
    }
  }
  return final_layer_body(d, cfg->channels, img_rows, vec, w->w_ada, w->b_ada, w->w_out, w->b_out, pred,
                          workspace, st);
}

}  // extern "C"
