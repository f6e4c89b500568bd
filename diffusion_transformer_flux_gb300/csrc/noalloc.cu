// noalloc.cu -- flow_match_noise_and_loss_noalloc: the rectified-flow noise and loss for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: real-time or embedded hosts
// whose memory budget is fixed at start-up, and plug-ins living inside another framework's
// process that must not touch its allocator.  flow_match_noise_and_loss needs a caller-provided
// workspace for the per-block partial sums of the loss; this variant keeps them instead in the
// file-scope device array below, so the caller passes only inputs and outputs.
//
// The array holds kNoAllocPartials floats (1 KiB) on every GPU that loads the library, until the
// process exits.  One partial sum covers kFlowElemsPerPartial = 8192 elements (the loss kernel's
// per-block share, which the workspace entry point uses too, so both reduce in the same order),
// and a call handles at most kNoAllocPartials * 8192 = 2,097,152 elements (batch *
// n_per_sample); larger calls are rejected with MMDIT_ERR_UNSUPPORTED before anything is
// launched.
//
// Every call on a device shares the array and leaves its last contents there.  Each call
// rewrites all the partial sums it reads before reading them, so nothing has to start at zero,
// but two calls whose kernels overlap on the GPU (different streams, no ordering between them)
// race on the array.  Order such calls on one stream or with events.
//
// The array's name is a host-side stand-in in host code, not a device address.  The first
// call on each device, with that device current, looks the address up with
// cudaGetSymbolAddress; that lookup is a CUDA API call, so the first call on a device should
// come before any stream capture.  The address is kept for the life of the process: a
// cudaDeviceReset of a device invalidates it, and this entry point must not be called on that
// device after such a reset.
#include <mutex>

#include "../../include/mmdit.h"
#include "internal.h"

namespace mmdit {
namespace {

constexpr int kNoAllocPartials = 256;
constexpr int64_t kNoAllocMaxElems = kNoAllocPartials * kFlowElemsPerPartial;  // 2,097,152
static_assert(kNoAllocPartials <= kFlowMaxPartials, "one partial per block, with no grid-stride wrap");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::mutex g_noalloc_mutex;
float* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_partials on the current device (looked up once per device).
cudaError_t noalloc_partials(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mmdit

extern "C" mmdit_status flow_match_noise_and_loss_noalloc(int32_t dtype, const void* z0,
                                                          const void* z1, const float* t,
                                                          int32_t batch, int64_t n_per_sample,
                                                          void* z_t, const void* pred, float* loss,
                                                          void* stream) {
  using namespace mmdit;
  auto err = [](mmdit_status s, const char* m) {
    return static_cast<mmdit_status>(set_last_error(s, m));
  };
  if (dtype != MMDIT_F32 && dtype != MMDIT_BF16)
    return err(MMDIT_ERR_INVALID_ARG, "flow_match_noise_and_loss_noalloc: dtype must be MMDIT_F32 or MMDIT_BF16");
  if (batch < 0 || n_per_sample < 0)
    return err(MMDIT_ERR_INVALID_ARG, "flow_match_noise_and_loss_noalloc: negative size");
  if (n_per_sample % 8 != 0)
    return err(MMDIT_ERR_UNSUPPORTED, "flow_match_noise_and_loss_noalloc: n_per_sample must be a multiple of 8");
  // compared before multiplying, so that no product can overflow
  if (batch > 0 && n_per_sample > kNoAllocMaxElems / batch)
    return err(MMDIT_ERR_UNSUPPORTED,
               "flow_match_noise_and_loss_noalloc: batch * n_per_sample exceeds the 2,097,152 "
               "elements its fixed 256-entry device scratch covers; use flow_match_noise_and_loss "
               "with a workspace");
  if ((pred == nullptr) != (loss == nullptr))
    return err(MMDIT_ERR_INVALID_ARG, "flow_match_noise_and_loss_noalloc: pred and loss go together");
  if (!z0 || !z1 || !al16(z0) || !al16(z1) || (z_t && (!t || !al16(z_t))) ||
      (pred && (!al16(pred) || !al16(loss))))
    return err(MMDIT_ERR_INVALID_ARG, "flow_match_noise_and_loss_noalloc: NULL or misaligned pointer");
  if (pred && z_t && (z_t == z0 || z_t == z1))
    return err(MMDIT_ERR_INVALID_ARG, "flow_match_noise_and_loss_noalloc: z_t may not alias z0/z1 with the loss");
  const int64_t n_total = static_cast<int64_t>(batch) * n_per_sample;
  if (n_total == 0) return MMDIT_OK;
  // the same count (and so the same grid and reduction order) as the workspace entry point
  const int n_partials = flow_partial_blocks(n_total);
  if (n_partials > kNoAllocPartials)
    return err(MMDIT_ERR_UNSUPPORTED, "flow_match_noise_and_loss_noalloc: partial-sum count exceeds the scratch");
  float* partials = nullptr;
  cudaError_t e = noalloc_partials(&partials);
  if (e != cudaSuccess) return err(MMDIT_ERR_CUDA, cudaGetErrorString(e));
  pdl_begin_call();  // the first kernel waits for everything enqueued before the call
  e = launch_flow_match(dtype, z0, z1, t, batch, n_per_sample, z_t, pred, loss, partials,
                        n_partials, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return err(MMDIT_ERR_CUDA, cudaGetErrorString(e));
  return MMDIT_OK;
}
