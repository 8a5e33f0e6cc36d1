// spec_verify_chain_no_alloc: chain verification whose scratch memory is a
// fixed array compiled into the library, for callers that cannot allocate
// device memory themselves.
//
// The array below lives in the library's device image: every GPU that loads
// the library holds SV_NO_ALLOC_SCRATCH_BYTES of it until the process exits.
// Host code never dereferences `g_no_alloc_scratch`: on the host its name is
// only a stand-in for the symbol, so the device address is looked up once
// per device with cudaGetSymbolAddress (with that device current) and that
// address is what the kernels receive.
#include <atomic>
#include <mutex>

#include "sv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[SV_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::atomic<void *> g_scratch_addr[kMaxDev];
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device, looked up on
// the first call made with that device current; nullptr on failure.  The
// address belongs to the device's primary context as it was at that first
// call: it is not looked up again after cudaDeviceReset, nor for a context
// the caller made current through the driver API.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  p = g_scratch_addr[dev].load(std::memory_order_relaxed);
  if (p) return p;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_no_alloc_scratch) != cudaSuccess || addr == nullptr) {
    (void)cudaGetLastError();  // leave no sticky error behind for the caller
    return nullptr;
  }
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace

extern "C" {

SV_API sv_status spec_verify_chain_no_alloc(const void *target_logits, sv_dtype tdt,
                                            const void *draft, sv_dtype ddt, int draft_is_probs,
                                            const int32_t *draft_tokens,
                                            const float *temperatures, const float *uniforms,
                                            int B, int gamma, int V, int32_t *out_tokens,
                                            int32_t *out_num_accepted, float *out_diag,
                                            int32_t *out_row_status, sv_stream_t stream) {
  if (B < 1 || gamma < 1 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
    return SV_ERR_INVALID_ARG;
  const int rows = (gamma + 1) + (draft_is_probs ? 0 : gamma);
  const size_t need = spec_verify_workspace_bytes(B, rows, V, tdt);
  if (need == 0) return SV_ERR_INVALID_ARG;
  if (need > (size_t)SV_NO_ALLOC_SCRATCH_BYTES) return SV_ERR_UNSUPPORTED;
  void *scratch = scratch_on_current_device();
  if (scratch == nullptr) return SV_ERR_CUDA;
  // The array starts zeroed (a static device array) and only these calls
  // write it.  Each call leaves its 4 KB state header valid for the next
  // one, whatever the shapes, so the regular entry point can run on it
  // without further initialisation.
  return spec_verify_chain(target_logits, tdt, draft, ddt, draft_is_probs, draft_tokens,
                           temperatures, uniforms, B, gamma, V, out_tokens, out_num_accepted,
                           out_diag, out_row_status, scratch,
                           (size_t)SV_NO_ALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
