// Diagnostics: the library's bounded device-side waits, run on a flag that
// nothing sets, so that a caller (the test-suite) can check that each wait
// gives up after its bound and reports a status instead of hanging, and that
// the context stays usable afterwards.
#include "sv_launch.cuh"

namespace sv {

// scratch: 8 zeroed 64-bit words.  [0] the counter-reset "ready" word,
// [1] the call's error word, [2..5] two chunk partials that carry no call's
// tag.  None is ever set here.
__global__ void sv_wait_selftest_kernel(int which, unsigned long long *scratch,
                                        int32_t *out_status) {
  if (threadIdx.x >= 32) return;
  if (which == 0) {
    PassParams P{};
    P.claim_ready = scratch;  // stays 0, never this call's epoch
    P.claim_err = scratch + 1;
    const unsigned long long E = 1;
    const bool ok = counters_reset_wait(P, E);
    if (lane_id() == 0) {
      const bool flagged = __ldcg(scratch + 1) == E;
      *out_status = ok ? SV_ROW_OK : (flagged ? SV_ROW_TIMEOUT : SV_ROW_NONFINITE);
    }
  } else {
    // the decide kernel's poll of a row's partials, on partials that never
    // carry the awaited tag: it gives up after kPollSpins rounds (the decide
    // kernel then takes the dependency wait)
    float2 za, zb;
    const bool ok = warp_rows_softmax2_poll(reinterpret_cast<const Part *>(scratch + 2), 2,
                                            nullptr, 0, 1.f, 1u, kPollSpins, za, zb);
    if (lane_id() == 0) *out_status = ok ? SV_ROW_OK : SV_ROW_TIMEOUT;
  }
}

}  // namespace sv

extern "C" {

SV_API sv_status spec_verify_wait_selftest(int which, void *scratch, int32_t *out_status,
                                           sv_stream_t stream) {
  if (!scratch || !out_status || (which != 0 && which != 1)) return SV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scratch) & 15) || (reinterpret_cast<uintptr_t>(out_status) & 3))
    return SV_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 64, s) != cudaSuccess) return SV_ERR_CUDA;
  sv::sv_wait_selftest_kernel<<<1, 32, 0, s>>>(which,
                                              static_cast<unsigned long long *>(scratch),
                                              out_status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
