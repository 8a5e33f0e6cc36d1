// Host-side launch of the persistent verification kernel.
#pragma once

#include <atomic>

#include "sv_kernel.cuh"

namespace sv {

constexpr int kMaxDevices = 64;

// Launches one instantiation with the call's schedule.  The grid is one
// wave of resident CTAs (SM count x occupancy), capped by the unit count;
// CTAs pull units from the workspace counter.
template <int MODE, int TDT, int DDT, bool PROBS, int PHASES>
sv_status launch_phase(const KParams &P0, const Sched &s, cudaStream_t stream) {
  if (s.total <= 0) return SV_OK;
  auto kern = sv_verify_kernel<MODE, TDT, DDT, PROBS, PHASES>;
  static std::atomic<int> occ_cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  int occ = occ_cache[dev].load(std::memory_order_relaxed);
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, 0) != cudaSuccess ||
        occ <= 0)
      return SV_ERR_CUDA;
    occ_cache[dev].store(occ, std::memory_order_relaxed);
  }
  const int sms = sm_count(dev);
  if (sms <= 0) return SV_ERR_CUDA;
  const long long cap = (long long)sms * occ;
  KParams P = P0;
  P.sched = s;
  const int grid = (int)(s.total < cap ? s.total : cap);
  kern<<<grid, kThreads, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_verify(const KParams &P, cudaStream_t stream) {
  const int B = P.B, A = P.rows * P.tiles;
  if (cudaMemsetAsync(P.hdr, 0, P.ctrl_bytes, stream) != cudaSuccess) return SV_ERR_CUDA;
  if constexpr (MODE == MODE_CHAIN) {
    // Phase A (+ decisions), then Phase B (+ finalisation) in stream order.
    const int Bc = P.tiles;
    const sv_status st =
        launch_phase<MODE, TDT, DDT, PROBS, 1>(P, Sched{B, A, 0, B, B * A}, stream);
    if (st != SV_OK) return st;
    return launch_phase<MODE, TDT, DDT, PROBS, 2>(P, Sched{B, 0, Bc, 0, B * Bc}, stream);
  }
  return launch_phase<MODE, TDT, DDT, PROBS, 1>(P, Sched{B, A, 0, B, B * A}, stream);
}

template <int TDT>
sv_status launch_chain_t(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream) {
  if (probs) return launch_verify<MODE_CHAIN, TDT, SV_F32, true>(P, stream);
  switch (ddt) {
    case SV_F32: return launch_verify<MODE_CHAIN, TDT, SV_F32, false>(P, stream);
    case SV_BF16: return launch_verify<MODE_CHAIN, TDT, SV_BF16, false>(P, stream);
    case SV_F16: return launch_verify<MODE_CHAIN, TDT, SV_F16, false>(P, stream);
  }
  return SV_ERR_UNSUPPORTED;
}

}  // namespace sv
