// Host-side launch of the persistent verification kernel.
#pragma once

#include <atomic>

#include "sv_stream.cuh"

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

// Streaming kernel: one persistent CTA per SM.
template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_stream(const KParams &P0, cudaStream_t stream) {
  auto kern = sv_stream_kernel<MODE, TDT, DDT, PROBS>;
  static std::atomic<int> attr_done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  if (!attr_done[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStreamSmemBytes) != cudaSuccess)
      return SV_ERR_CUDA;
    attr_done[dev].store(1, std::memory_order_relaxed);
  }
  const int sms = sm_count(dev);
  if (sms <= 0) return SV_ERR_CUDA;
  const int esT = (TDT == SV_F32) ? 4 : 2, esD = (DDT == SV_F32) ? 4 : 2;
  const StreamLayout L = make_stream_layout(P0.B, P0.rows, P0.V, esT, esD, PROBS);
  char *w = reinterpret_cast<char *>(P0.hdr);
  SParams S{};
  S.target = P0.target;
  S.draft = P0.draft;
  S.draft_tokens = P0.draft_tokens;
  S.temps = P0.temps;
  S.unif = P0.unif;
  S.parent = P0.parent;
  S.node_tokens = P0.node_tokens;
  S.B = P0.B;
  S.gamma = P0.gamma;
  S.V = P0.V;
  S.N = P0.N;
  S.max_depth = P0.max_depth;
  S.rows = P0.rows;
  S.tilesT = L.tilesT;
  S.tilesD = L.tilesD;
  S.tilesMax = L.tilesMax;
  S.tilesB = L.tilesB;
  S.TA_T = L.TA_T;
  S.TA_D = L.TA_D;
  S.TB = L.TB;
  if (MODE == MODE_CHAIN) {
    const int G1 = P0.gamma + 1;
    S.unitsA = G1 * L.tilesT + (PROBS ? 0 : P0.gamma * L.tilesD);
  } else {
    S.unitsA = P0.rows * L.tilesT;
  }
  S.totalA = P0.B * S.unitsA;
  S.out_tokens = P0.out_tokens;
  S.out_nacc = P0.out_nacc;
  S.out_status = P0.out_status;
  S.out_path = P0.out_path;
  S.out_diag = P0.out_diag;
  S.hdr = reinterpret_cast<StreamHeader *>(w);
  S.a_count = reinterpret_cast<unsigned *>(w + L.a_count);
  S.b_count = reinterpret_cast<unsigned *>(w + L.b_count);
  S.row_done = reinterpret_cast<unsigned *>(w + L.row_done);
  S.qitems = reinterpret_cast<unsigned *>(w + L.qitems);
  S.dec = reinterpret_cast<Decision *>(w + L.dec);
  S.partA = reinterpret_cast<float2 *>(w + L.partA);
  S.partB = reinterpret_cast<float *>(w + L.partB);
  S.partT = reinterpret_cast<float2 *>(w + L.partT);
  S.partBT = reinterpret_cast<float *>(w + L.partBT);
  if (cudaMemsetAsync(w, 0, L.ctrl, stream) != cudaSuccess) return SV_ERR_CUDA;
  kern<<<sms, kStreamThreads, kStreamSmemBytes, stream>>>(S);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Rows of both logit arrays start on 16-byte boundaries.
inline bool rows_aligned(const void *p, int V, int es) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0 && ((size_t)V * es) % 16 == 0;
}

template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_verify(const KParams &P, cudaStream_t stream) {
  {
    const int esT = (TDT == SV_F32) ? 4 : 2, esD = (DDT == SV_F32) ? 4 : 2;
    bool ok = rows_aligned(P.target, P.V, esT);
    if (MODE == MODE_CHAIN) ok = ok && rows_aligned(P.draft, P.V, esD);
    // Phase-B queue items pack b * tilesB + t in 27 bits
    if (MODE == MODE_CHAIN) ok = ok && (long long)P.B * ((P.V + 4095) / 4096) < (1LL << 26);
    if (ok && P.use_stream) return launch_stream<MODE, TDT, DDT, PROBS>(P, stream);
  }
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
