// Host-side launches of the two-launch path (the stats kernel, then the
// decide kernel as its programmatic dependent) for every entry point, dtype
// and row alignment.
#pragma once

#include <atomic>

#include "sv_cluster.cuh"

namespace sv {

constexpr int kMaxDevices = 64;
constexpr int kTreeCarveout = 42;  // percent of the largest shared-memory carveout

// Partials are polled (merged before the dependency wait) only by the first
// kPollCalls calls of the process: their tags, below, are then all
// distinct, so a partial left in a workspace by an earlier call never
// carries a polling call's tag.  Later calls take the dependency wait.
constexpr unsigned long long kPollCalls = 1ull << 31;

// The 32-bit tag of a call's partials: (2 id + 1) times an odd constant,
// modulo 2^32.  It is odd, so never the tag of a zeroed word, and distinct
// for ids below 2^31; the multiplication spreads consecutive ids over the
// whole range, so small integers left in recycled memory do not resemble
// early calls' tags.
inline unsigned partial_tag(unsigned long long call_id) {
  return (unsigned)((call_id << 1) | 1ull) * 0x9E3779B1u;
}

// Stats units (warp-chunks) of the two-launch path for this call; -1 if the
// count does not fit the kernels' 32-bit unit indices.
template <int MODE, int TDT, int DDT, bool PROBS>
long long pass_units(const KParams &P, const PassLayout &L) {
  long long total;
  if (MODE == MODE_TREE || MODE == MODE_DRAFT) total = (long long)P.B * P.N * L.cT;
  else total = (long long)P.B * L.cT + (long long)P.gamma * P.B * (L.cT + L.cD);
  return total < (1LL << 31) - 1 ? total : -1;
}

// Two-launch path: the stats kernel over every needed row, then the decide
// kernel as its programmatic dependent (its CTAs launch while the stats
// kernel drains and wait on the device for its completion).
template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
sv_status launch_pass_t(const KParams &P0, const PassLayout &L, long long total,
                        cudaStream_t stream) {
  constexpr bool unaligned = UNAL;
  auto stats = sv_stats_kernel<MODE, TDT, DDT, PROBS, UNAL>;
  auto decide = sv_decide_kernel<MODE, TDT, DDT, PROBS, UNAL>;
  static std::atomic<int> occ_cache[kMaxDevices], occd_cache[kMaxDevices], per_cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  int occ = occ_cache[dev].load(std::memory_order_relaxed);
  int occd = occd_cache[dev].load(std::memory_order_relaxed);
  int per = per_cache[dev].load(std::memory_order_relaxed);
  if (occ == 0 || occd == 0) {
    // Tree calls keep their decide CTAs resident beside the stats kernel
    // (below), which needs both kernels on one shared-memory carveout (an SM
    // holding CTAs of one configuration takes no CTA of another): about
    // 100 KB, room for two decide CTAs, leaving the L1 room for the stats
    // kernel's loads in flight.
    if (MODE == MODE_TREE &&
        (cudaFuncSetAttribute(stats, cudaFuncAttributePreferredSharedMemoryCarveout,
                              kTreeCarveout) != cudaSuccess ||
         cudaFuncSetAttribute(decide, cudaFuncAttributePreferredSharedMemoryCarveout,
                              kTreeCarveout) != cudaSuccess))
      return SV_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stats, kPassThreads, 0) != cudaSuccess ||
        occ <= 0 ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occd, decide, kPassThreads, 0) !=
            cudaSuccess ||
        occd <= 0)
      return SV_ERR_CUDA;
    // decide CTAs that fit the registers of one stats CTA (registers are
    // allocated per warp in steps of 8 per thread)
    cudaFuncAttributes fs, fd;
    if (cudaFuncGetAttributes(&fs, stats) != cudaSuccess ||
        cudaFuncGetAttributes(&fd, decide) != cudaSuccess)
      return SV_ERR_CUDA;
    const int regs_s = (fs.numRegs + 7) / 8 * 8, regs_d = (fd.numRegs + 7) / 8 * 8;
    per = regs_d > 0 ? regs_s / regs_d : 0;
    per_cache[dev].store(per, std::memory_order_relaxed);
    occ_cache[dev].store(occ, std::memory_order_relaxed);
    occd_cache[dev].store(occd, std::memory_order_relaxed);
  }
  const int sms = sm_count(dev);
  if (sms <= 0) return SV_ERR_CUDA;
  char *w = P0.ws;
  PassParams S{};
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
  S.cT = L.cT;
  S.cD = L.cD;
  S.cMax = L.cMax;
  S.cR = L.cR;
  S.unaligned = unaligned ? 1 : 0;
  int H = 1;
  if (MODE == MODE_CHAIN) {
    // about 8 residual chunks per decide CTA (one per warp), while the
    // decide grid stays within one wave of resident CTAs
    H = (L.cR + kPassWarps - 1) / kPassWarps;
    const int cap = (occd * sms) / P0.B;
    if (H > cap) H = cap;
    if (H > 32) H = 32;
    if (H < 1) H = 1;
  }
  S.H = H;
  S.total = (int)total;
  S.fd_cT = make_fastdiv((unsigned)L.cT);
  S.fd_cP = make_fastdiv((unsigned)(L.cT + L.cD));
  S.fd_blk = make_fastdiv((unsigned)((long long)P0.B * (L.cT + L.cD) < (1LL << 31)
                                         ? P0.B * (L.cT + L.cD) : 1));
  S.fd_N = make_fastdiv((unsigned)(P0.N > 0 ? P0.N : 1));
  S.out_tokens = P0.out_tokens;
  S.out_nacc = P0.out_nacc;
  S.out_status = P0.out_status;
  S.out_path = P0.out_path;
  S.out_diag = P0.out_diag;
  S.claim = reinterpret_cast<unsigned *>(w + L.claim);
  S.claim_err = reinterpret_cast<unsigned long long *>(w + L.err);
  S.claim_ready = reinterpret_cast<unsigned long long *>(w + L.ready);
  S.claim_stamp = reinterpret_cast<unsigned long long *>(w + L.stamp);
  S.epoch_base = reinterpret_cast<unsigned long long *>(w + L.epoch_base);
  S.epoch_cur = reinterpret_cast<unsigned long long *>(w + L.epoch_cur);
  const unsigned long long call_id = next_call_id();
  S.part_tag = partial_tag(call_id);
  S.done = reinterpret_cast<unsigned *>(w + L.done);
  S.part = reinterpret_cast<Part *>(w + L.part);
  S.resid = reinterpret_cast<float *>(w + L.resid);
  const long long want = (total + kPassWarps - 1) / kPassWarps;
  const long long cap = (long long)sms * occ;
  int grid = (int)(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  // Trees whose stats grid would fill every SM leave stats slots free for
  // their decide CTAs (one per tree; a stats slot holds the registers of
  // `per` of them): those are then resident from the start, fetch their
  // code during the stream and merge each tree's node rows as its partials
  // arrive.
  bool tree_room = false;
  if (MODE == MODE_TREE && grid == cap && per >= 1) {
    const long long fewer = (P0.B + per - 1) / per;
    if (fewer * 8 <= cap) {  // (many trees: at most an eighth of the grid is given up)
      grid -= (int)fewer;
      tree_room = true;
    }
  }
  // Merging as partials arrive pays off when the stats work is many times
  // what its resident warps hold: the decide CTAs then only become resident
  // in the stats kernel's tail.  On a small call they would be resident
  // from the start and poll through the whole stats kernel.  A call captured
  // into a CUDA graph never polls: every replay carries the tag fixed at
  // capture, so an earlier replay's partials would look like its own.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) {
    (void)cudaGetLastError();
    capture = cudaStreamCaptureStatusActive;
  }
  // Trees poll when their stats grid left room for the decide CTAs.
  S.poll = capture == cudaStreamCaptureStatusNone && call_id < kPollCalls &&
           (total >= 16LL * grid * kPassWarps || tree_room);
  // Both kernels are programmatic dependents of the work before them: the
  // stats kernel of whatever the stream ran last (it waits on the device
  // before touching the workspace), the decide kernel of the stats kernel.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cs{};
    cs.gridDim = dim3((unsigned)grid);
    cs.blockDim = dim3(kPassThreads);
    cs.dynamicSmemBytes = 0;
    cs.stream = stream;
    cs.attrs = attr;
    cs.numAttrs = 1;
    if (cudaLaunchKernelEx(&cs, stats, S) != cudaSuccess) return SV_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(MODE == MODE_DRAFT ? (P0.B + kPassWarps - 1) / kPassWarps
                                                  : P0.B * H));  // a draft row per warp
  cfg.blockDim = dim3(kPassThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decide, S) != cudaSuccess) {
    // The claim counters were used and will not be reset, and the epoch
    // will not advance: clear the error, ready and stamp words, so that the
    // next call on this workspace (which reuses this call's epoch) resets
    // the counters itself and finds no word left by this call.
    (void)cudaMemsetAsync(w + L.err, 0, L.stamp + sizeof(unsigned long long) - L.err, stream);
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

// Rows on the 16-byte grid and rows off it run separate instantiations, so
// the aligned one carries no edge masks.
template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_pass(const KParams &P0, const PassLayout &L, long long total, bool unaligned,
                      cudaStream_t stream) {
  return unaligned ? launch_pass_t<MODE, TDT, DDT, PROBS, true>(P0, L, total, stream)
                   : launch_pass_t<MODE, TDT, DDT, PROBS, false>(P0, L, total, stream);
}

// Every row of an array starts on a 16-byte boundary.
inline bool rows_aligned(const void *p, int V, int es) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0 && ((size_t)V * es) % 16 == 0;
}

// The cluster path's shape for a call, if it takes that path: CS CTAs per
// batch row (or tree), S vocabulary entries per CTA, rstride bytes per kept
// row slice, dynamic shared memory bytes.  Every cluster of the call must be
// resident at once (cudaOccupancyMaxActiveClusters, asked once per device
// and cluster size with the most shared memory a call of the kernel takes).
// Chains: every kept slice fits kClusterSmemMax.  Trees: rows on 16-byte
// boundaries, at most kClusterTreeBytesMax of node rows in the call and at
// most 1 MB of node-row slices per CTA.
struct ClusterPlan {
  int CS, S, rstride;
  size_t smem;
};

constexpr size_t kTreeUnitSmemMax = 16 * 1024;  // tree unit partials per CTA
constexpr long long kClusterTreeBytesMax = 8LL << 20;  // node-row bytes of a small tree call
constexpr int kClusterSlots = 4;                       // cluster sizes 1, 2, 4, 8
constexpr int kClusterMinSlice = 1024;                 // vocabulary entries per chain CTA

template <int MODE, int TDT, int DDT, bool PROBS>
void *cluster_kernel() {
  if constexpr (MODE == MODE_TREE)
    return reinterpret_cast<void *>(sv_cluster_tree_kernel<TDT>);
  else
    return reinterpret_cast<void *>(sv_cluster_chain_kernel<MODE, TDT, DDT, PROBS>);
}

// Clusters of CS CTAs (CS = 1, 2, 4, 8 -> slot 0..3) that fit on the device
// at once; 0 if the kernel cannot be set up.  (Clusters of 16, a
// non-portable size, measured slower on the single-round chains.)
template <int MODE, int TDT, int DDT, bool PROBS>
int cluster_capacity(int dev, int slot) {
  static std::atomic<int> cache[kMaxDevices][kClusterSlots];
  int v = cache[dev][slot].load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  const void *kern = cluster_kernel<MODE, TDT, DDT, PROBS>();
  const size_t smem = MODE == MODE_TREE ? kTreeUnitSmemMax : (size_t)kClusterSmemMax;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
      cudaSuccess) {
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = 1u << slot;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1u << slot);
    cfg.blockDim = dim3(MODE == MODE_TREE ? kPassThreads : kClThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  if (n <= 0) (void)cudaGetLastError();
  cache[dev][slot].store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n > 0 ? n : 0;
}

template <int MODE, int TDT, int DDT, bool PROBS>
bool cluster_plan(const KParams &P, int dev, ClusterPlan &cp) {
  if (force_stream_path() || dev < 0 || dev >= kMaxDevices) return false;
  constexpr int esT = (TDT == SV_F32) ? 4 : 2, esD = (DDT == SV_F32) ? 4 : 2;
  if (MODE == MODE_TREE) {
    if (!rows_aligned(P.target, P.V, esT) || P.N > SV_MAX_TREE_NODES) return false;
    // a large call takes the cluster path only when its clusters put a CTA
    // on every SM; otherwise the streaming path's full grid reads faster
    const bool small = (long long)P.B * P.N * P.V * esT <= kClusterTreeBytesMax;
    const int sms = sm_count(dev);
    constexpr int E = Chunk<TDT>::kElems;
    for (int slot = kClusterSlots - 1; slot >= 0; --slot) {
      const int CS = 1 << slot;
      const int S = (int)align_up((size_t)((P.V + CS - 1) / CS), 8);
      const size_t smem = (size_t)P.N * ((S + E - 1) / E) * sizeof(float2);
      if ((long long)P.N * S * esT > (1LL << 20) || smem > kTreeUnitSmemMax) return false;
      if (!small && (long long)P.B * CS < sms) return false;
      if (P.B > cluster_capacity<MODE, TDT, DDT, PROBS>(dev, slot)) continue;
      cp = ClusterPlan{CS, S, 0, smem};
      return true;
    }
    return false;
  }
  if (MODE != MODE_CHAIN && MODE != MODE_CHAIN_GREEDY) return false;
  // the smallest cluster whose kept slices fit, then larger ones while the
  // slices keep at least kClusterMinSlice entries and the clusters still fit
  const int es = esT > esD ? esT : esD;
  const int keep = MODE == MODE_CHAIN ? 2 * P.gamma + 1 : P.gamma + 1;
  int chosen = -1;
  ClusterPlan best{};
  for (int slot = 0; slot < kClusterSlots; ++slot) {
    const int CS = 1 << slot;
    const int S = (int)align_up((size_t)((P.V + CS - 1) / CS), 8);
    const int rstride = (int)align_up((size_t)S * es, 16);
    // the kept slices, then (stochastic chains) the draw's weights
    const size_t smem = (size_t)keep * rstride +
                        (MODE == MODE_CHAIN ? align_up((size_t)S * sizeof(float), 16) : 0);
    if (smem > (size_t)kClusterSmemMax) continue;
    if (chosen >= 0 && S < kClusterMinSlice) break;
    if (P.B > cluster_capacity<MODE, TDT, DDT, PROBS>(dev, slot)) break;
    chosen = slot;
    best = ClusterPlan{CS, S, rstride, smem};
  }
  if (chosen < 0) return false;
  cp = best;
  return true;
}

// One launch of the cluster path: B clusters of CS CTAs, a programmatic
// dependent of the work before it in the stream.
template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_cluster(const KParams &P0, const ClusterPlan &cp, cudaStream_t stream) {
  ClusterParams C{};
  C.target = P0.target;
  C.draft = P0.draft;
  C.draft_tokens = P0.draft_tokens;
  C.temps = P0.temps;
  C.unif = P0.unif;
  C.parent = P0.parent;
  C.node_tokens = P0.node_tokens;
  C.B = P0.B;
  C.gamma = P0.gamma;
  C.V = P0.V;
  C.N = P0.N;
  C.max_depth = P0.max_depth;
  C.S = cp.S;
  C.rstride = cp.rstride;
  C.out_tokens = P0.out_tokens;
  C.out_nacc = P0.out_nacc;
  C.out_status = P0.out_status;
  C.out_path = P0.out_path;
  C.out_diag = P0.out_diag;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cp.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(P0.B * cp.CS));
  cfg.blockDim = dim3(MODE == MODE_TREE ? kPassThreads : kClThreads);
  cfg.dynamicSmemBytes = cp.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if constexpr (MODE == MODE_TREE)
    return cudaLaunchKernelEx(&cfg, sv_cluster_tree_kernel<TDT>, C) == cudaSuccess ? SV_OK
                                                                                   : SV_ERR_CUDA;
  else
    return cudaLaunchKernelEx(&cfg, sv_cluster_chain_kernel<MODE, TDT, DDT, PROBS>, C) ==
                   cudaSuccess
               ? SV_OK
               : SV_ERR_CUDA;
}

template <int MODE, int TDT, int DDT, bool PROBS>
sv_status launch_verify(const KParams &P, cudaStream_t stream) {
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    ClusterPlan cp;
    if (cluster_plan<MODE, TDT, DDT, PROBS>(P, dev, cp))
      return launch_cluster<MODE, TDT, DDT, PROBS>(P, cp, stream);
  }
  constexpr int esT = (TDT == SV_F32) ? 4 : 2, esD = (DDT == SV_F32) ? 4 : 2;
  const bool stream_draft = MODE == MODE_CHAIN && !PROBS;
  // (the residual sweep also reads probability drafts by vectors)
  const bool unaligned = !rows_aligned(P.target, P.V, esT) ||
                         (MODE == MODE_CHAIN && !rows_aligned(P.draft, P.V, esD));
  const PassLayout L = make_pass_layout(P.B, P.rows, P.V, esT, esD, stream_draft, unaligned);
  const long long total = pass_units<MODE, TDT, DDT, PROBS>(P, L);
  if (total < 0 || (long long)P.B * 16 >= (1LL << 31)) return SV_ERR_UNSUPPORTED;
  return launch_pass<MODE, TDT, DDT, PROBS>(P, L, total, unaligned, stream);
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
