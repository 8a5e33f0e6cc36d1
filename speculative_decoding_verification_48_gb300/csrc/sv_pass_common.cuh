// Shared definitions of the two-launch (streaming) verification path: chunk
// geometry, parameters, workspace layout, vector loads and warp-level merge /
// crossing helpers.
//
//   sv_stats_kernel   streams every logit row once.  Each warp reduces
//                     "warp-chunks" of 4 KB (32 lanes x 8 x 16-byte vectors)
//                     to a partial — (max, sum exp2) for a softmax row,
//                     (max, first index) for an argmax row — and stores it.
//                     Warps take chunks from striped claim counters (one
//                     atomic per chunk) and take no block barrier.
//   sv_decide_kernel  launched as a programmatic dependent of the first:
//                     merges the partials of each batch row, runs the accept
//                     tests / greedy match / tree walk, draws the bonus token
//                     from the partials of row gamma, and splits the residual
//                     sweep of a rejected row pair over several CTAs; the
//                     last of them finds the crossing chunk and rescans it.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kPassThreads = 256;
constexpr int kPassWarps = kPassThreads / 32;
constexpr int kChunkBytes = 4096;  // one warp-chunk of the stats kernel
constexpr int kChunkVecs = 8;      // 16-byte vectors per lane per warp-chunk
constexpr int kResidBytes = 2048;  // one residual chunk of a row pair
constexpr int kClaimStripes = 16;  // stats-kernel claim counters
constexpr int kClaimStride = 32;   // 128 bytes between counters
constexpr int kClaimProbes = 4096; // bound of the end-of-work probe loop
constexpr long long kReadySpins = 4000000;  // bound of the counter-reset wait (about a second)
constexpr int kPollSpins = 512;     // rounds of partial polling before the dependency wait
constexpr unsigned long long kStampValid = 0x5356434c41494d30ull;

template <int DT> struct Chunk {
  static constexpr int kEs = (int)sizeof(typename Elt<DT>::T);
  static constexpr int kVec = 16 / kEs;             // elements per 16-byte vector
  static constexpr int kElems = kChunkBytes / kEs;  // 1024 (2-byte types) or 512
  static constexpr int kPer = kElems / 32;          // elements per lane
};

// Residual chunks of a row pair: 2 KB of the wider of the two element types.
template <int TDT, int DDT> struct PairChunk {
  static constexpr int kEs = Chunk<TDT>::kEs > Chunk<DDT>::kEs ? Chunk<TDT>::kEs : Chunk<DDT>::kEs;
  static constexpr int kElems = kResidBytes / kEs;
  static constexpr int kVec = 16 / kEs;   // elements per vector, both rows
  static constexpr int kVecs = kElems / (32 * kVec);
  static constexpr int kPer = kElems / 32;
};

// Quotient by a divisor that is fixed for a call, without a hardware divide
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, floor(n / d) = (umulhi(n, m) + n) >> l,
// exact for 0 <= n < 2^31 and 1 <= d < 2^31 (the sum then fits 32 bits).
struct FastDiv {
  unsigned d, m, l;
};

inline FastDiv make_fastdiv(unsigned d) {
  unsigned l = 0;
  while ((1ull << l) < d) ++l;
  const unsigned long long m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, (unsigned)m, l};
}

__device__ __forceinline__ unsigned fdiv(unsigned n, const FastDiv &f) {
  return (__umulhi(n, f.m) + n) >> f.l;
}

// A warp-chunk partial: two values (max and scaled sum of a softmax chunk,
// or value and first index of an argmax chunk), each in its own 64-bit word
// with the call's tag in the high half.  Each word is written by one 64-bit
// store, so a reader that finds the tag in both words holds both values of
// this call, without waiting for the whole stats grid.
struct Part {
  unsigned long long a, b;
};

struct PassParams {
  const void *target;  // chain: [B, gamma+1, V]; tree: [B*N, V]
  const void *draft;   // [B, gamma, V] logits or fp32 probabilities
  const int32_t *draft_tokens;
  const float *temps;
  const float *unif;
  const int32_t *parent;
  const int32_t *node_tokens;
  int B, gamma, V, N, max_depth, rows;
  int cT, cD, cMax;  // warp-chunks per target row / draft row (0 if not streamed) / max
  int cR;            // residual chunks per row pair
  int H;             // decide CTAs per batch row
  int total;         // stats units (warp-chunks, skipped ones included)
  FastDiv fd_cT, fd_cP, fd_blk, fd_N;  // divisors of the unit decode: cT, cT + cD, B (cT + cD), N
  int32_t *out_tokens, *out_nacc, *out_status, *out_path;
  float *out_diag;
  unsigned *claim;   // [kClaimStripes * kClaimStride] stats-kernel claim counters
  unsigned long long *claim_err;    // == this call's epoch: its stats kernel hit a bound
  unsigned long long *claim_ready;  // == this call's epoch: its stats kernel zeroed the counters
  unsigned long long *claim_stamp;  // == kStampValid: the counters are zero (left so by the
                                    // previous call's decide kernel)
  unsigned long long *epoch_base;   // epoch of the last call that completed on this workspace
  unsigned long long *epoch_cur;    // epoch of the running call (epoch_base + 1)
  unsigned *done;    // [B] residual-sweep arrivals
  Part *part;        // [B][rows][cMax] warp-chunk partials
  unsigned part_tag; // odd, from the host's call id: marks this call's partials
  int poll;          // 1: the decide kernel merges as partials arrive (large calls)
  int unaligned;     // 1: some streamed row does not start on a 16-byte boundary
  float *resid;      // [B][cR] residual mass per chunk of the rejected row pair
};

// Workspace: a header of kPassHeaderBytes (claim counters; error, ready,
// stamp and epoch words), done[B], tagged partials, residual chunk sums.
//
// The header must be zero before the first call on the memory (and after
// the caller used the memory for anything else).  From then on every call
// keeps it valid: each call's decide kernel leaves the counters zeroed,
// records the call's epoch and stamps the counters valid, and a stats kernel
// that finds no valid stamp zeroes the counters itself before any claim.
//
// Epochs are counted on the device, one per call on the workspace (CUDA
// graph replays included): the stats kernel takes E = epoch_base + 1 after
// its dependency wait and publishes it in epoch_cur; the decide kernel reads
// epoch_cur after its own wait, and its CTA 0 sets epoch_base = E.  The
// error and ready words are compared with E, so a value left by an earlier
// call or replay never matches.
//
// Nothing after the header needs initialisation: done[] is zeroed by the
// stats kernel and partials carry their call's tag.
struct PassLayout {
  size_t claim, err, ready, stamp, epoch_base, epoch_cur, done, part, resid, total;
  int cT, cD, cMax, cR;
};

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Rows off the 16-byte grid are read on the 16-byte grid of their own
// address: a row's first chunk starts up to one vector before the row, so it
// may take one chunk more (and its pair sweep one residual chunk more).
inline PassLayout make_pass_layout(int B, int rows, int V, int esT, int esD, bool stream_draft,
                                   bool unaligned) {
  PassLayout L;
  const int esR = esT > esD ? esT : esD;
  L.cT = ceil_div(V + (unaligned ? 16 / esT - 1 : 0), kChunkBytes / esT);
  L.cD = stream_draft ? ceil_div(V + (unaligned ? 16 / esD - 1 : 0), kChunkBytes / esD) : 0;
  L.cMax = L.cT > L.cD ? L.cT : L.cD;
  L.cR = ceil_div(V + (unaligned ? 16 / esR - 1 : 0), kResidBytes / esR);
  L.claim = 0;
  L.err = (size_t)kClaimStripes * kClaimStride * 4;
  L.ready = L.err + 128;
  L.stamp = L.ready + 128;
  L.epoch_base = L.stamp + 128;
  L.epoch_cur = L.epoch_base + 128;
  size_t off = kPassHeaderBytes;
  L.done = off;  off = align_up(off + (size_t)B * 4, 256);
  L.part = off;  off = align_up(off + (size_t)B * rows * L.cMax * sizeof(Part), 256);
  L.resid = off; off = align_up(off + (size_t)B * L.cR * sizeof(float), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p) {
  return *reinterpret_cast<const volatile unsigned *>(p);
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// 16-byte streaming load through the non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_nc16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_nc8(const void *p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

// VEC elements of dtype DT starting at p (VEC * size = 8 or 16 bytes, aligned).
template <int DT, int VEC>
__device__ __forceinline__ void vec_load(const typename Elt<DT>::T *p, float *o) {
  constexpr int kB = VEC * (int)sizeof(typename Elt<DT>::T);
  static_assert(kB == 16 || kB == 8, "vector loads are 8 or 16 bytes");
  if constexpr (kB == 16) Elt<DT>::unpack(ld_nc16(p), o);
  else Elt<DT>::unpack(ld_nc8(p), o);
}

// One raw vector of VEC elements of DT (8 or 16 bytes), loaded now and
// unpacked when used.
// Asynchronous copy of 8 or 16 bytes from global to shared memory (no
// register staging); completion is per thread, after cp_async_wait_all.
template <int BYTES>
__device__ __forceinline__ void cp_async(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  if constexpr (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

template <int DT, int VEC> struct RawVec {
  static constexpr int kB = VEC * (int)sizeof(typename Elt<DT>::T);
  static_assert(kB == 16 || kB == 8, "vector loads are 8 or 16 bytes");
  using R = typename std::conditional<kB == 16, uint4, uint2>::type;
  R r;
  __device__ __forceinline__ void load(const typename Elt<DT>::T *p) {
    if constexpr (kB == 16) r = ld_nc16(p);
    else r = ld_nc8(p);
  }
  __device__ __forceinline__ void unpack(float *o) const { Elt<DT>::unpack(r, o); }
};

// Residual term max(0, p(x) - q(x)) of the sweep: p(x) = 2^((l_p(x) - M_p) c
// - log2 Z_p), one FADD, one FFMA and one ex2 per side (q is read as given
// for probability drafts).  The row maximum is subtracted before the scale,
// so the exponent of an element near the maximum is small and exact to a
// few ulp even at a tiny temperature (large c).  Identical rows give
// identical p and q, hence exactly zero; NaN propagates.
struct ResidCoef {
  float c, Mp, lzp, Mq, lzq;  // scale, then each side's maximum and log2 normaliser
};

// Packed pairs of fp32 (sm_100+ two-wide FMA / ADD): one instruction for
// two lanes of work.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The residual term for two neighbouring elements through the two-wide
// FADD and FMA (rounded per lane, p - q rounded once).
template <bool PROBS>
__device__ __forceinline__ float2 resid_pair(float lp0, float lp1, float lq0, float lq1,
                                             const ResidCoef &k) {
  const unsigned long long c2 = f2_pack(k.c, k.c);
  const unsigned long long dp = f2_add(f2_pack(lp0, lp1), f2_pack(-k.Mp, -k.Mp));
  const float2 pe = f2_unpack(f2_fma(dp, c2, f2_pack(-k.lzp, -k.lzp)));
  const unsigned long long p2 = f2_pack(ex2(pe.x), ex2(pe.y));
  unsigned long long q2;
  if (PROBS) {
    q2 = f2_pack(lq0, lq1);
  } else {
    const unsigned long long dq = f2_add(f2_pack(lq0, lq1), f2_pack(-k.Mq, -k.Mq));
    const float2 qe = f2_unpack(f2_fma(dq, c2, f2_pack(-k.lzq, -k.lzq)));
    q2 = f2_pack(ex2(qe.x), ex2(qe.y));
  }
  const float2 d = f2_unpack(f2_fma(q2, f2_pack(-1.f, -1.f), p2));  // p - q
  return make_float2(max_nan(0.f, d.x), max_nan(0.f, d.y));
}

// Wait for the grid this one depends on (programmatic dependent launch);
// returns at once when the launch had no such dependency.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the dependent grid start launching (its CTAs still wait in
// grid_dependency_wait until this grid has completed and flushed).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long part_word(float v, unsigned tag) {
  return ((unsigned long long)tag << 32) | __float_as_uint(v);
}
__device__ __forceinline__ void part_store(Part *p, float x, float y, unsigned tag) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(part_word(x, tag)),
               "l"(part_word(y, tag))
               : "memory");
}
// The values of a partial read after the dependency wait (complete by then).
__device__ __forceinline__ float2 part_value(const Part *p) {
  const ulonglong2 w = __ldcg(reinterpret_cast<const ulonglong2 *>(p));
  return make_float2(__uint_as_float((unsigned)w.x), __uint_as_float((unsigned)w.y));
}
// One poll of a partial that may still be written.
__device__ __forceinline__ void part_poll(const Part *p, unsigned long long &a,
                                          unsigned long long &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool part_tagged(unsigned long long a, unsigned long long b,
                                            unsigned tag) {
  return (unsigned)(a >> 32) == tag && (unsigned)(b >> 32) == tag;
}

// Softmax merge of two partials (m, s), s = sum 2^((x - m) c).  -inf maxima
// carry no mass; NaN anywhere gives NaN.
__device__ __forceinline__ float2 softmax_merge(float2 a, float2 b, float c) {
  const float M = max_nan(a.x, b.x);
  const float za = (a.x == -CUDART_INF_F) ? 0.f : a.y * ex2((a.x - M) * c);
  const float zb = (b.x == -CUDART_INF_F) ? 0.f : b.y * ex2((b.x - M) * c);
  return make_float2(M, za + zb);
}

// Merge of one softmax row's `cnt` chunk partials by the whole warp: lanes
// take chunks lane, lane + 32, ... (eight loads in flight per lane), then the
// lane results are combined.  Returns (M, Z) with Z = sum_x 2^((x - M) c).
static __device__ __noinline__ float2 warp_row_softmax(const Part *part, int cnt, float c) {
  const int lane = lane_id();
  float2 acc = make_float2(-CUDART_INF_F, 0.f);
  for (int i0 = 0; i0 < cnt; i0 += 256) {
    float2 pt[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = i0 + lane + 32 * k;
      pt[k] = i < cnt ? part_value(part + i) : make_float2(-CUDART_INF_F, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) acc = softmax_merge(acc, pt[k], c);
  }
  const float M = warp_max_nan(acc.x);
  const float z = (acc.x == -CUDART_INF_F) ? 0.f : acc.y * ex2((acc.x - M) * c);
  return make_float2(M, warp_sum(z));
}

// Two softmax rows merged by one warp with the loads of both in flight at
// once (each row at most 256 chunks); `pb2` may be null.
__device__ __forceinline__ void warp_rows_softmax2(const Part *pa, int ca, const Part *pb2,
                                                   int cb, float c, float2 &ra, float2 &rb) {
  const int lane = lane_id();
  float2 xa[8], xb[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = lane + 32 * k;
    xa[k] = i < ca ? part_value(pa + i) : make_float2(-CUDART_INF_F, 0.f);
    xb[k] = (pb2 && i < cb) ? part_value(pb2 + i) : make_float2(-CUDART_INF_F, 0.f);
  }
  float2 aa = make_float2(-CUDART_INF_F, 0.f), ab = aa;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    aa = softmax_merge(aa, xa[k], c);
    ab = softmax_merge(ab, xb[k], c);
  }
  const float Ma = warp_max_nan(aa.x), Mb = warp_max_nan(ab.x);
  const float za = (aa.x == -CUDART_INF_F) ? 0.f : aa.y * ex2((aa.x - Ma) * c);
  const float zb = (ab.x == -CUDART_INF_F) ? 0.f : ab.y * ex2((ab.x - Mb) * c);
  ra = make_float2(Ma, warp_sum(za));
  rb = make_float2(Mb, warp_sum(zb));
}

// warp_rows_softmax2 for rows of at most 64 chunks, run before the
// dependency wait: each lane holds up to two chunk partials of each row and
// re-reads those that do not carry this call's tag yet, at most `spins`
// rounds.  True, with the merged rows, once every partial carries the tag;
// false if the bound ran out (the caller then waits and merges again).
__device__ __forceinline__ bool warp_rows_softmax2_poll(const Part *pa, int ca, const Part *pb2,
                                                        int cb, float c, unsigned tag,
                                                        int spins, float2 &ra, float2 &rb) {
  const int lane = lane_id();
  unsigned long long wa[2][2], wb[2][2];
  bool na[2], nb[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    na[k] = lane + 32 * k < ca;
    nb[k] = pb2 != nullptr && lane + 32 * k < cb;
    wa[k][0] = wa[k][1] = wb[k][0] = wb[k][1] = 0ull;
  }
  for (int it = 0;; ++it) {
    bool pending = false;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (na[k]) part_poll(pa + lane + 32 * k, wa[k][0], wa[k][1]);
      if (nb[k]) part_poll(pb2 + lane + 32 * k, wb[k][0], wb[k][1]);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      na[k] = na[k] && !part_tagged(wa[k][0], wa[k][1], tag);
      nb[k] = nb[k] && !part_tagged(wb[k][0], wb[k][1], tag);
      pending |= na[k] || nb[k];
    }
    if (!__any_sync(0xffffffffu, pending)) break;
    if (it >= spins) return false;
    __nanosleep(128);
  }
  float2 aa = make_float2(-CUDART_INF_F, 0.f), ab = aa;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (lane + 32 * k < ca)
      aa = softmax_merge(aa, make_float2(__uint_as_float((unsigned)wa[k][0]),
                                         __uint_as_float((unsigned)wa[k][1])), c);
    if (pb2 != nullptr && lane + 32 * k < cb)
      ab = softmax_merge(ab, make_float2(__uint_as_float((unsigned)wb[k][0]),
                                         __uint_as_float((unsigned)wb[k][1])), c);
  }
  const float Ma = warp_max_nan(aa.x), Mb = warp_max_nan(ab.x);
  const float za = (aa.x == -CUDART_INF_F) ? 0.f : aa.y * ex2((aa.x - Ma) * c);
  const float zb = (ab.x == -CUDART_INF_F) ? 0.f : ab.y * ex2((ab.x - Mb) * c);
  ra = make_float2(Ma, warp_sum(za));
  rb = make_float2(Mb, warp_sum(zb));
  return true;
}

// Merge of one argmax row's chunk partials (value, global first index): the
// largest value, and the lowest index among chunks holding it.  NaN anywhere
// gives a NaN value.
static __device__ __noinline__ float2 warp_row_argmax(const Part *part, int cnt) {
  const int lane = lane_id();
  float best = -CUDART_INF_F;
  int idx = 0x7fffffff;
  bool nan = false;
  for (int i0 = 0; i0 < cnt; i0 += 256) {
    float2 pt[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = i0 + lane + 32 * k;
      pt[k] = i < cnt ? part_value(part + i) : make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      nan |= isnan(pt[k].x);
      const int ik = __float_as_int(pt[k].y);
      if (pt[k].x > best || (pt[k].x == best && ik < idx)) {
        best = pt[k].x;
        idx = ik;
      }
    }
  }
  const bool anynan = __any_sync(0xffffffffu, nan);
  const float M = warp_max_nan(best);
  const int I = warp_min_int(best == M ? idx : 0x7fffffff);
  return make_float2(anynan ? CUDART_NAN_F : M, __int_as_float(I));
}

}  // namespace sv
