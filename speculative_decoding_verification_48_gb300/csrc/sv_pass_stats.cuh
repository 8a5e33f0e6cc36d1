// Row statistics pass: every logit row the verification needs is read once
// from HBM and reduced to warp-chunk partials.
//
// Softmax rows ("論文解説: Speculative Sampling", §実装のポイント: both models'
// rows go through softmax(logits / T)): (m, s) with m the chunk maximum and
// s = sum_x 2^(x c - m c), c = log2(e) / T.  Argmax rows (greedy rows,
// "投機的デコーディングとは？" §ドラフト生成と並列検証の仕組み, and tree nodes, SpecInfer
// explainer §推論方法): (max value, lowest index holding it).
//
// Work is a list of warp-chunks that warps claim one at a time from striped
// counters (below), so the grid reads one contiguous front of memory and
// fast warps take more chunks than slow ones.
// Each warp keeps the next chunk's eight 16-byte loads per lane in flight
// while it reduces the current one.
//
// Rows need not start on 16-byte boundaries: a row's chunks lie on the
// 16-byte grid of its own address (its first chunk starts up to 15 bytes
// before the row).  Every aligned 16-byte block holding an element of the
// row is loaded whole, and the slots outside the row are masked when the
// chunk is reduced.  A block holding a byte of the row never lies on another
// page, so the loads stay within mapped memory.  For chains the list runs from the last
// draft position to the first: the rows that the residual sweep is most
// likely to re-read (early positions, where the first rejection usually
// falls) are then the most recently read when the sweep starts, and still in
// L2.  Warp-chunks a row does not need (draft rows of greedy rows, every row
// of a row with an invalid temperature) cost nothing.
#pragma once

#include "sv_pass_sample.cuh"

namespace sv {

enum ChunkKind { CK_SKIP = 0, CK_SOFTMAX = 1, CK_ARGMAX = 2 };

struct ChunkRef {
  const void *src;  // first byte of the warp-chunk (16-byte aligned)
  Part *dst;        // its partial
  unsigned tag;     // this call's partial tag
  int kind;
  int x0;           // vocabulary index of the chunk's slot 0 (negative: before the row)
  int lo, n;        // the slots [lo, n) hold row elements
  int draft;        // 1: element type DDT, else TDT
  float c;
};

// Elements of a row before its first 16-byte boundary (0 on aligned paths).
template <int DT>
__device__ __forceinline__ int row_offset16(const void *row) {
  return (int)((reinterpret_cast<uintptr_t>(row) & 15) / sizeof(typename Elt<DT>::T));
}

template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
__device__ __forceinline__ ChunkRef decode_chunk(const PassParams &P, int k) {
  ChunkRef r;
  int b, row, ci, draft = 0, pos = 0;
  if (MODE == MODE_TREE || MODE == MODE_DRAFT) {
    // global row b * N + n (a draft batch has N = 1 row per batch entry)
    const int gr = (int)fdiv((unsigned)k, P.fd_cT);
    ci = k - gr * P.cT;
    b = (int)fdiv((unsigned)gr, P.fd_N);
    row = gr - b * P.N;
  } else {
    const int g = P.gamma;
    const int cP = P.cT + P.cD;
    const int head = P.B * P.cT;  // position gamma: target rows only
    if (k < head) {
      pos = g;
      b = (int)fdiv((unsigned)k, P.fd_cT);
      ci = k - b * P.cT;
    } else {
      const int k2 = k - head;
      const int blk = (int)fdiv((unsigned)k2, P.fd_blk);
      pos = g - 1 - blk;
      const int r2 = k2 - blk * P.B * cP;
      b = (int)fdiv((unsigned)r2, P.fd_cP);
      const int t = r2 - b * cP;
      draft = t >= P.cT;
      ci = draft ? t - P.cT : t;
    }
    row = draft ? g + 1 + pos : pos;
  }
  const int E = draft ? Chunk<DDT>::kElems : Chunk<TDT>::kElems;
  const int ES = draft ? Chunk<DDT>::kEs : Chunk<TDT>::kEs;
  const char *rowp;
  if (draft) {
    rowp = static_cast<const char *>(P.draft) + ((size_t)b * P.gamma + pos) * P.V * ES;
  } else {
    const int rows_per = (MODE == MODE_TREE || MODE == MODE_DRAFT) ? P.N : P.gamma + 1;
    rowp = static_cast<const char *>(P.target) + ((size_t)b * rows_per + row) * P.V * ES;
  }
  const int off = UNAL ? (int)((reinterpret_cast<uintptr_t>(rowp) & 15) / ES) : 0;
  r.x0 = ci * E - off;
  r.lo = ci == 0 ? off : 0;
  r.n = min(E, P.V - r.x0);
  r.src = rowp + (ptrdiff_t)r.x0 * ES;
  r.draft = draft;
  r.dst = P.part + ((size_t)b * P.rows + row) * P.cMax + ci;
  r.tag = P.part_tag;
  r.c = 0.f;
  if (MODE == MODE_CHAIN || MODE == MODE_DRAFT) {
    const float T = __ldg(P.temps + b);
    if (bad_temperature(T)) r.kind = CK_SKIP;
    else if (T > 0.f) { r.kind = CK_SOFTMAX; r.c = kLog2e / T; }
    else r.kind = draft ? CK_SKIP : CK_ARGMAX;
  } else {
    r.kind = CK_ARGMAX;
  }
  return r;
}

// Packed -inf of one 32-bit word of each element type.
template <int DT> __device__ __forceinline__ unsigned neg_inf_word() {
  return DT == SV_F32 ? 0xff800000u : (DT == SV_BF16 ? 0xff80ff80u : 0xfc00fc00u);
}

// The lane's eight 16-byte vectors of a warp-chunk: vector l + 32 u holds
// slots [VEC (l + 32 u), VEC (l + 32 u) + VEC).  Vectors with no slot of
// the row are filled with -inf instead of loaded.
template <int DT, bool UNAL>
__device__ __forceinline__ void chunk_issue_t(const ChunkRef &r, uint4 (&buf)[kChunkVecs]) {
  constexpr int VEC = Chunk<DT>::kVec, ES = Chunk<DT>::kEs;
  const int lane = lane_id();
  const unsigned ni = neg_inf_word<DT>();
#pragma unroll
  for (int u = 0; u < kChunkVecs; ++u) {
    const int e = (lane + 32 * u) * VEC;
    if (e < r.n && (!UNAL || e + VEC > r.lo))
      buf[u] = ld_nc16(static_cast<const char *>(r.src) + (ptrdiff_t)e * ES);
    else
      buf[u] = make_uint4(ni, ni, ni, ni);
  }
}

template <int TDT, int DDT, bool UNAL>
__device__ __forceinline__ void chunk_issue(const ChunkRef &r, uint4 (&buf)[kChunkVecs]) {
  if (r.kind == CK_SKIP) return;
  if (TDT == DDT || !r.draft) chunk_issue_t<TDT, UNAL>(r, buf);
  else chunk_issue_t<DDT, UNAL>(r, buf);
}

// The vector of slots e .. e + VEC - 1 with the slots outside [lo, hi) set
// to -inf.
template <int DT>
__device__ __forceinline__ uint4 mask_vec(uint4 v, int e, int lo, int hi) {
  unsigned w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (DT == SV_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!(e + i >= lo && e + i < hi)) w[i] = 0xff800000u;
  } else {
    const unsigned ni = DT == SV_BF16 ? 0xff80u : 0xfc00u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int x = e + 2 * i;
      const unsigned a = (x >= lo && x < hi) ? (w[i] & 0xffffu) : ni;
      const unsigned b = (x + 1 >= lo && x + 1 < hi) ? (w[i] & 0xffff0000u) : (ni << 16);
      w[i] = a | b;
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// NaN-propagating max of two packed words (2 x bf16, 2 x f16 or 1 x f32).
template <int DT> __device__ __forceinline__ unsigned packed_max(unsigned a, unsigned b) {
  unsigned d;
  if constexpr (DT == SV_BF16) asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else if constexpr (DT == SV_F16) asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.NaN.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// The larger of the elements in a packed word, as f32 (NaN if either is).
template <int DT> __device__ __forceinline__ float packed_word_max(unsigned w) {
  if constexpr (DT == SV_F32) {
    return __uint_as_float(w);
  } else {
    float lo, hi;
    if constexpr (DT == SV_BF16) {
      lo = __uint_as_float(w << 16);
      hi = __uint_as_float(w & 0xffff0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
      lo = f.x;
      hi = f.y;
    }
    return max_nan(lo, hi);
  }
}

// Reduces a loaded chunk; slots outside the row are masked (rows off the
// 16-byte grid only: on the aligned path a row ends on a vector boundary and
// the vectors past it were filled with -inf).
template <int DT, bool UNAL>
__device__ __forceinline__ void chunk_reduce(const ChunkRef &r, uint4 (&buf)[kChunkVecs]) {
  using C = Chunk<DT>;
  constexpr int VEC = C::kVec;
  const int lane = lane_id();
  if (UNAL && (r.lo > 0 || r.n < C::kElems)) {  // a row's first or last chunk
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int e = (lane + 32 * u) * VEC;
      if (e < r.lo || e + VEC > r.n) buf[u] = mask_vec<DT>(buf[u], e, r.lo, r.n);
    }
  }
  // chunk maximum on packed words
  unsigned mw[4] = {buf[0].x, buf[0].y, buf[0].z, buf[0].w};
#pragma unroll
  for (int u = 1; u < kChunkVecs; ++u) {
    mw[0] = packed_max<DT>(mw[0], buf[u].x);
    mw[1] = packed_max<DT>(mw[1], buf[u].y);
    mw[2] = packed_max<DT>(mw[2], buf[u].z);
    mw[3] = packed_max<DT>(mw[3], buf[u].w);
  }
  const float m = warp_max_nan(
      packed_word_max<DT>(packed_max<DT>(packed_max<DT>(mw[0], mw[1]), packed_max<DT>(mw[2], mw[3]))));
  float2 out;
  if (r.kind == CK_SOFTMAX) {
    // s = sum 2^(x c - m c).  The exponent is one FFMA against mc = RN(m c);
    // that scales every term by 2^d, d = m c - mc (exact by FMA), which is
    // divided out once.  A huge |m c| (tiny T) or a non-finite m falls back
    // to (x - m) c, which also turns +inf / NaN into a NaN sum.
    const float c = r.c;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
    float scale = 1.f;
    if (m != -CUDART_INF_F) {
      const float mc = m * c;
      if (fabsf(mc) <= 1.0e37f) {
        const float d = fmaf(m, c, -mc);
        // element pairs through the two-wide FMA and ADD
        const unsigned long long c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
        unsigned long long acc[2] = {0ull, 0ull};  // (+0, +0) pairs
#pragma unroll
        for (int u = 0; u < kChunkVecs; ++u) {
          float v[VEC];
          Elt<DT>::unpack(buf[u], v);
#pragma unroll
          for (int t = 0; t < VEC; t += 2) {
            const float2 e = f2_unpack(f2_fma(f2_pack(v[t], v[t + 1]), c2, nmc2));
            acc[(t >> 1) & 1] = f2_add(acc[(t >> 1) & 1], f2_pack(ex2(e.x), ex2(e.y)));
          }
        }
        const float2 a0 = f2_unpack(acc[0]), a1 = f2_unpack(acc[1]);
        s4[0] = a0.x; s4[1] = a0.y; s4[2] = a1.x; s4[3] = a1.y;
        scale = ex2(-d);
      } else {
#pragma unroll
        for (int u = 0; u < kChunkVecs; ++u) {
          float v[VEC];
          Elt<DT>::unpack(buf[u], v);
#pragma unroll
          for (int t = 0; t < VEC; ++t) s4[t & 3] += ex2((v[t] - m) * c);
        }
      }
    }
    out = make_float2(m, warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3])) * scale);
  } else {
    int idx = 0x7fffffff;
#pragma unroll
    for (int u = kChunkVecs - 1; u >= 0; --u) {
      float v[VEC];
      Elt<DT>::unpack(buf[u], v);
#pragma unroll
      for (int t = VEC - 1; t >= 0; --t) {
        const int e = (lane + 32 * u) * VEC + t;
        if (v[t] == m && (!UNAL || (e >= r.lo && e < r.n))) idx = e;  // descending: keeps the lowest
      }
    }
    idx = warp_min_int(idx);
    out = make_float2(m, __int_as_float(idx == 0x7fffffff ? idx : r.x0 + idx));
  }
  if (lane == 0) part_store(r.dst, out.x, out.y, r.tag);
}

template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
__device__ __forceinline__ void chunk_process(const ChunkRef &r, uint4 (&buf)[kChunkVecs]) {
  if (r.kind == CK_SKIP) return;
  if (TDT == DDT || !r.draft) chunk_reduce<TDT, UNAL>(r, buf);
  else chunk_reduce<DDT, UNAL>(r, buf);
}

// Work claims.  Warp w of the grid takes chunk w first, without a claim;
// the chunks after the grid's first k0 = gridDim.x * kPassWarps are claimed
// dynamically from kClaimStripes counters, counter s handing out the chunks
// k = k0 + kClaimStripes * i + s in order, so all stripes advance through
// the list together (one contiguous front in memory, the list order kept)
// while no single address takes every atomic.  A warp starts on stripe
// (warp index mod kClaimStripes); when its stripe runs dry it reads every
// counter at once and moves to a stripe with chunks left.  Returns -1 once
// every stripe is exhausted.
struct Claimer {
  int s;
  long long k0;
};

// Flags this call (epoch E) as unfinished: its decide kernel then reports
// SV_ROW_TIMEOUT on every row.
__device__ __forceinline__ void claim_fail(const PassParams &P, unsigned long long E) {
  if (lane_id() == 0) *reinterpret_cast<volatile unsigned long long *>(P.claim_err) = E;
}

// Bounded wait until this call's stats kernel (epoch E) has zeroed the
// counters (slow path only); false, with the call flagged, if the bound is
// hit.
__device__ __forceinline__ bool counters_reset_wait(const PassParams &P, unsigned long long E) {
  bool ok = true;
  if (lane_id() == 0) {
    ok = false;
    for (long long it = 0; it < kReadySpins; ++it) {
      if (ld_acquire_u64(P.claim_ready) == E) {
        ok = true;
        break;
      }
      __nanosleep(32);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) claim_fail(P, E);
  return ok;
}

__device__ __forceinline__ unsigned claim_issue(const PassParams &P, const Claimer &c) {
  unsigned v = 0;
  if (lane_id() == 0) v = atomicAdd(P.claim + c.s * kClaimStride, 1u);
  return v;
}

// The chunk of the claim in flight on the warp's current stripe (the one
// claim in flight is always resolved before the warp can move to another
// stripe), or -1 when that stripe is exhausted: lanes below kClaimStripes
// then hold in cnt a read of every counter, issued here and first used by
// claim_probe after the warp's current chunk, so the stripe change costs
// the chunk no round trip.
__device__ __forceinline__ int claim_take(const PassParams &P, const Claimer &c, unsigned pend,
                                          unsigned &cnt) {
  const int lane = lane_id();
  const long long k = c.k0 + (long long)__shfl_sync(0xffffffffu, pend, 0) * kClaimStripes + c.s;
  if (k < P.total) return (int)k;
  cnt = lane < kClaimStripes ? ld_volatile_u32(P.claim + lane * kClaimStride) : 0xffffffffu;
  return -1;
}

// A claim on a stripe with chunks left, from the counters read by
// claim_take (read again after a lost race); -1 once every stripe is
// exhausted.  Every probe finds a stripe with chunks left or ends the loop;
// a claim lost to a race only repeats the probe, so the bound is never
// reached in practice — if it were, the call is flagged rather than left
// unfinished.
static __device__ __noinline__ int claim_probe(const PassParams &P, Claimer &c, unsigned cnt,
                                               unsigned long long E) {
  const int lane = lane_id();
  for (int probe = 0;; ++probe) {
    if (probe == kClaimProbes) {
      claim_fail(P, E);
      return -1;
    }
    if (probe > 0)
      cnt = lane < kClaimStripes ? ld_volatile_u32(P.claim + lane * kClaimStride) : 0xffffffffu;
    const bool has = lane < kClaimStripes && c.k0 + (long long)cnt * kClaimStripes + lane < P.total;
    const unsigned m = __ballot_sync(0xffffffffu, has);
    if (!m) return -1;
    c.s = __ffs(m) - 1;
    const long long k =
        c.k0 + (long long)__shfl_sync(0xffffffffu, claim_issue(P, c), 0) * kClaimStripes + c.s;
    if (k < P.total) return (int)k;
  }
}

template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
__global__ void __launch_bounds__(kPassThreads, 2) sv_stats_kernel(const PassParams P) {
  // This kernel is a programmatic dependent of whatever the stream ran
  // before (typically the previous call's decide kernel, or the kernel that
  // wrote the logits): neither the inputs nor the workspace are touched
  // before that work has completed.
  grid_dependency_wait();
  // Only then may the decide kernel launch (its CTAs take the place of
  // finished stats CTAs and wait on the device for this grid to complete):
  // it reads inputs before that wait, so the work that wrote them must be
  // complete, even where that work let its own dependents launch early.
  grid_dependents_launch();
  // The warp's first chunk needs no claim: its loads are in flight while
  // the counters are checked and the first claim is made.
  const int kw = blockIdx.x * kPassWarps + warp_id();
  Claimer cl{kw % kClaimStripes, (long long)gridDim.x * kPassWarps};
  uint4 b0[kChunkVecs], b1[kChunkVecs];
  int ka = kw < P.total ? kw : -1;
  ChunkRef ra;
  ra.kind = CK_SKIP;
  if (ka >= 0) {
    ra = decode_chunk<MODE, TDT, DDT, PROBS, UNAL>(P, ka);
    chunk_issue<TDT, DDT, UNAL>(ra, b0);
  }
  // This call's epoch.  epoch_base is written only by this call's decide
  // kernel after this grid has completed, so every CTA reads the same value.
  const unsigned long long E = __ldcg(P.epoch_base) + 1ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) *P.epoch_cur = E;
  // residual-sweep arrival counters of this call start at zero (the decide
  // kernel reads them only after this grid has completed)
  for (int i = blockIdx.x * kPassThreads + threadIdx.x; i < P.B; i += gridDim.x * kPassThreads)
    P.done[i] = 0u;
  // Claim counters: zero and stamped valid by the previous call's decide
  // kernel, else (fresh or overwritten workspace) zeroed here by thread 0 of
  // CTA 0 while every warp waits.  The stamp is not written while this grid
  // runs, so all warps take the same path.  A plain load suffices: the
  // dependency wait above made the previous kernel's writes visible (an
  // acquire would also hold this warp's claim behind its chunk loads).
  const bool stamped = __ldcg(P.claim_stamp) == kStampValid;
  if (!stamped && blockIdx.x == 0 && threadIdx.x == 0) {
    for (int s = 0; s < kClaimStripes; ++s) P.claim[s * kClaimStride] = 0u;
    __threadfence();
    st_release_u64(P.claim_ready, E);
  }
  if (!stamped && !counters_reset_wait(P, E)) return;
  if (ka >= 0) {  // (a warp without a first chunk has none to claim either)
    unsigned pend = claim_issue(P, cl);  // the next claim is in flight while a chunk is reduced
    unsigned cnt = 0xffffffffu;
    // two chunks per iteration so both buffers have static names
    while (true) {
      int kb = claim_take(P, cl, pend, cnt);
      ChunkRef rb;
      rb.kind = CK_SKIP;
      if (kb >= 0) {
        rb = decode_chunk<MODE, TDT, DDT, PROBS, UNAL>(P, kb);
        chunk_issue<TDT, DDT, UNAL>(rb, b1);
        pend = claim_issue(P, cl);
      }
      chunk_process<MODE, TDT, DDT, PROBS, UNAL>(ra, b0);
      if (kb < 0) {
        kb = claim_probe(P, cl, cnt, E);
        if (kb < 0) break;
        rb = decode_chunk<MODE, TDT, DDT, PROBS, UNAL>(P, kb);
        chunk_issue<TDT, DDT, UNAL>(rb, b1);
        pend = claim_issue(P, cl);
      }
      ka = claim_take(P, cl, pend, cnt);
      if (ka >= 0) {
        ra = decode_chunk<MODE, TDT, DDT, PROBS, UNAL>(P, ka);
        chunk_issue<TDT, DDT, UNAL>(ra, b0);
        pend = claim_issue(P, cl);
      }
      chunk_process<MODE, TDT, DDT, PROBS, UNAL>(rb, b1);
      if (ka < 0) {
        ka = claim_probe(P, cl, cnt, E);
        if (ka < 0) break;
        ra = decode_chunk<MODE, TDT, DDT, PROBS, UNAL>(P, ka);
        chunk_issue<TDT, DDT, UNAL>(ra, b0);
        pend = claim_issue(P, cl);
      }
    }
  }
}

}  // namespace sv
