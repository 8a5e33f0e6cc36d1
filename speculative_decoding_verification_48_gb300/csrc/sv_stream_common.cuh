// Shared definitions of the streaming verification kernel (sm_103a): tile
// geometry, parameters, shared-memory layout, mbarrier / bulk-copy PTX, and
// the per-warp reductions the consumer warps run over one stage.
#pragma once

#include "sv_kernel.cuh"

namespace sv {

constexpr int kCW = 16;                            // consumer warps
constexpr int kStreamWarps = kCW + 4;              // + producer, bookkeeper, decider, scheduler
constexpr int kStreamThreads = kStreamWarps * 32;  // 640
constexpr int kStages = 6;
constexpr int kStageBytes = 32768;
constexpr int kDQ = 64;                            // decider queue entries
constexpr int kBookBatch = 16;                     // units per bookkeeper fence (<= 32)
constexpr int kPR = 32;                            // slice-partial ring (consumers -> bookkeeper)
constexpr int kClaim = 8;                          // Phase-A units per claim
constexpr int kPoll = 8;                           // units between queue-counter polls
constexpr int kRing = 16;                          // scheduler -> producer descriptors
constexpr int kSchedBatch = 8;                     // descriptors per scheduler step
constexpr long long kStreamWait = 4000000000LL;    // bound of every wait, in clocks

// Elements per Phase-A tile (one row) and per Phase-B tile (a row pair).
template <int DT> struct TileA {
  static constexpr int kElems = kStageBytes / (int)sizeof(typename Elt<DT>::T);
  static constexpr int kSlice = kElems / kCW;  // elements per consumer warp
};
template <int TDT, int DDT> struct TileB {
  static constexpr bool kNarrow = sizeof(typename Elt<TDT>::T) == 2 &&
                                  sizeof(typename Elt<DDT>::T) == 2;
  static constexpr int kElems = kNarrow ? 8192 : 4096;
  static constexpr int kSlice = kElems / kCW;
  static constexpr int kVec = Elt<TDT>::kVec < Elt<DDT>::kVec ? Elt<TDT>::kVec : Elt<DDT>::kVec;
};

// U_NOOP units count toward their row (e.g. draft rows of a greedy row);
// U_SKIP units (rejected descriptors) count toward nothing.
enum UnitKind { U_STOP = 0, U_NOOP = 1, U_SOFTMAX = 2, U_ARGMAX = 3, U_RESID = 4, U_SKIP = 5 };
enum DecItem { D_CHAIN = 1, D_FINAL = 2, D_TREE = 3 };

struct StreamHeader {
  unsigned a_next;          // Phase-A claim counter
  unsigned q_head;          // Phase-B queue: tickets handed out
  unsigned q_reserved;      // Phase-B queue: slots reserved by publishers
  unsigned decisions_done;  // batch rows decided
  unsigned error;           // a bounded wait ran out somewhere
};

struct SParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const float *temps;
  const float *unif;
  const int32_t *parent;
  const int32_t *node_tokens;
  int B, gamma, V, N, max_depth, rows;
  int tilesT, tilesD, tilesMax, tilesB;  // tiles per target row / draft row / Phase-B pair
  int TA_T, TA_D, TB;                    // elements per tile
  int unitsA;                            // Phase-A units per batch row
  int totalA;
  int32_t *out_tokens, *out_nacc, *out_status, *out_path;
  float *out_diag;
  StreamHeader *hdr;
  unsigned *a_count, *b_count, *row_done, *qitems;
  Decision *dec;
  float2 *partA;   // [B][rows][tilesMax][kCW]  warp-slice partials
  float2 *partT;   // [B][rows][tilesMax]       tile partials
  float *partB;    // [B][tilesB][kCW]          residual mass per warp slice
  float *partBT;   // [B][tilesB]               residual mass per tile
};

// Unit descriptor.  `target` is the number of Phase-A units that complete
// the unit's batch row (units the scheduler does not emit are not counted).
struct StageMeta {
  int kind, b, row, tile, n, isdraft, j, target;
  float c, Mp, invZp, Mq, invZq, pad2[3];
};

struct alignas(16) StreamSmem {
  uint64_t full[kStages], empty[kStages];  // producer <-> consumers, per stage
  uint64_t pdone[kPR], pfree[kPR];         // consumers <-> bookkeeper, per partial slot
  StageMeta meta[kStages];
  StageMeta pmeta[kPR];
  float2 wpart[kPR][kCW];
  int dq[kDQ];
  volatile int dq_push, dq_pop, ctl_done, pad;
  StageMeta ring[kRing];
  volatile int ring_head, ring_tail, pad2[2];
  // decider scratch
  float rowM[kMaxRows], rowZ[kMaxRows];
  int rowI[kMaxRows];
  int a[SV_MAX_TREE_NODES], par[SV_MAX_TREE_NODES], tok[SV_MAX_TREE_NODES];
  int path[32];
};

constexpr size_t kStreamSmemBytes = sizeof(StreamSmem) + 128 + (size_t)kStages * kStageBytes;
static_assert(kStreamSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");

// ---------------------------------------------------------------------------
// mbarrier, bulk copy, fences
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false if it ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, long long t0) {
  while (true) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kStreamWait) return false;
  }
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Release/acquire fence at device scope (lighter than the sequentially
// consistent __threadfence()).
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// Relaxed (morally strong) device-scope store; after a release fence it
// publishes everything written before the fence.
__device__ __forceinline__ void st_relaxed_u32(unsigned *p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p) {
  return *reinterpret_cast<const volatile unsigned *>(p);
}

// Phase-B queue items pack (batch row, tile, rejected position j):
// ((b * tilesB + t) << 5 | j) + 1, so 0 marks a slot not yet written.
__device__ __forceinline__ unsigned pack_item(int b, int t, int tilesB, int j) {
  return ((unsigned)(b * tilesB + t) << 5 | (unsigned)j) + 1u;
}

// ---------------------------------------------------------------------------
// Consumer reductions over one warp slice of a stage.  Slice sizes are
// compile-time, so each lane's groups load and reduce fully unrolled with
// independent accumulators.
// ---------------------------------------------------------------------------

template <int DT, int VEC>
__device__ __forceinline__ void smem_group(const unsigned char *base, int g, float *o) {
  using E = Elt<DT>;
  constexpr int kB = VEC * (int)sizeof(typename E::T);
  if constexpr (kB == 16) {
    E::unpack(reinterpret_cast<const uint4 *>(base)[g], o);
  } else {
    E::unpack(reinterpret_cast<const uint2 *>(base)[g], o);
  }
}

// The lane's KG groups of VEC elements of warp slice `cw` (slice of SLICE
// elements), element x of group k is s0 + (lane + 32 k) * VEC + t.  Slots at
// or past n hold `pad`.
template <int DT, int VEC, int SLICE>
__device__ __forceinline__ void slice_load(const unsigned char *stage, int cw, int n, float pad,
                                           float (&v)[SLICE / 32]) {
  constexpr int KG = SLICE / (32 * VEC);
  const int s0 = cw * SLICE;
  const unsigned char *base = stage + (size_t)s0 * sizeof(typename Elt<DT>::T);
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < KG; ++k) smem_group<DT, VEC>(base, lane + 32 * k, &v[k * VEC]);
  if (s0 + SLICE > n) {
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int t = 0; t < VEC; ++t)
        if (s0 + (lane + 32 * k) * VEC + t >= n) v[k * VEC + t] = pad;
  }
}

// (m, s): m = slice max, s = sum exp2((v - m) c).  The exponent argument is
// one FFMA, v c - mc with mc = round(m c); that shifts every term of the
// slice by the same factor 2^d, d = m c - mc (computed exactly with an FMA),
// which is divided out once.  Overflowing m c falls back to (v - m) c.
template <int DT>
__device__ __forceinline__ float2 warp_softmax_slice(const unsigned char *stage, int n, int cw,
                                                     float c) {
  constexpr int VEC = Elt<DT>::kVec, SLICE = TileA<DT>::kSlice, PER = SLICE / 32;
  float v[PER];
  slice_load<DT, VEC, SLICE>(stage, cw, n, -CUDART_INF_F, v);
  float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
  for (int i = 0; i < PER; ++i) m4[i & 3] = max_nan(m4[i & 3], v[i]);
  const float m = warp_max_nan(max_nan(max_nan(m4[0], m4[1]), max_nan(m4[2], m4[3])));
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  float scale = 1.f;
  if (m != -CUDART_INF_F) {
    const float mc = m * c;
    if (fabsf(mc) <= 1.0e37f) {
      const float d = fmaf(m, c, -mc);
#pragma unroll
      for (int i = 0; i < PER; ++i) s4[i & 3] += ex2(fmaf(v[i], c, -mc));
      scale = ex2(-d);
    } else {
#pragma unroll
      for (int i = 0; i < PER; ++i) s4[i & 3] += ex2((v[i] - m) * c);
    }
  }
  return make_float2(m, warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3])) * scale);
}

template <int DT>
__device__ __forceinline__ float2 warp_argmax_slice(const unsigned char *stage, int n, int cw,
                                                    int x0) {
  constexpr int VEC = Elt<DT>::kVec, SLICE = TileA<DT>::kSlice, PER = SLICE / 32;
  float v[PER];
  slice_load<DT, VEC, SLICE>(stage, cw, n, -CUDART_INF_F, v);
  float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
  for (int i = 0; i < PER; ++i) m4[i & 3] = max_nan(m4[i & 3], v[i]);
  const float m = warp_max_nan(max_nan(max_nan(m4[0], m4[1]), max_nan(m4[2], m4[3])));
  const int s0 = cw * SLICE, lane = lane_id();
  int idx = 0x7fffffff;
#pragma unroll
  for (int i = PER - 1; i >= 0; --i) {
    const int e = s0 + (lane + 32 * (i / VEC)) * VEC + (i % VEC);
    if (e < n && v[i] == m) idx = e;  // descending scan keeps the lowest index
  }
  idx = warp_min_int(idx);
  return make_float2(m, __int_as_float(idx == 0x7fffffff ? idx : x0 + idx));
}

template <int TDT, int DDT, bool PROBS>
__device__ __forceinline__ float warp_resid_slice(const unsigned char *stage, int n, int cw,
                                                  const StageMeta &mt) {
  using TB = TileB<TDT, DDT>;
  constexpr int VEC = TB::kVec, SLICE = TB::kSlice, PER = SLICE / 32;
  float a[PER], q[PER];
  slice_load<TDT, VEC, SLICE>(stage, cw, n, -CUDART_INF_F, a);
  slice_load<DDT, VEC, SLICE>(stage + (size_t)TB::kElems * sizeof(typename Elt<TDT>::T), cw, n,
                              PROBS ? 0.f : -CUDART_INF_F, q);
  Decision d;
  d.c = mt.c; d.Mp = mt.Mp; d.invZp = mt.invZp; d.Mq = mt.Mq; d.invZq = mt.invZq;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < PER; ++i) s4[i & 3] += residual_term<PROBS>(a[i], q[i], d);
  return warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3]));
}

}  // namespace sv
