// Streaming verification kernel for sm_103a: one persistent CTA per SM with a
// shared-memory ring filled by TMA bulk copies.
//
// Warp roles of a CTA:
//   warp 0  producer    claims units (Phase-B queue first, then the next
//                       Phase-A unit from a device-wide counter) and issues
//                       cp.async.bulk copies of the unit's tile(s) into a
//                       ring stage, completing on the stage's full barrier;
//   warps 3..18 consumers  each reduces its 1/16 slice of a stage to a
//                       warp partial — softmax (max, sum exp2) / argmax
//                       (max, first index) / residual mass — with warp
//                       shuffles only, and arrives on the stage's done
//                       barrier;
//   warp 1  bookkeeper  copies the warp partials of finished stages to global
//                       memory, releases the stages, and counts each unit
//                       into its batch row (one fence per batch of stages);
//                       the unit that completes a row queues a decision;
//   warp 2  decider     merges a row's partials and makes its decision
//                       (accept tests + first-reject scan, greedy match, or
//                       the tree walk), draws the bonus token, or publishes
//                       the row's Phase-B tiles to a device-wide queue; after
//                       the last Phase-B tile of a row it finds the crossing
//                       tile and warp slice of u * R and rescans that slice.
//
// Rows must start on 16-byte boundaries (V * element size a multiple of 16
// and 16-byte aligned bases); other shapes use the register-tile kernel.
//
// Method references: "論文解説: Speculative Sampling — ドラフトモデルによる
// LLMデコード高速化" §技術的詳細 ステップ3 (accept test), §修正付き棄却サンプリング
// (residual), §期待される高速化 (gamma + 1 tokens: bonus draw);
// "投機的デコーディングとは？" §ドラフト生成と並列検証の仕組み (greedy);
// SpecInfer explainer §推論方法 (tree walk).
#pragma once

#include "sv_kernel.cuh"

namespace sv {

constexpr int kCW = 16;                            // consumer warps
constexpr int kStreamWarps = kCW + 3;
constexpr int kStreamThreads = kStreamWarps * 32;  // 608
constexpr int kStages = 6;
constexpr int kStageBytes = 32768;
constexpr int kDQ = 64;                            // decider queue entries
constexpr int kBookBatch = 4;                      // stages per bookkeeper fence
constexpr long long kStreamWait = 4000000000LL;    // bound of every wait, in clocks

enum UnitKind { U_STOP = 0, U_NOOP = 1, U_SOFTMAX = 2, U_ARGMAX = 3, U_RESID = 4 };
enum DecItem { D_CHAIN = 1, D_FINAL = 2, D_TREE = 3 };

struct StreamHeader {
  unsigned a_next;          // Phase-A claim counter
  unsigned q_head;          // Phase-B queue: next index to claim
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
  float2 *partA;  // [B][rows][tilesMax][kCW]
  float *partB;   // [B][tilesB][kCW]
};

struct StageMeta {
  int kind, b, row, tile, n, isdraft, j, pad;
  float c, Mp, invZp, Mq, invZq, pad2[3];
};

struct alignas(16) StreamSmem {
  uint64_t full[kStages], done[kStages], empty[kStages];
  StageMeta meta[kStages];
  float2 wpart[kStages][kCW];
  int dq[kDQ];
  volatile int dq_push, dq_pop, ctl_done, pad;
  // decider scratch
  float rowM[kMaxRows], rowZ[kMaxRows];
  int rowI[kMaxRows];
  int a[SV_MAX_TREE_NODES], par[SV_MAX_TREE_NODES], tok[SV_MAX_TREE_NODES];
  int path[32];
};

constexpr size_t kStreamSmemBytes = sizeof(StreamSmem) + 128 + (size_t)kStages * kStageBytes;
static_assert(kStreamSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy helpers
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
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
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

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Phase-B queue items pack (batch row, tile, rejected position j):
// ((b * tilesB + t) << 5 | j) + 1, so 0 marks a slot not yet written.
__device__ __forceinline__ unsigned pack_item(int b, int t, int tilesB, int j) {
  return ((unsigned)(b * tilesB + t) << 5 | (unsigned)j) + 1u;
}

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p) {
  return *reinterpret_cast<const volatile unsigned *>(p);
}

// ---------------------------------------------------------------------------
// Consumer reductions over one warp slice of a stage
// ---------------------------------------------------------------------------

// Elements of a group of VEC entries read from shared memory.
template <int DT, int VEC>
__device__ __forceinline__ void smem_group(const void *base, int g, float *o) {
  using E = Elt<DT>;
  constexpr int kB = VEC * (int)sizeof(typename E::T);
  if constexpr (kB == 16) {
    const uint4 r = reinterpret_cast<const uint4 *>(base)[g];
    E::unpack(r, o);
  } else {
    const uint2 r = reinterpret_cast<const uint2 *>(base)[g];
    E::unpack(r, o);
  }
}

// Warp slice geometry: the stage's n valid elements (of a tile of `tile`
// elements) are split in kCW slices of tile / kCW elements; lane l reads the
// VEC-element groups l, l + 32, ... of its warp's slice.
template <int DT, int VEC, class F>
__device__ __forceinline__ void slice_for_each(const void *stage, int tile, int n, int cw,
                                               float pad, F f) {
  const int E = tile / kCW;
  const int groups = E / VEC;
  const int s0 = cw * E;
  const int lane = lane_id();
  const char *base = reinterpret_cast<const char *>(stage) +
                     (size_t)s0 * sizeof(typename Elt<DT>::T);
  for (int g = lane; g < groups; g += 32) {
    const int x = s0 + g * VEC;
    float o[VEC];
    smem_group<DT, VEC>(base, g, o);
    if (x + VEC <= n) {
#pragma unroll
      for (int t = 0; t < VEC; ++t) f(o[t], x + t);
    } else {
#pragma unroll
      for (int t = 0; t < VEC; ++t) f(x + t < n ? o[t] : pad, x + t);
    }
  }
}

template <int DT>
__device__ __forceinline__ float2 warp_softmax_slice(const void *stage, int tile, int n, int cw,
                                                     float c) {
  constexpr int VEC = Elt<DT>::kVec;
  float m = -CUDART_INF_F;
  slice_for_each<DT, VEC>(stage, tile, n, cw, -CUDART_INF_F,
                          [&](float v, int) { m = max_nan(m, v); });
  m = warp_max_nan(m);
  float s = 0.f;
  if (m != -CUDART_INF_F) {
    slice_for_each<DT, VEC>(stage, tile, n, cw, -CUDART_INF_F,
                            [&](float v, int) { s += ex2((v - m) * c); });
  }
  return make_float2(m, warp_sum(s));
}

template <int DT>
__device__ __forceinline__ float2 warp_argmax_slice(const void *stage, int tile, int n, int cw,
                                                    int x0) {
  constexpr int VEC = Elt<DT>::kVec;
  float m = -CUDART_INF_F;
  slice_for_each<DT, VEC>(stage, tile, n, cw, -CUDART_INF_F,
                          [&](float v, int) { m = max_nan(m, v); });
  m = warp_max_nan(m);
  int idx = 0x7fffffff;
  slice_for_each<DT, VEC>(stage, tile, n, cw, -CUDART_INF_F, [&](float v, int e) {
    if (e < n && v == m && e < idx) idx = e;
  });
  idx = warp_min_int(idx);
  return make_float2(m, __int_as_float(idx == 0x7fffffff ? idx : x0 + idx));
}

template <int TDT, int DDT, bool PROBS>
__device__ __forceinline__ float warp_resid_slice(const void *stage, int tile, int n, int cw,
                                                  const StageMeta &mt) {
  constexpr int VEC = Elt<TDT>::kVec < Elt<DDT>::kVec ? Elt<TDT>::kVec : Elt<DDT>::kVec;
  const int E = tile / kCW;
  const int groups = E / VEC;
  const int s0 = cw * E;
  const char *pb = reinterpret_cast<const char *>(stage) +
                   (size_t)s0 * sizeof(typename Elt<TDT>::T);
  const char *qb = reinterpret_cast<const char *>(stage) +
                   (size_t)tile * sizeof(typename Elt<TDT>::T) +
                   (size_t)s0 * sizeof(typename Elt<DDT>::T);
  Decision d;
  d.c = mt.c; d.Mp = mt.Mp; d.invZp = mt.invZp; d.Mq = mt.Mq; d.invZq = mt.invZq;
  float s = 0.f;
  for (int g = lane_id(); g < groups; g += 32) {
    const int x = s0 + g * VEC;
    float a[VEC], q[VEC];
    smem_group<TDT, VEC>(pb, g, a);
    smem_group<DDT, VEC>(qb, g, q);
#pragma unroll
    for (int t = 0; t < VEC; ++t)
      if (x + t < n) s += residual_term<PROBS>(a[t], q[t], d);
  }
  return warp_sum(s);
}

// ---------------------------------------------------------------------------
// Decider helpers (one warp)
// ---------------------------------------------------------------------------

// First index i in [0, cnt) where the running sum of w(i) exceeds target;
// base receives the sum before it.  Falls back to the last i with w > 0.
template <class WF>
__device__ __forceinline__ int warp_prefix_cross(int cnt, float target, WF w, float &base) {
  const int lane = lane_id();
  float acc = 0.f, last_base = 0.f;
  int last_i = -1;
  for (int c0 = 0; c0 < cnt; c0 += 32) {
    const int i = c0 + lane;
    const float v = i < cnt ? w(i) : 0.f;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, acc + incl > target);
    const unsigned pos = __ballot_sync(0xffffffffu, v > 0.f);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const float excl = __shfl_sync(0xffffffffu, incl - v, l);
      base = acc + excl;
      return c0 + l;
    }
    if (pos) {
      const int l = 31 - __clz(pos);
      last_base = acc + __shfl_sync(0xffffffffu, incl - v, l);
      last_i = c0 + l;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  base = last_base;
  return last_i;
}

template <class WF>
__device__ __forceinline__ float warp_total(int cnt, WF w) {
  float s = 0.f;
  for (int i = lane_id(); i < cnt; i += 32) s += w(i);
  return warp_sum(s);
}

// Rescan of `n` consecutive elements with weights wf(e) (e local): lane l
// owns [l * per, (l + 1) * per).  Returns the local index of the crossing.
template <class WF>
__device__ __forceinline__ int warp_rescan(int n, float base, float target, WF wf) {
  const int lane = lane_id();
  const int per = (n + 31) / 32;
  const int e0 = lane * per;
  float tsum = 0.f;
  int lastpos = -1;
  for (int k = 0; k < per; ++k) {
    const int e = e0 + k;
    const float w = e < n ? wf(e) : 0.f;
    tsum += w;
    if (w > 0.f) lastpos = e;
  }
  float incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const float start = base + incl - tsum;
  const unsigned hit = __ballot_sync(0xffffffffu, start + tsum > target);
  const int last_any = warp_max_int(lastpos);
  if (!hit) return last_any < 0 ? 0 : last_any;
  const int l = __ffs(hit) - 1;
  int k = -1;
  if (lane == l) {
    float acc = start;
    for (int kk = 0; kk < per && k < 0; ++kk) {
      const int e = e0 + kk;
      const float w = e < n ? wf(e) : 0.f;
      acc += w;
      if (acc > target) k = e;
    }
    if (k < 0) k = lastpos >= 0 ? lastpos : e0;
  }
  return __shfl_sync(0xffffffffu, k, l);
}

// Draw from softmax row `row` (tiles of TA elements, partials [tiles][kCW]).
template <int DT>
__device__ int warp_sample_row(const typename Elt<DT>::T *row, const float2 *part, int tiles,
                               int TA, int V, float M, float c, float u) {
  const int cnt = tiles * kCW;
  auto w = [&](int i) {
    const float2 pt = __ldcg(part + i);
    return pt.x != -CUDART_INF_F ? pt.y * ex2((pt.x - M) * c) : 0.f;
  };
  const float R = warp_total(cnt, w);
  const float target = u * R;
  float base = 0.f;
  int i = warp_prefix_cross(cnt, target, w, base);
  if (i < 0) i = 0;
  const int E = TA / kCW;
  const int x0 = min((i / kCW) * TA + (i % kCW) * E, V - 1);
  const int n = min(E, V - x0);
  const typename Elt<DT>::T *sb = row + x0;
  return x0 + warp_rescan(n, base, target,
                          [&](int e) { return ex2((Elt<DT>::load1(sb + e) - M) * c); });
}

__device__ __forceinline__ float2 warp_merge_softmax_n(const float2 *part, int cnt, float c) {
  return warp_merge_softmax(part, cnt, c);
}

// ---------------------------------------------------------------------------
// Decisions (decider warp)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void warp_error_row(const SParams &P, int b, int status, int width,
                                               int32_t *tokens_base, int32_t *path_base) {
  for (int s = lane_id(); s < width; s += 32) {
    tokens_base[s] = -1;
    if (path_base) path_base[s] = -1;
  }
  if (lane_id() == 0) {
    P.out_nacc[b] = 0;
    if (P.out_status) P.out_status[b] = status;
  }
}

template <bool CHAIN, int TDT, int DDT, bool PROBS>
__device__ void stream_decide_chain(const SParams &P, int b, StreamSmem &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int g = P.gamma, G1 = g + 1, V = P.V;
  const int lane = lane_id();
  const float T = CHAIN ? __ldg(P.temps + b) : 0.f;
  const bool badT = bad_temperature(T);
  const bool greedy = T <= 0.f;
  const float c = kLog2e / T;
  const int nrows = greedy ? G1 : P.rows;
  const TT *tgt = reinterpret_cast<const TT *>(P.target) + (size_t)b * G1 * V;
  int32_t *ot = P.out_tokens + (size_t)b * G1;
  const float2 *pbase = P.partA + (size_t)b * P.rows * P.tilesMax * kCW;

  if (!badT) {
    for (int r = 0; r < nrows; ++r) {
      const int tiles = r < G1 ? P.tilesT : P.tilesD;
      const float2 *pp = pbase + (size_t)r * P.tilesMax * kCW;
      if (greedy) {
        const float2 mi = warp_merge_argmax(pp, tiles * kCW);
        if (lane == 0) { sm.rowM[r] = mi.x; sm.rowI[r] = __float_as_int(mi.y); }
      } else {
        const float2 mz = warp_merge_softmax(pp, tiles * kCW, c);
        if (lane == 0) { sm.rowM[r] = mz.x; sm.rowZ[r] = mz.y; }
      }
    }
  }
  __syncwarp();

  const int i = lane;
  const bool act = i < g;
  const int x = act ? __ldg(P.draft_tokens + (size_t)b * g + i) : 0;
  const bool tok_ok = x >= 0 && x < V;
  const unsigned gmask = (g >= 32) ? 0xffffffffu : ((1u << g) - 1u);
  int status = 0, j = g;
  if (badT) {
    status = SV_ROW_BAD_TEMPERATURE;
  } else if (greedy) {
    bool nf = false;
    for (int r = lane; r < G1; r += 32) nf |= isnan(sm.rowM[r]);
    const bool match = act && tok_ok && x == sm.rowI[i];
    const unsigned mm = __ballot_sync(0xffffffffu, match) & gmask;
    const unsigned badtok = __ballot_sync(0xffffffffu, act && !tok_ok);
    const unsigned nfm = __ballot_sync(0xffffffffu, nf);
    j = (~mm & gmask) ? __ffs(~mm & gmask) - 1 : g;
    status = (badtok ? SV_ROW_BAD_TOKEN : 0) | (nfm ? SV_ROW_NONFINITE : 0);
    if (CHAIN && act && P.out_diag)
      reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + i] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    float p = 0.f, q = 0.f;
    bool acc = false;
    if (act && tok_ok) {
      const float lp = Elt<TDT>::load1(tgt + (size_t)i * V + x);
      p = ex2((lp - sm.rowM[i]) * c) / sm.rowZ[i];
      if (PROBS) {
        q = __ldg(reinterpret_cast<const float *>(P.draft) + ((size_t)b * g + i) * V + x);
      } else {
        const DTy *drow = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + i) * V;
        q = ex2((Elt<DDT>::load1(drow + x) - sm.rowM[G1 + i]) * c) / sm.rowZ[G1 + i];
      }
      acc = __ldg(P.unif + (size_t)b * G1 + i) * q < p;
    }
    bool nf = false;
    for (int r = lane; r < nrows; r += 32) {
      const float Z = sm.rowZ[r];
      nf |= !(Z > 0.f && Z <= 3.0e38f);
    }
    if (PROBS) nf |= act && tok_ok && !isfinite(q);
    const unsigned am = __ballot_sync(0xffffffffu, acc) & gmask;
    const unsigned badtok = __ballot_sync(0xffffffffu, act && !tok_ok);
    const unsigned nfm = __ballot_sync(0xffffffffu, nf);
    j = (~am & gmask) ? __ffs(~am & gmask) - 1 : g;
    status = (badtok ? SV_ROW_BAD_TOKEN : 0) | (nfm ? SV_ROW_NONFINITE : 0);
    if (act && P.out_diag) {
      const float ap = (q > 0.f) ? fminf(1.f, p / q) : (p > 0.f ? 1.f : 0.f);
      reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + i] = make_float4(p, q, ap, 0.f);
    }
  }

  bool residual = false;
  if (status) {
    warp_error_row(P, b, status, G1, ot, nullptr);
  } else {
    for (int s = lane; s < G1; s += 32) {
      if (s < j) ot[s] = __ldg(P.draft_tokens + (size_t)b * g + s);
      else if (s > j) ot[s] = -1;
      else if (greedy) ot[s] = sm.rowI[j];
    }
    if (lane == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
    }
    if (!greedy) {
      if (j == g) {
        const float2 *pg = pbase + (size_t)g * P.tilesMax * kCW;
        const int k = warp_sample_row<TDT>(tgt + (size_t)g * V, pg, P.tilesT, P.TA_T, V,
                                           sm.rowM[g], c, __ldg(P.unif + (size_t)b * G1 + g));
        if (lane == 0) ot[g] = k;
      } else {
        residual = true;
      }
    }
  }
  __syncwarp();
  if (lane == 0) {
    if (residual) {
      Decision *d = P.dec + b;
      d->kind = DEC_RESIDUAL;
      d->j = j;
      d->c = c;
      d->Mp = sm.rowM[j];
      d->invZp = 1.f / sm.rowZ[j];
      d->Mq = PROBS ? 0.f : sm.rowM[G1 + j];
      d->invZq = PROBS ? 1.f : 1.f / sm.rowZ[G1 + j];
      d->u = __ldg(P.unif + (size_t)b * G1 + g);
      __threadfence();
      const unsigned base = atomicAdd(&P.hdr->q_reserved, (unsigned)P.tilesB);
      for (int t = 0; t < P.tilesB; ++t)
        st_release(P.qitems + base + t, pack_item(b, t, P.tilesB, j));
    } else {
      __threadfence();
      P.row_done[b] = 1;
    }
    __threadfence();
    atomicAdd(&P.hdr->decisions_done, 1u);
  }
  __syncwarp();
}

template <int TDT, int DDT, bool PROBS>
__device__ void stream_finalize(const SParams &P, int b) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int g = P.gamma, G1 = g + 1, V = P.V;
  const int lane = lane_id();
  const Decision *dp = P.dec + b;
  Decision d;
  d.j = __ldcg(&dp->j);
  d.c = __ldcg(&dp->c);
  d.Mp = __ldcg(&dp->Mp);
  d.invZp = __ldcg(&dp->invZp);
  d.Mq = __ldcg(&dp->Mq);
  d.invZq = __ldcg(&dp->invZq);
  d.u = __ldcg(&dp->u);
  const int j = d.j;
  const float *pb = P.partB + (size_t)b * P.tilesB * kCW;
  const int cnt = P.tilesB * kCW;
  auto w = [&](int i) { return __ldcg(pb + i); };
  // sequential order of the partials: tile-major, slice-minor
  float R = 0.f;
  {
    float acc = 0.f;
    for (int c0 = 0; c0 < cnt; c0 += 32) {
      const int i = c0 + lane;
      acc += warp_sum(i < cnt ? w(i) : 0.f);
    }
    R = acc;
  }
  const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)b * G1 + j) * V;
  int32_t *ot = P.out_tokens + (size_t)b * G1;
  if (isnan(R) || isinf(R)) {
    warp_error_row(P, b, SV_ROW_NONFINITE, G1, ot, nullptr);
  } else {
    int k;
    if (!(R > 0.f)) {
      const float2 *pp = P.partA + ((size_t)b * P.rows + j) * P.tilesMax * kCW;
      k = warp_sample_row<TDT>(prow, pp, P.tilesT, P.TA_T, V, d.Mp, d.c, d.u);
    } else {
      const float target = d.u * R;
      float base = 0.f;
      int i = warp_prefix_cross(cnt, target, w, base);
      if (i < 0) i = 0;
      const int E = P.TB / kCW;
      const int x0 = min((i / kCW) * P.TB + (i % kCW) * E, V - 1);
      const int n = min(E, V - x0);
      const TT *pt = prow + x0;
      const DTy *qt = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + j) * V + x0;
      k = x0 + warp_rescan(n, base, target, [&](int e) {
            return residual_term<PROBS>(Elt<TDT>::load1(pt + e), Elt<DDT>::load1(qt + e), d);
          });
    }
    if (lane == 0) {
      ot[j] = k;
      if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    P.row_done[b] = 1;
  }
}

template <int DT>
__device__ void stream_decide_tree(const SParams &P, int b, StreamSmem &sm) {
  const int N = P.N, V = P.V, D = P.max_depth;
  const int lane = lane_id();
  const float2 *part = P.partA + (size_t)b * P.rows * P.tilesMax * kCW;
  int flags = 0;
  for (int r = 0; r < N; ++r) {
    const float2 mi = warp_merge_argmax(part + (size_t)r * P.tilesMax * kCW, P.tilesT * kCW);
    if (lane == 0) {
      sm.a[r] = __float_as_int(mi.y);
      if (isnan(mi.x)) flags |= SV_ROW_NONFINITE;
    }
  }
  for (int n = lane; n < N; n += 32) {
    const int par = __ldg(P.parent + (size_t)b * N + n);
    const int tok = __ldg(P.node_tokens + (size_t)b * N + n);
    sm.par[n] = par;
    sm.tok[n] = tok;
    if (n == 0 ? par != -1 : (par < 0 || par >= n)) flags |= SV_ROW_BAD_TREE;
    if (n > 0 && (tok < 0 || tok >= V)) flags |= SV_ROW_BAD_TOKEN;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) flags |= __shfl_xor_sync(0xffffffffu, flags, o);
  __syncwarp();
  const int W = D + 1;
  int32_t *op = P.out_path + (size_t)b * W;
  int32_t *ot = P.out_tokens + (size_t)b * W;
  if (flags) {
    warp_error_row(P, b, flags, W, ot, op);
  } else {
    int cur = 0, d = 0;
    while (d < D) {
      const int a = sm.a[cur];
      int found = -1;
      for (int base = cur + 1; base < N && found < 0; base += 32) {
        const int cidx = base + lane;
        const bool m = cidx < N && sm.par[cidx] == cur && sm.tok[cidx] == a;
        const unsigned bm = __ballot_sync(0xffffffffu, m);
        if (bm) found = base + __ffs(bm) - 1;
      }
      if (found < 0) break;
      if (lane == 0) sm.path[d] = found;
      cur = found;
      ++d;
    }
    __syncwarp();
    if (lane < W) {
      op[lane] = lane < d ? sm.path[lane] : -1;
      ot[lane] = lane < d ? sm.tok[sm.path[lane]] : (lane == d ? sm.a[cur] : -1);
    }
    if (lane == 0) {
      P.out_nacc[b] = d;
      if (P.out_status) P.out_status[b] = 0;
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    P.row_done[b] = 1;
    atomicAdd(&P.hdr->decisions_done, 1u);
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Producer (one thread).  Phase-A claims run two deep and the temperature of
// the next claimed row and the queue counters are loaded one iteration
// ahead, so the thread rarely waits on global memory while stages are free.
template <int MODE, int TDT, int DDT, bool PROBS>
__device__ void stream_producer(const SParams &P, StreamSmem &sm, unsigned char *stages) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int G1 = P.gamma + 1;
  const unsigned totalA = (unsigned)P.totalA;
  unsigned c0 = atomicAdd(&P.hdr->a_next, 1u);
  unsigned c1 = atomicAdd(&P.hdr->a_next, 1u);
  float T0 = 0.f;
  if (MODE == MODE_CHAIN && c0 < totalA) T0 = __ldg(P.temps + c0 / (unsigned)P.unitsA);
  unsigned qh = 0, qr = 0;
  int last_data_stage = -1;
  unsigned last_data_phase = 0;
  bool timed_out = false;
  for (int it = 0;; ++it) {
    const int s = it % kStages;
    const unsigned ph = (unsigned)(it / kStages) & 1u;
    if (it >= kStages && !mbar_wait(&sm.empty[s], ph ^ 1u, clock64())) timed_out = true;
    StageMeta &mt = sm.meta[s];
    unsigned char *dst = stages + (size_t)s * kStageBytes;
    int kind = U_STOP;
    const long long t0 = clock64();
    while (!timed_out) {
      if constexpr (MODE == MODE_CHAIN) {
        // Phase-B tiles first: they are L2-hot and unblock finalisation.
        if (qh < qr) {
          const unsigned h = qh;
          qh = qr;
          if (atomicCAS(&P.hdr->q_head, h, h + 1) == h) {
            unsigned w = ld_acquire(P.qitems + h);
            const long long tw = clock64();
            while (w == 0 && clock64() - tw < kStreamWait) w = ld_acquire(P.qitems + h);
            if (w == 0) { timed_out = true; break; }
            const unsigned v = w - 1u;
            const int j = (int)(v & 31u), bt = (int)(v >> 5);
            const int bb = bt / P.tilesB, tt = bt % P.tilesB;
            const int x0 = tt * P.TB;
            const int n = min(P.TB, P.V - x0);
            const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)bb * G1 + j) * P.V + x0;
            const DTy *qrow = reinterpret_cast<const DTy *>(P.draft) +
                              ((size_t)bb * P.gamma + j) * P.V + x0;
            const unsigned pbytes = (unsigned)(n * sizeof(TT));
            const unsigned qbytes = (unsigned)(n * sizeof(DTy));
            mbar_expect_tx(&sm.full[s], pbytes + qbytes);
            bulk_g2s(dst, prow, pbytes, &sm.full[s]);
            bulk_g2s(dst + (size_t)P.TB * sizeof(TT), qrow, qbytes, &sm.full[s]);
            const Decision *d = P.dec + bb;
            mt.c = __ldcg(&d->c);
            mt.Mp = __ldcg(&d->Mp);
            mt.invZp = __ldcg(&d->invZp);
            mt.Mq = __ldcg(&d->Mq);
            mt.invZq = __ldcg(&d->invZq);
            mt.j = j;
            mt.b = bb;
            mt.row = 0;
            mt.tile = tt;
            mt.isdraft = 0;
            mt.n = n;
            kind = U_RESID;
            last_data_stage = s;
            last_data_phase = ph;
            break;
          }
        }
      }
      if (c0 < totalA) {
        const int ua = (int)c0;
        const float T = T0;
        c0 = c1;
        c1 = atomicAdd(&P.hdr->a_next, 1u);
        if (MODE == MODE_CHAIN && c0 < totalA) T0 = __ldg(P.temps + c0 / (unsigned)P.unitsA);
        const int bb = ua / P.unitsA, ri = ua % P.unitsA;
        int row, tile, isdraft = 0;
        if (MODE != MODE_CHAIN || ri < G1 * P.tilesT) {
          row = ri / P.tilesT;
          tile = ri % P.tilesT;
        } else {
          const int rd = ri - G1 * P.tilesT;
          row = G1 + rd / P.tilesD;
          tile = rd % P.tilesD;
          isdraft = 1;
        }
        kind = U_ARGMAX;
        float c = 0.f;
        if constexpr (MODE == MODE_CHAIN) {
          if (bad_temperature(T) || (isdraft && T <= 0.f)) kind = U_NOOP;
          else if (T > 0.f) { kind = U_SOFTMAX; c = kLog2e / T; }
        }
        mt.b = bb;
        mt.row = row;
        mt.tile = tile;
        mt.isdraft = isdraft;
        mt.c = c;
        if (kind != U_NOOP) {
          const int TA = isdraft ? P.TA_D : P.TA_T;
          const int x0 = tile * TA;
          const int n = min(TA, P.V - x0);
          mt.n = n;
          const char *src;
          unsigned bytes;
          if (isdraft) {
            src = reinterpret_cast<const char *>(reinterpret_cast<const DTy *>(P.draft) +
                                                 ((size_t)bb * P.gamma + (row - G1)) * P.V + x0);
            bytes = (unsigned)(n * sizeof(DTy));
          } else {
            const int rows_per = (MODE == MODE_TREE) ? P.N : G1;
            src = reinterpret_cast<const char *>(reinterpret_cast<const TT *>(P.target) +
                                                 ((size_t)bb * rows_per + row) * P.V + x0);
            bytes = (unsigned)(n * sizeof(TT));
          }
          mbar_expect_tx(&sm.full[s], bytes);
          bulk_g2s(dst, src, bytes, &sm.full[s]);
          last_data_stage = s;
          last_data_phase = ph;
        }
        break;
      }
      // Phase A exhausted.
      if (MODE != MODE_CHAIN) break;
      const unsigned dd = ld_acquire(&P.hdr->decisions_done);
      qh = ld_volatile_u32(&P.hdr->q_head);
      qr = ld_volatile_u32(&P.hdr->q_reserved);
      if (qh < qr) continue;
      if (dd >= (unsigned)P.B) break;   // every decision made, every tile claimed
      __nanosleep(256);
      if (clock64() - t0 > kStreamWait) { timed_out = true; break; }
    }
    if (timed_out) kind = U_STOP;
    mt.kind = kind;
    mbar_arrive(&sm.full[s]);
    if (kind == U_STOP) break;
    if constexpr (MODE == MODE_CHAIN) {
      // counters for the next iteration's claim (loads in flight meanwhile)
      qh = ld_volatile_u32(&P.hdr->q_head);
      qr = ld_volatile_u32(&P.hdr->q_reserved);
    }
  }
  if (timed_out) {
    atomicOr(&P.hdr->error, 1u);
    // let the copies still in flight land before the CTA can exit
    if (last_data_stage >= 0) mbar_wait(&sm.full[last_data_stage], last_data_phase, clock64());
    for (int b = 0; b < P.B; ++b)
      if (ld_volatile_u32(P.row_done + b) == 0 && P.out_status) P.out_status[b] = SV_ROW_TIMEOUT;
  }
}

template <int MODE, int TDT, int DDT, bool PROBS>
__global__ void __launch_bounds__(kStreamThreads, 1) sv_stream_kernel(const SParams P) {
  extern __shared__ unsigned char smem_raw[];
  StreamSmem &sm = *reinterpret_cast<StreamSmem *>(smem_raw);
  unsigned char *stages = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(StreamSmem) + 127) & ~uintptr_t(127));
  const int warp = warp_id(), lane = lane_id();
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.done[s], kCW);
      mbar_init(&sm.empty[s], 1);
    }
    sm.dq_push = 0;
    sm.dq_pop = 0;
    sm.ctl_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) stream_producer<MODE, TDT, DDT, PROBS>(P, sm, stages);
    return;
  }

  if (warp >= 3) {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 3;
    for (int it = 0;; ++it) {
      const int s = it % kStages;
      const unsigned ph = (unsigned)(it / kStages) & 1u;
      if (!mbar_wait(&sm.full[s], ph, clock64())) {
        if (lane == 0) atomicOr(&P.hdr->error, 1u);
        return;
      }
      const StageMeta mt = sm.meta[s];
      if (mt.kind == U_STOP) {
        if (lane == 0) mbar_arrive(&sm.done[s]);
        break;
      }
      const void *st = stages + (size_t)s * kStageBytes;
      float2 part = make_float2(0.f, 0.f);
      if (mt.kind == U_SOFTMAX) {
        part = mt.isdraft ? warp_softmax_slice<DDT>(st, P.TA_D, mt.n, cw, mt.c)
                          : warp_softmax_slice<TDT>(st, P.TA_T, mt.n, cw, mt.c);
      } else if (mt.kind == U_ARGMAX) {
        part = warp_argmax_slice<TDT>(st, P.TA_T, mt.n, cw, mt.tile * P.TA_T);
      } else if (mt.kind == U_RESID) {
        if constexpr (MODE == MODE_CHAIN)
          part.x = warp_resid_slice<TDT, DDT, PROBS>(st, P.TB, mt.n, cw, mt);
      }
      if (lane == 0) {
        sm.wpart[s][cw] = part;
        mbar_arrive(&sm.done[s]);
      }
      __syncwarp();
    }
    return;
  }

  if (warp == 1) {
    // ------------------------------------------------------------ bookkeeper
    bool stop = false;
    for (int it = 0; !stop;) {
      const int s0 = it % kStages;
      if (!mbar_wait(&sm.done[s0], (unsigned)(it / kStages) & 1u, clock64())) {
        if (lane == 0) atomicOr(&P.hdr->error, 1u);
        break;
      }
      int nb = 1;
      while (nb < kBookBatch &&
             mbar_test(&sm.done[(it + nb) % kStages], (unsigned)((it + nb) / kStages) & 1u))
        ++nb;
      unsigned *cnt[kBookBatch];
      unsigned target[kBookBatch];
      int item[kBookBatch], bsel[kBookBatch];
      int used = 0;
      for (int k = 0; k < nb; ++k) {
        const int s = (it + k) % kStages;
        const StageMeta &mt = sm.meta[s];
        if (mt.kind == U_STOP) { stop = true; break; }
        if (mt.kind == U_SOFTMAX || mt.kind == U_ARGMAX) {
          if (lane < kCW)
            P.partA[(((size_t)mt.b * P.rows + mt.row) * P.tilesMax + mt.tile) * kCW + lane] =
                sm.wpart[s][lane];
        } else if (mt.kind == U_RESID) {
          if (lane < kCW)
            P.partB[((size_t)mt.b * P.tilesB + mt.tile) * kCW + lane] = sm.wpart[s][lane].x;
        }
        if (mt.kind == U_RESID) {
          cnt[used] = P.b_count + mt.b;
          target[used] = (unsigned)P.tilesB;
          item[used] = D_FINAL;
        } else {
          cnt[used] = P.a_count + mt.b;
          target[used] = (unsigned)P.unitsA;
          item[used] = (MODE == MODE_TREE) ? D_TREE : D_CHAIN;
        }
        bsel[used] = mt.b;
        ++used;
      }
      __syncwarp();
      if (lane == 0) {
        for (int k = 0; k < used; ++k) mbar_arrive(&sm.empty[(it + k) % kStages]);
        __threadfence();
        unsigned prev[kBookBatch];
        for (int k = 0; k < used; ++k) prev[k] = atomicAdd(cnt[k], 1u);
        bool any_last = false;
        for (int k = 0; k < used; ++k) any_last |= (prev[k] == target[k] - 1);
        if (any_last) __threadfence();  // acquire side: other CTAs' partials are visible
        for (int k = 0; k < used; ++k) {
          if (prev[k] == target[k] - 1) {
            const long long tq = clock64();
            while (sm.dq_push - sm.dq_pop >= kDQ && clock64() - tq < kStreamWait) __nanosleep(64);
            sm.dq[sm.dq_push % kDQ] = (item[k] << 28) | bsel[k];
            __threadfence_block();
            sm.dq_push = sm.dq_push + 1;
          }
        }
      }
      __syncwarp();
      it += used;
      if (stop) {
        // the STOP stage needs no release: the producer has finished
        break;
      }
    }
    if (lane == 0) {
      __threadfence_block();
      sm.ctl_done = 1;
    }
    return;
  }

  // -------------------------------------------------------------- decider
  {
    const long long t0 = clock64();
    while (true) {
      int item = 0, have = 0, fin = 0;
      if (lane == 0) {
        if (sm.dq_pop != sm.dq_push) {
          item = reinterpret_cast<volatile int *>(sm.dq)[sm.dq_pop % kDQ];
          have = 1;
        } else if (sm.ctl_done) {
          fin = (sm.dq_pop == sm.dq_push);
        }
      }
      have = __shfl_sync(0xffffffffu, have, 0);
      fin = __shfl_sync(0xffffffffu, fin, 0);
      item = __shfl_sync(0xffffffffu, item, 0);
      if (have) {
        __threadfence();
        const int kind = item >> 28, b = item & 0x0fffffff;
        if constexpr (MODE == MODE_TREE) {
          stream_decide_tree<TDT>(P, b, sm);
        } else if constexpr (MODE == MODE_CHAIN_GREEDY) {
          stream_decide_chain<false, TDT, DDT, false>(P, b, sm);
        } else {
          if (kind == D_FINAL) stream_finalize<TDT, DDT, PROBS>(P, b);
          else stream_decide_chain<true, TDT, DDT, PROBS>(P, b, sm);
        }
        __syncwarp();
        if (lane == 0) sm.dq_pop = sm.dq_pop + 1;
        continue;
      }
      if (fin) break;
      __nanosleep(128);
      if (clock64() - t0 > 4 * kStreamWait) {
        if (lane == 0) atomicOr(&P.hdr->error, 1u);
        break;
      }
    }
  }
}

// Workspace layout of the streaming kernel; the control block [0, ctrl) is
// zeroed by every call.
struct StreamLayout {
  size_t a_count, b_count, row_done, qitems, ctrl, dec, partA, partB, total;
  int tilesT, tilesD, tilesMax, tilesB, TA_T, TA_D, TB;
};

inline StreamLayout make_stream_layout(int B, int rows, int V, int esT, int esD, bool probs) {
  StreamLayout L;
  L.TA_T = kStageBytes / esT;
  L.TA_D = kStageBytes / esD;
  L.TB = (esT == 2 && esD == 2) ? 8192 : 4096;
  L.tilesT = (V + L.TA_T - 1) / L.TA_T;
  L.tilesD = probs ? 0 : (V + L.TA_D - 1) / L.TA_D;
  L.tilesMax = L.tilesT > L.tilesD ? L.tilesT : L.tilesD;
  L.tilesB = (V + L.TB - 1) / L.TB;
  size_t off = 256;  // StreamHeader
  L.a_count = off;  off = align_up(off + (size_t)B * 4, 256);
  L.b_count = off;  off = align_up(off + (size_t)B * 4, 256);
  L.row_done = off; off = align_up(off + (size_t)B * 4, 256);
  L.qitems = off;   off = align_up(off + (size_t)B * L.tilesB * 4, 256);
  L.ctrl = off;
  L.dec = off;      off = align_up(off + (size_t)B * sizeof(Decision), 256);
  L.partA = off;    off = align_up(off + (size_t)B * rows * L.tilesMax * kCW * sizeof(float2), 256);
  L.partB = off;    off = align_up(off + (size_t)B * L.tilesB * kCW * sizeof(float), 256);
  L.total = off;
  return L;
}

}  // namespace sv
