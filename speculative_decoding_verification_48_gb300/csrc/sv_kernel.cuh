// Verification kernels for sm_103a.
//
// One persistent kernel template serves the three entry points.  CTAs pull
// "units" from a device-wide counter in schedule order:
//
//   Phase A unit  (row, tile): streams kTile logits of one row once and
//                 writes a partial — (tile max, sum of exp2((l - max) c)) for
//                 a softmax row, (max value, first index) for an argmax row.
//                 The CTA that completes the last Phase-A unit of a batch
//                 row (arrival counter) merges the partials and makes the
//                 row's decision: accept tests + first-reject scan (chain),
//                 greedy match (chain greedy) or the tree walk (tree).
//   Phase B unit  (tile): for a chain row rejected at position j, the tile
//                 sum of the residual max(0, p_j - q_j).  The CTA that
//                 completes the last Phase-B unit finds the crossing tile of
//                 u * R from the tile sums and rescans that tile only.
//
// The bonus draw (all drafts accepted) needs no extra sweep: the Phase-A
// partials of row gamma already give the tile masses of p_gamma.
//
// Method references: "論文解説: Speculative Sampling — ドラフトモデルによる
// LLMデコード高速化" §技術的詳細 ステップ3 (accept test) and
// §修正付き棄却サンプリング (residual); "投機的デコーディングとは？" §ドラフト生成と
// 並列検証の仕組み (greedy); SpecInfer explainer §推論方法 (tree walk).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <type_traits>

#include "sv_internal.h"

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTinyT = 1e-20f;
// Bound of the Phase-B wait for a row decision, in SM clock cycles (about
// one second at 2 GHz).
constexpr long long kWaitCycles = 2000000000LL;

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either input is NaN
__device__ __forceinline__ float max_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// 16-byte streaming load: read-only path, no L1 allocation, 256-byte L2
// prefetch of the surrounding sector group.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
      : "=r"(r.x), "=r"(r.y)
      : "l"(p));
  return r;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a flag that another CTA sets: its value, or 0 once
// kWaitCycles clock cycles (about a second) have passed without it.
__device__ __forceinline__ unsigned wait_flag_bounded(const unsigned *flag) {
  unsigned f = ld_acquire(flag);
  if (!f) {
    const long long t0 = clock64();
    while (!f) {
      __nanosleep(200);
      f = ld_acquire(flag);
      if (!f && clock64() - t0 > kWaitCycles) break;
    }
  }
  return f;
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------

template <int DT> struct Elt;

template <> struct Elt<SV_F32> {
  using T = float;
  static constexpr int kVec = 4;
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    o[0] = __uint_as_float(r.x); o[1] = __uint_as_float(r.y);
    o[2] = __uint_as_float(r.z); o[3] = __uint_as_float(r.w);
  }
  __device__ static __forceinline__ float load1(const T *p) { return __ldg(p); }
};

template <> struct Elt<SV_BF16> {
  using T = __nv_bfloat16;
  static constexpr int kVec = 8;
  // bf16 -> f32 is a 16-bit left shift of the bit pattern (exact).
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ void unpack(const uint2 &r, float *o) {
    o[0] = __uint_as_float(r.x << 16); o[1] = __uint_as_float(r.x & 0xffff0000u);
    o[2] = __uint_as_float(r.y << 16); o[3] = __uint_as_float(r.y & 0xffff0000u);
  }
  __device__ static __forceinline__ float load1(const T *p) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __uint_as_float(static_cast<unsigned>(b) << 16);
  }
};

template <> struct Elt<SV_F16> {
  using T = __half;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 f = __half22float2(h);
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ void unpack(const uint2 &r, float *o) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  }
  __device__ static __forceinline__ float load1(const T *p) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __half2float(__ushort_as_half(b));
  }
};

// One tile of one row held by the CTA in registers.  Thread `tid` owns the
// VEC-element vectors k * kThreads + tid (k < kLoads), so each warp-wide load
// covers 32 consecutive vectors.  VEC defaults to 16 bytes of the dtype;
// a row pair of different dtypes uses the smaller width so both rows map
// element x to the same thread and slot.  Vectors not fully inside the row,
// and rows not aligned to the vector size, use scalar loads.
template <int DT, int VEC = Elt<DT>::kVec> struct Tile {
  using E = Elt<DT>;
  using T = typename E::T;
  static constexpr int kBytes = VEC * (int)sizeof(T);
  static_assert(kBytes == 16 || kBytes == 8, "vector loads are 8 or 16 bytes");
  using Raw = typename std::conditional<kBytes == 16, uint4, uint2>::type;
  static constexpr int kLoads = kPer / VEC;
  Raw raw[kLoads];
  const T *base;
  int n;
  bool aligned;

  __device__ __forceinline__ void load(const T *row, int x0, int n_) {
    base = row + x0;
    n = n_;
    aligned = (reinterpret_cast<uintptr_t>(base) & (kBytes - 1)) == 0;
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const int e = (k * kThreads + threadIdx.x) * VEC;
      if (aligned && e + VEC <= n) {
        if constexpr (kBytes == 16) raw[k] = ld_stream16(base + e);
        else raw[k] = ld_stream8(base + e);
      }
    }
  }

  // Values of vector k (slots past the row end get `pad`); returns the local
  // index of its first element.
  __device__ __forceinline__ int get(int k, float *o, float pad) const {
    const int e = (k * kThreads + threadIdx.x) * VEC;
    if (aligned && e + VEC <= n) {
      E::unpack(raw[k], o);
    } else {
#pragma unroll
      for (int t = 0; t < VEC; ++t) o[t] = (e + t < n) ? E::load1(base + e + t) : pad;
    }
    return e;
  }

  // f(value, local index) over the thread's elements in ascending order.
  template <class F> __device__ __forceinline__ void for_each(float pad, F f) const {
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      float o[VEC];
      const int e = get(k, o, pad);
#pragma unroll
      for (int t = 0; t < VEC; ++t) f(o[t], e + t);
    }
  }
};

// ---------------------------------------------------------------------------
// Shared memory
// ---------------------------------------------------------------------------

struct SmemBase {
  float redf[kWarps];
  int redi[kWarps];
  unsigned unit[2];
  int flag, flag2, j, status, ts, k;
  float base, target, R;
  Decision dec;
};

struct SmemChain : SmemBase {
  float rowM[kMaxRows];
  float rowZ[kMaxRows];
  int rowI[kMaxRows];
};

struct SmemTree : SmemBase {
  int a[SV_MAX_TREE_NODES];
  int par[SV_MAX_TREE_NODES];
  int tok[SV_MAX_TREE_NODES];
  int path[32];
};

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reductions; every thread gets the result.
__device__ __forceinline__ float block_max_nan(float v, SmemBase &sm) {
  v = warp_max_nan(v);
  if (lane_id() == 0) sm.redf[warp_id()] = v;
  __syncthreads();
  float r = sm.redf[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max_nan(r, sm.redf[w]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum(float v, SmemBase &sm) {
  v = warp_sum(v);
  if (lane_id() == 0) sm.redf[warp_id()] = v;
  __syncthreads();
  float r = sm.redf[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r += sm.redf[w];
  __syncthreads();
  return r;
}
__device__ __forceinline__ int block_min_int(int v, SmemBase &sm) {
  v = warp_min_int(v);
  if (lane_id() == 0) sm.redi[warp_id()] = v;
  __syncthreads();
  int r = sm.redi[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, sm.redi[w]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ int block_max_int(int v, SmemBase &sm) {
  v = warp_max_int(v);
  if (lane_id() == 0) sm.redi[warp_id()] = v;
  __syncthreads();
  int r = sm.redi[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max(r, sm.redi[w]);
  __syncthreads();
  return r;
}
// Exclusive prefix sum over threads in thread order.
__device__ __forceinline__ float block_excl_scan(float v, SmemBase &sm) {
  const int lane = lane_id(), warp = warp_id();
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) sm.redf[warp] = incl;
  __syncthreads();
  float off = 0.f;
  for (int w = 0; w < warp; ++w) off += sm.redf[w];
  __syncthreads();
  return off + excl;
}

// ---------------------------------------------------------------------------
// Phase A: per-tile partials
// ---------------------------------------------------------------------------

// (m, s): m = max logit of the tile, s = sum_x exp2((l(x) - m) * c).
// NaN anywhere makes both NaN; a +inf makes s NaN.
template <int DT>
__device__ __forceinline__ float2 tile_softmax(const typename Elt<DT>::T *row, int x0, int n,
                                               float c, SmemBase &sm) {
  Tile<DT> tile;
  tile.load(row, x0, n);
  float m = -CUDART_INF_F;
  tile.for_each(-CUDART_INF_F, [&](float v, int) { m = max_nan(m, v); });
  m = block_max_nan(m, sm);
  float s = 0.f;
  if (m != -CUDART_INF_F) {
    tile.for_each(-CUDART_INF_F, [&](float v, int) { s += ex2((v - m) * c); });
  }
  s = block_sum(s, sm);
  return make_float2(m, s);
}

// (max value, first local index of it); NaN anywhere makes the value NaN.
template <int DT>
__device__ __forceinline__ float2 tile_argmax(const typename Elt<DT>::T *row, int x0, int n,
                                              SmemBase &sm) {
  Tile<DT> tile;
  tile.load(row, x0, n);
  float m = -CUDART_INF_F;
  tile.for_each(-CUDART_INF_F, [&](float v, int) { m = max_nan(m, v); });
  m = block_max_nan(m, sm);
  int idx = 0x7fffffff;
  tile.for_each(-CUDART_INF_F, [&](float v, int e) {
    if (idx == 0x7fffffff && e < n && v == m) idx = e;
  });
  idx = block_min_int(idx, sm);
  return make_float2(m, __int_as_float(idx == 0x7fffffff ? idx : x0 + idx));
}

// max(0, p(x) - q(x)) from the logits (or the given probability q).  Both
// products are rounded separately (no FMA contraction), so identical target
// and draft rows give exactly zero.
template <bool PROBS>
__device__ __forceinline__ float residual_term(float lp, float lq, const Decision &d) {
  const float p = __fmul_rn(ex2(__fmul_rn(lp - d.Mp, d.c)), d.invZp);
  const float q = PROBS ? lq : __fmul_rn(ex2(__fmul_rn(lq - d.Mq, d.c)), d.invZq);
  return max_nan(0.f, __fsub_rn(p, q));
}

// Residual tile mass sum_x max(0, p(x) - q(x)) over one tile of the row
// pair (p_j, q_j); NaN propagates.
template <int TDT, int DDT, bool PROBS>
__device__ __forceinline__ float tile_residual(const typename Elt<TDT>::T *prow,
                                               const typename Elt<DDT>::T *qrow, int x0, int n,
                                               const Decision &d, SmemBase &sm) {
  constexpr int VEC = Elt<TDT>::kVec < Elt<DDT>::kVec ? Elt<TDT>::kVec : Elt<DDT>::kVec;
  Tile<TDT, VEC> tp;
  Tile<DDT, VEC> tq;
  tp.load(prow, x0, n);
  tq.load(qrow, x0, n);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < Tile<TDT, VEC>::kLoads; ++k) {
    float a[VEC], b[VEC];
    tp.get(k, a, -CUDART_INF_F);
    tq.get(k, b, PROBS ? 0.f : -CUDART_INF_F);
#pragma unroll
    for (int t = 0; t < VEC; ++t) s += residual_term<PROBS>(a[t], b[t], d);
  }
  return block_sum(s, sm);
}

// ---------------------------------------------------------------------------
// Inverse-CDF crossing inside one tile
// ---------------------------------------------------------------------------

// Local index k in [0, n) of the first element where base + cumsum(w) >
// target; thread i owns the contiguous elements [32 i, 32 i + 32).  If no
// element crosses (rounding), the last element with w > 0 is returned.  The
// crossing thread recomputes its 32 weights rather than keeping them.
template <class WF>
__device__ __forceinline__ int crossing_scan(int n, float base, float target, WF wf,
                                             SmemBase &sm) {
  const int e0 = threadIdx.x * kPer;
  float tsum = 0.f;
  int lastpos = -1;
#pragma unroll 8
  for (int k = 0; k < kPer; ++k) {
    const int e = e0 + k;
    const float w = (e < n) ? wf(e) : 0.f;
    tsum += w;
    if (w > 0.f) lastpos = e;
  }
  const float start = base + block_excl_scan(tsum, sm);
  const bool cross = start + tsum > target;
  const int first = block_min_int(cross ? (int)threadIdx.x : 0x7fffffff, sm);
  const int last_any = block_max_int(lastpos, sm);
  if (first == 0x7fffffff) return last_any < 0 ? 0 : last_any;
  if ((int)threadIdx.x == first) {
    float acc = start;
    int k = -1;
    for (int kk = 0; kk < kPer && k < 0; ++kk) {
      const int e = e0 + kk;
      const float w = (e < n) ? wf(e) : 0.f;
      acc += w;
      if (acc > target) k = e;
    }
    sm.k = (k >= 0) ? k : (lastpos >= 0 ? lastpos : e0);
  }
  __syncthreads();
  const int k = sm.k;
  __syncthreads();
  return k;
}

// Categorical draw from softmax row `row` using its Phase-A partials:
// tile masses w_t = s_t * exp2((m_t - M) c) in tile order, the crossing tile
// of u * sum_t w_t, then a rescan of that tile.  Returns a vocabulary index.
template <int DT>
__device__ int sample_row_from_partials(const typename Elt<DT>::T *row, const float2 *part,
                                        int tiles, int V, float M, float c, float u,
                                        SmemBase &sm) {
  if (threadIdx.x == 0) {
    float R = 0.f;
    for (int t = 0; t < tiles; ++t) {
      const float2 pt = __ldcg(part + t);
      if (pt.x != -CUDART_INF_F) R += pt.y * ex2((pt.x - M) * c);
    }
    const float target = u * R;
    float acc = 0.f, base = 0.f, last_base = 0.f;
    int ts = -1, last_t = -1;
    for (int t = 0; t < tiles; ++t) {
      const float2 pt = __ldcg(part + t);
      const float w = (pt.x != -CUDART_INF_F) ? pt.y * ex2((pt.x - M) * c) : 0.f;
      if (w > 0.f) { last_t = t; last_base = acc; }
      if (acc + w > target) { ts = t; base = acc; break; }
      acc += w;
    }
    if (ts < 0) { ts = last_t; base = last_base; }
    sm.ts = ts; sm.base = base; sm.target = target;
  }
  __syncthreads();
  const int ts = sm.ts < 0 ? 0 : sm.ts;
  const float base = sm.base, target = sm.target;
  __syncthreads();
  const int x0 = ts * kTile, n = min(kTile, V - x0);
  const typename Elt<DT>::T *tb = row + x0;
  const int k = crossing_scan(n, base, target,
                              [&](int e) { return ex2((Elt<DT>::load1(tb + e) - M) * c); }, sm);
  return x0 + k;
}

// ---------------------------------------------------------------------------
// Row merges (one warp per row)
// ---------------------------------------------------------------------------

// Softmax row: M = max_t m_t, Z = sum_t s_t exp2((m_t - M) c).
__device__ __forceinline__ float2 warp_merge_softmax(const float2 *part, int tiles, float c) {
  float M = -CUDART_INF_F;
  for (int t = lane_id(); t < tiles; t += 32) M = max_nan(M, __ldcg(part + t).x);
  M = warp_max_nan(M);
  float Z = 0.f;
  for (int t = lane_id(); t < tiles; t += 32) {
    const float2 pt = __ldcg(part + t);
    if (pt.x != -CUDART_INF_F) Z += pt.y * ex2((pt.x - M) * c);
    else Z += pt.y;  // 0, or NaN from a NaN tile
  }
  return make_float2(M, warp_sum(Z));
}

// Argmax row: (max value, lowest index attaining it).  NaN value if any
// tile held a NaN.
__device__ __forceinline__ float2 warp_merge_argmax(const float2 *part, int tiles) {
  float best = -CUDART_INF_F;
  for (int t = lane_id(); t < tiles; t += 32) best = max_nan(best, __ldcg(part + t).x);
  best = warp_max_nan(best);
  int idx = 0x7fffffff;
  for (int t = lane_id(); t < tiles; t += 32) {
    const float2 pt = __ldcg(part + t);
    if (pt.x == best) idx = min(idx, __float_as_int(pt.y));
  }
  return make_float2(best, __int_as_float(warp_min_int(idx)));
}

// ---------------------------------------------------------------------------
// Decisions
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool bad_temperature(float T) {
  return isnan(T) || (T > 0.f && T < kTinyT);
}

__device__ __forceinline__ void write_error_row(const KParams &P, int b, int status, int width,
                                                int32_t *tokens_base, int32_t *path_base) {
  for (int s = threadIdx.x; s < width; s += kThreads) {
    tokens_base[s] = -1;
    if (path_base) path_base[s] = -1;
  }
  if (threadIdx.x == 0) {
    P.out_nacc[b] = 0;
    if (P.out_status) P.out_status[b] = status;
  }
}

// Chain row decision (stochastic rows and greedy rows of spec_verify_chain,
// and every row of spec_verify_chain_greedy).
template <int MODE, int TDT, int DDT, bool PROBS>
__device__ void decide_chain(const KParams &P, int b, SmemChain &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int g = P.gamma, G1 = g + 1, V = P.V, tiles = P.tiles;
  const int lane = lane_id(), warp = warp_id();
  const float T = (MODE == MODE_CHAIN) ? __ldg(P.temps + b) : 0.f;
  const bool badT = bad_temperature(T);
  const bool greedy = T <= 0.f;
  const float c = kLog2e / T;
  const int nrows = greedy ? G1 : P.rows;
  const float2 *prow_part = P.partA + (size_t)b * P.rows * tiles;
  const TT *tgt = reinterpret_cast<const TT *>(P.target) + (size_t)b * G1 * V;
  int32_t *ot = P.out_tokens + (size_t)b * G1;

  // 1. merge the partials of every row read
  if (!badT) {
    for (int r = warp; r < nrows; r += kWarps) {
      const float2 *pp = prow_part + (size_t)r * tiles;
      if (greedy) {
        const float2 mi = warp_merge_argmax(pp, tiles);
        if (lane == 0) { sm.rowM[r] = mi.x; sm.rowI[r] = __float_as_int(mi.y); }
      } else {
        const float2 mz = warp_merge_softmax(pp, tiles, c);
        if (lane == 0) { sm.rowM[r] = mz.x; sm.rowZ[r] = mz.y; }
      }
    }
  }
  __syncthreads();

  // 2. per-position tests, one lane per draft position, first-reject scan
  if (warp == 0) {
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
      if (act && P.out_diag) {
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + i] = z;
      }
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
          const float lq = Elt<DDT>::load1(drow + x);
          q = ex2((lq - sm.rowM[G1 + i]) * c) / sm.rowZ[G1 + i];
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
    if (lane == 0) { sm.j = j; sm.status = status; }
  }
  __syncthreads();
  const int j = sm.j, status = sm.status;
  int kind = DEC_DONE;

  // 3. outputs
  if (status) {
    write_error_row(P, b, status, G1, ot, nullptr);
  } else {
    for (int s = threadIdx.x; s < G1; s += kThreads) {
      if (s < j) ot[s] = __ldg(P.draft_tokens + (size_t)b * g + s);
      else if (s > j) ot[s] = -1;
      else if (greedy) ot[s] = sm.rowI[j];
    }
    if (threadIdx.x == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
    }
    if (!greedy) {
      if (j == g) {
        // bonus token from p_gamma, straight from the Phase-A partials
        const int k = sample_row_from_partials<TDT>(tgt + (size_t)g * V,
                                                    prow_part + (size_t)g * tiles, tiles, V,
                                                    sm.rowM[g], c,
                                                    __ldg(P.unif + (size_t)b * G1 + g), sm);
        if (threadIdx.x == 0) ot[g] = k;
      } else {
        kind = DEC_RESIDUAL;
      }
    }
  }

  // 4. publish the decision for the Phase-B units and reset the arrival count
  if (threadIdx.x == 0) {
    if (P.phase_b) {
      Decision *d = P.dec + b;
      d->kind = kind;
      d->j = j;
      if (kind == DEC_RESIDUAL) {
        d->c = c;
        d->Mp = sm.rowM[j];
        d->invZp = 1.f / sm.rowZ[j];
        d->Mq = PROBS ? 0.f : sm.rowM[G1 + j];
        d->invZq = PROBS ? 1.f : 1.f / sm.rowZ[G1 + j];
        d->u = __ldg(P.unif + (size_t)b * G1 + g);
      }
      __threadfence();
      st_release(P.flag + b, 1u);
    }
    P.a_count[b] = 0;
  }
}

// Last Phase-B unit of a rejected row: crossing tile of u * R, rescan.
template <int TDT, int DDT, bool PROBS>
__device__ void finalize_residual(const KParams &P, int b, const Decision &d, SmemChain &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int g = P.gamma, G1 = g + 1, V = P.V, tiles = P.tiles, j = d.j;
  const float *pb = P.partB + (size_t)b * tiles;
  if (threadIdx.x == 0) {
    float R = 0.f;
    for (int t = 0; t < tiles; ++t) R += __ldcg(pb + t);
    const float target = d.u * R;
    float acc = 0.f, base = 0.f, last_base = 0.f;
    int ts = -1, last_t = -1;
    if (R > 0.f && R <= 3.0e38f) {
      for (int t = 0; t < tiles; ++t) {
        const float w = __ldcg(pb + t);
        if (w > 0.f) { last_t = t; last_base = acc; }
        if (acc + w > target) { ts = t; base = acc; break; }
        acc += w;
      }
      if (ts < 0) { ts = last_t; base = last_base; }
    }
    sm.R = R; sm.ts = ts; sm.base = base; sm.target = target;
  }
  __syncthreads();
  const float R = sm.R, base = sm.base, target = sm.target;
  const int ts = sm.ts;
  __syncthreads();
  const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)b * G1 + j) * V;
  int32_t *ot = P.out_tokens + (size_t)b * G1;
  if (isnan(R) || isinf(R)) {
    write_error_row(P, b, SV_ROW_NONFINITE, G1, ot, nullptr);
    return;
  }
  int k;
  if (!(R > 0.f)) {
    // zero residual mass: draw from p_j
    const float2 *pp = P.partA + ((size_t)b * P.rows + j) * tiles;
    k = sample_row_from_partials<TDT>(prow, pp, tiles, V, d.Mp, d.c, d.u, sm);
  } else {
    const int x0 = ts * kTile, n = min(kTile, V - x0);
    const TT *pt = prow + x0;
    const DTy *qt = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + j) * V + x0;
    k = x0 + crossing_scan(n, base, target, [&](int e) {
          return residual_term<PROBS>(Elt<TDT>::load1(pt + e), Elt<DDT>::load1(qt + e), d);
        }, sm);
  }
  if (threadIdx.x == 0) {
    ot[j] = k;
    if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
  }
}

// Tree decision: argmax per node, validation, walk from the root.
template <int DT>
__device__ void decide_tree(const KParams &P, int b, SmemTree &sm) {
  const int N = P.N, V = P.V, tiles = P.tiles, D = P.max_depth;
  const int lane = lane_id(), warp = warp_id();
  if (threadIdx.x == 0) sm.status = 0;
  __syncthreads();
  const float2 *part = P.partA + (size_t)b * N * tiles;
  int flags = 0;
  for (int r = warp; r < N; r += kWarps) {
    const float2 mi = warp_merge_argmax(part + (size_t)r * tiles, tiles);
    if (lane == 0) {
      sm.a[r] = __float_as_int(mi.y);
      if (isnan(mi.x)) flags |= SV_ROW_NONFINITE;
    }
  }
  for (int n = threadIdx.x; n < N; n += kThreads) {
    const int par = __ldg(P.parent + (size_t)b * N + n);
    const int tok = __ldg(P.node_tokens + (size_t)b * N + n);
    sm.par[n] = par;
    sm.tok[n] = tok;
    if (n == 0 ? par != -1 : (par < 0 || par >= n)) flags |= SV_ROW_BAD_TREE;
    if (n > 0 && (tok < 0 || tok >= V)) flags |= SV_ROW_BAD_TOKEN;
  }
  if (flags) atomicOr(&sm.status, flags);
  __syncthreads();
  const int status = sm.status;
  const int W = D + 1;
  int32_t *op = P.out_path + (size_t)b * W;
  int32_t *ot = P.out_tokens + (size_t)b * W;
  if (status) {
    write_error_row(P, b, status, W, ot, op);
  } else if (warp == 0) {
    int cur = 0, d = 0;
    while (d < D) {
      const int a = sm.a[cur];
      int found = -1;
      for (int base = cur + 1; base < N && found < 0; base += 32) {
        const int c = base + lane;
        const bool m = c < N && sm.par[c] == cur && sm.tok[c] == a;
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
  if (threadIdx.x == 0) P.a_count[b] = 0;
}

// ---------------------------------------------------------------------------
// Units
// ---------------------------------------------------------------------------

struct UnitRef {
  bool isA;
  int b, idx;
};

__device__ __forceinline__ UnitRef decode_unit(int u, const Sched &s) {
  const int LA = s.L * s.A;
  if (u < LA) return {true, u / s.A, u % s.A};
  u -= LA;
  const int blk = s.A + s.Bc;
  const int mid = (s.B - s.L) * blk;
  if (u < mid) {
    const int k = u / blk, r = u % blk;
    if (r < s.A) return {true, k + s.L, r};
    return {false, k, r - s.A};
  }
  u -= mid;
  return {false, s.B - s.L + u / s.Bc, u % s.Bc};
}

template <int MODE, int TDT, int DDT, bool PROBS, class Smem>
__device__ void run_unit_A(const KParams &P, int b, int idx, Smem &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int r = idx / P.tiles, t = idx % P.tiles;
  const int x0 = t * kTile, n = min(kTile, P.V - x0);
  const int V = P.V;
  float2 part = make_float2(0.f, 0.f);
  bool have = false;
  if (MODE == MODE_CHAIN) {
    const float T = __ldg(P.temps + b);
    const int G1 = P.gamma + 1;
    if (!bad_temperature(T)) {
      if (r < G1) {
        const TT *row = reinterpret_cast<const TT *>(P.target) + ((size_t)b * G1 + r) * V;
        part = (T <= 0.f) ? tile_argmax<TDT>(row, x0, n, sm)
                          : tile_softmax<TDT>(row, x0, n, kLog2e / T, sm);
        have = true;
      } else if (!PROBS && T > 0.f) {
        const DTy *row =
            reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * P.gamma + (r - G1)) * V;
        part = tile_softmax<DDT>(row, x0, n, kLog2e / T, sm);
        have = true;
      }
    }
  } else {
    const int rows_per = (MODE == MODE_TREE) ? P.N : P.gamma + 1;
    const TT *row = reinterpret_cast<const TT *>(P.target) + ((size_t)b * rows_per + r) * V;
    part = tile_argmax<TDT>(row, x0, n, sm);
    have = true;
  }
  if (threadIdx.x == 0) {
    if (have) P.partA[((size_t)b * P.rows + r) * P.tiles + t] = part;
    __threadfence();
    const unsigned prev = atomicAdd(P.a_count + b, 1u);
    sm.flag = (prev == (unsigned)(P.sched.A - 1));
  }
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    if constexpr (MODE == MODE_TREE) decide_tree<TDT>(P, b, sm);
    else decide_chain<MODE, TDT, DDT, PROBS>(P, b, sm);
  }
}

template <int TDT, int DDT, bool PROBS>
__device__ void run_unit_B(const KParams &P, int b, int t, SmemChain &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  if (threadIdx.x == 0) {
    const unsigned f = wait_flag_bounded(P.flag + b);
    sm.flag = f ? 1 : 0;
    if (f) {
      const Decision *d = P.dec + b;
      sm.dec.kind = __ldcg(&d->kind);
      sm.dec.j = __ldcg(&d->j);
      sm.dec.c = __ldcg(&d->c);
      sm.dec.Mp = __ldcg(&d->Mp);
      sm.dec.invZp = __ldcg(&d->invZp);
      sm.dec.Mq = __ldcg(&d->Mq);
      sm.dec.invZq = __ldcg(&d->invZq);
      sm.dec.u = __ldcg(&d->u);
    } else {
      atomicOr(P.err + b, SV_ROW_TIMEOUT);
    }
  }
  __syncthreads();
  const Decision d = sm.dec;
  const bool ok = sm.flag;
  const int V = P.V, g = P.gamma, G1 = g + 1;
  if (ok && d.kind == DEC_RESIDUAL) {
    const int x0 = t * kTile, n = min(kTile, V - x0);
    const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)b * G1 + d.j) * V;
    const DTy *qrow = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + d.j) * V;
    const float s = tile_residual<TDT, DDT, PROBS>(prow, qrow, x0, n, d, sm);
    if (threadIdx.x == 0) P.partB[(size_t)b * P.tiles + t] = s;
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(P.b_count + b, 1u);
    sm.flag2 = (prev == (unsigned)(P.sched.Bc - 1));
  }
  __syncthreads();
  if (sm.flag2) {
    __threadfence();
    const int err = __ldcg(P.err + b);
    if (err) {
      write_error_row(P, b, err, G1, P.out_tokens + (size_t)b * G1, nullptr);
    } else if (ok && d.kind == DEC_RESIDUAL) {
      finalize_residual<TDT, DDT, PROBS>(P, b, d, sm);
    }
    if (threadIdx.x == 0) {
      P.b_count[b] = 0;
      P.err[b] = 0;
      P.flag[b] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------

// PHASES selects which unit kinds this instantiation executes (1 = Phase A
// with decisions, 2 = Phase B with finalisation, 3 = both), so a launch that
// runs one kind carries only that kind's registers.
template <int MODE, int TDT, int DDT, bool PROBS, int PHASES>
__global__ void __launch_bounds__(kThreads, 4) sv_verify_kernel(const KParams P) {
  using Smem = typename std::conditional<MODE == MODE_TREE, SmemTree, SmemChain>::type;
  __shared__ Smem sm;
  if (threadIdx.x == 0) sm.unit[0] = atomicAdd(&P.hdr->unit_counter, 1u);
  __syncthreads();
  int parity = 0;
  unsigned unit = sm.unit[0];
  while (unit < (unsigned)P.sched.total) {
    unsigned next = 0;
    if (threadIdx.x == 0) next = atomicAdd(&P.hdr->unit_counter, 1u);
    const UnitRef u = decode_unit((int)unit, P.sched);
    if (u.isA) {
      if constexpr ((PHASES & 1) != 0) run_unit_A<MODE, TDT, DDT, PROBS>(P, u.b, u.idx, sm);
    } else {
      if constexpr (MODE == MODE_CHAIN && (PHASES & 2) != 0)
        run_unit_B<TDT, DDT, PROBS>(P, u.b, u.idx, sm);
    }
    if (threadIdx.x == 0) sm.unit[parity ^ 1] = next;
    __syncthreads();
    parity ^= 1;
    unit = sm.unit[parity];
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned done = atomicAdd(&P.hdr->exit_counter, 1u);
    if (done == gridDim.x - 1) {
      P.hdr->unit_counter = 0;
      P.hdr->exit_counter = 0;
      __threadfence();
    }
  }
}

}  // namespace sv
