// Inverse-CDF draws: crossing search over chunk masses
// and rescan of the crossing chunk ("論文解説: Speculative Sampling",
// §修正付き棄却サンプリング; the draw is the inverse CDF in ascending vocabulary
// order: the smallest k with sum_{x<=k} w(x) > u * sum_x w(x)).
#pragma once

#include "sv_pass_common.cuh"

namespace sv {

// First index i in [0, cnt) where the running sum of w(i) exceeds target;
// `base` receives the sum before it.  If rounding leaves no such i, the last
// i with w(i) > 0 (and the sum before it); -1 if every w is zero.
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
      base = acc + __shfl_sync(0xffffffffu, incl - v, l);
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

// The lane's PER consecutive elements x0 + lane * PER + k (k < PER) of a row
// of V elements; elements outside [0, V) get `pad`.  Vector loads when the
// lane's elements all lie in the row and start on a 16-byte boundary,
// otherwise one element at a time (no byte outside the row is read).
template <int DT, int PER>
__device__ __forceinline__ void lane_row_load(const typename Elt<DT>::T *row, int x0, int V,
                                              float pad, float (&v)[PER]) {
  using E = Elt<DT>;
  constexpr int VEC = E::kVec;
  const int xs = x0 + lane_id() * PER;
  const typename E::T *p = row + xs;
  bool vec = xs >= 0 && xs + PER <= V;
  if constexpr (PER % VEC == 0) {
    vec = vec && (reinterpret_cast<uintptr_t>(p) & 15) == 0;
    if (vec) {
#pragma unroll
      for (int k = 0; k < PER / VEC; ++k) E::unpack(ld_nc16(p + k * VEC), &v[k * VEC]);
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) v[k] = (xs + k >= 0 && xs + k < V) ? E::load1(row + xs + k) : pad;
}

// Crossing inside a chunk whose lane-consecutive weights are w[PER]: the
// local index of the first element where base + cumsum > target, or the last
// positive element if rounding leaves none.
template <int PER>
__device__ __forceinline__ int warp_rescan(const float (&w)[PER], float base, float target) {
  const int lane = lane_id();
  float tsum = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    tsum += w[k];
    if (w[k] > 0.f) lastpos = lane * PER + k;
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
  float acc = start;
#pragma unroll
  for (int kk = 0; kk < PER; ++kk) {
    acc += w[kk];
    if (k < 0 && acc > target) k = lane * PER + kk;
  }
  if (k < 0) k = lastpos >= 0 ? lastpos : lane * PER;
  return __shfl_sync(0xffffffffu, k, l);
}

// Up to 32 K per-chunk weights held in registers: w[k] is the weight of
// index 32 k + lane (0 past cnt).  One round trip loads them all.
constexpr int kRegK = 16;

template <class WF>
__device__ __forceinline__ void warp_load_weights(int cnt, WF wf, float (&w)[kRegK]) {
  const int lane = lane_id();
#pragma unroll
  for (int k = 0; k < kRegK; ++k) {
    const int i = 32 * k + lane;
    w[k] = i < cnt ? wf(i) : 0.f;
  }
}

// warp_prefix_cross over register-held weights (cnt <= 32 kRegK).
__device__ __forceinline__ int warp_cross_regs(const float (&w)[kRegK], int cnt, float target,
                                               float &base) {
  const int lane = lane_id();
  float acc = 0.f, last_base = 0.f;
  int last_i = -1;
#pragma unroll
  for (int k = 0; k < kRegK; ++k) {
    if (32 * k < cnt) {
      const float v = w[k];
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
        base = acc + __shfl_sync(0xffffffffu, incl - v, l);
        return 32 * k + l;
      }
      if (pos) {
        const int l = 31 - __clz(pos);
        last_base = acc + __shfl_sync(0xffffffffu, incl - v, l);
        last_i = 32 * k + l;
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  base = last_base;
  return last_i;
}

// Crossing of u * R over per-chunk weights wf(i), i < cnt, R = their sum
// (returned in R): register-held when they fit (one round trip), else
// streamed 32 at a time.  Returns the chunk (>= 0) and the sum before it.
template <class WF>
__device__ __forceinline__ int warp_chunk_cross(int cnt, WF wf, float u, float &R, float &base) {
  int t;
  if (cnt <= 32 * kRegK) {
    float w[kRegK];
    warp_load_weights(cnt, wf, w);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kRegK; ++k) s += w[k];
    R = warp_sum(s);
    t = warp_cross_regs(w, cnt, u * R, base);
  } else {
    float s = 0.f;
    for (int i = lane_id(); i < cnt; i += 32) s += wf(i);
    R = warp_sum(s);
    t = warp_prefix_cross(cnt, u * R, wf, base);
  }
  return t < 0 ? 0 : t;
}

// Draw from softmax row `row` (V elements of DT, max M, scale c) with the
// row's chunk partials part[cnt]: the chunk masses
// s_i 2^((m_i - M) c) locate the crossing chunk of u * R, then that chunk is
// rescanned element by element.  Chunk i starts at vocabulary index
// i * kElems - off (off: the row's elements before its first 16-byte
// boundary, 0 for a row that starts on one).  Returns a vocabulary index.
template <int DT>
static __device__ __noinline__ int warp_sample_softmax_row(const typename Elt<DT>::T *row,
                                                           const Part *part, int cnt, int V,
                                                           float M, float c, float u,
                                                           int off = 0) {
  using C = Chunk<DT>;
  constexpr int HALF = C::kElems / 2, PER = HALF / 32;
  auto wt = [&](int i) {
    const float2 p = part_value(part + i);
    return p.x != -CUDART_INF_F ? p.y * ex2((p.x - M) * c) : 0.f;
  };
  float R = 0.f, base = 0.f;
  const int t = warp_chunk_cross(cnt, wt, u, R, base);
  const float target = u * R;
  // rescan the crossing chunk one half at a time (32 values per lane)
  int x0 = t * C::kElems - off;
  float v[PER];
  lane_row_load<DT, PER>(row, x0, V, -CUDART_INF_F, v);
  float hs = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    v[k] = ex2((v[k] - M) * c);
    hs += v[k];
  }
  hs = warp_sum(hs);
  if (base + hs <= target && x0 + HALF < V) {
    base += hs;
    x0 += HALF;
    lane_row_load<DT, PER>(row, x0, V, -CUDART_INF_F, v);
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = ex2((v[k] - M) * c);
  }
  return x0 + warp_rescan<PER>(v, base, target);
}

}  // namespace sv
