// Decider-warp helpers of the streaming kernel: row merges, inverse-CDF
// crossings and slice rescans.  Every step issues its loads for the whole
// warp at once, so a decision costs a handful of L2 round trips.
#pragma once

#include "sv_stream_common.cuh"

namespace sv {

// Lane-owned merge of one softmax row's tile partials (m_t, s_t):
// M = max m_t, Z = sum s_t exp2((m_t - M) c), single pass with rescaling.
// Partials are loaded eight at a time into registers before they are used,
// so each chunk costs one L2 round trip.  NaN in any partial makes Z NaN.
__device__ __forceinline__ float2 lane_merge_softmax(const float2 *part, int tiles, float c) {
  float M = -CUDART_INF_F, Z = 0.f;
  bool nan = false;
  for (int t0 = 0; t0 < tiles; t0 += 8) {
    float2 pt[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      pt[k] = (t0 + k < tiles) ? __ldcg(part + t0 + k) : make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      nan |= isnan(pt[k].x) || isnan(pt[k].y);
      if (pt[k].x == -CUDART_INF_F) continue;
      if (pt[k].x > M) {
        Z = Z * ex2((M - pt[k].x) * c) + pt[k].y;
        M = pt[k].x;
      } else {
        Z += pt[k].y * ex2((pt[k].x - M) * c);
      }
    }
  }
  return make_float2(nan ? CUDART_NAN_F : M, nan ? CUDART_NAN_F : Z);
}

// Lane-owned merge of one argmax row's tile partials (value, index): the
// strictly larger value wins, so equal maxima keep the earlier (lower) index.
__device__ __forceinline__ float2 lane_merge_argmax(const float2 *part, int tiles) {
  float2 best = make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
  bool nan = false, first = true;
  for (int t0 = 0; t0 < tiles; t0 += 8) {
    float2 pt[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      pt[k] = (t0 + k < tiles) ? __ldcg(part + t0 + k)
                               : make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (t0 + k >= tiles) continue;
      nan |= isnan(pt[k].x);
      if (first || pt[k].x > best.x) best = pt[k];
      first = false;
    }
  }
  if (nan) best.x = CUDART_NAN_F;
  return best;
}

// First index i in [0, cnt) where the running sum of w(i) exceeds target;
// `base` receives the sum before it.  Falls back to the last i with w > 0.
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

// The lane's PER consecutive elements [lane * PER, lane * PER + PER) of a
// slice starting at `base` (16-byte aligned), n valid elements; others `pad`.
template <int DT, int PER>
__device__ __forceinline__ void lane_chunk_load(const typename Elt<DT>::T *base, int n, float pad,
                                                float (&v)[PER]) {
  using E = Elt<DT>;
  constexpr int VEC = E::kVec;  // elements per 16 bytes
  const int e0 = lane_id() * PER;
  const typename E::T *p = base + e0;
  if (e0 + PER <= n) {
    if constexpr (PER % VEC == 0) {
#pragma unroll
      for (int k = 0; k < PER / VEC; ++k) E::unpack(__ldg(reinterpret_cast<const uint4 *>(p) + k), &v[k * VEC]);
    } else {
#pragma unroll
      for (int k = 0; k < PER; ++k) v[k] = E::load1(p + k);
    }
  } else {
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = (e0 + k < n) ? E::load1(p + k) : pad;
  }
}

// Inverse-CDF crossing inside a slice whose lane-chunk weights are w[PER]:
// the local index of the first element where base + cumsum > target, or the
// last positive element if rounding leaves none.
template <int PER>
__device__ __forceinline__ int warp_rescan_regs(const float (&w)[PER], float base, float target) {
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

// Draw from softmax row `row` (tiles of TileA<DT>::kElems elements) with the
// tile partials pt[tiles] and slice partials ps[tiles][kCW]: crossing tile,
// crossing warp slice, rescan of that slice.  Returns a vocabulary index.
template <int DT>
__device__ int warp_sample_row(const typename Elt<DT>::T *row, const float2 *pt,
                               const float2 *ps, int tiles, int V, float M, float c, float u) {
  constexpr int TA = TileA<DT>::kElems, SLICE = TileA<DT>::kSlice, PER = SLICE / 32;
  auto wt = [&](int i) {
    const float2 p = __ldcg(pt + i);
    return p.x != -CUDART_INF_F ? p.y * ex2((p.x - M) * c) : 0.f;
  };
  float R = 0.f;
  for (int i = lane_id(); i < tiles; i += 32) R += wt(i);
  R = warp_sum(R);
  const float target = u * R;
  float base = 0.f;
  int t = warp_prefix_cross(tiles, target, wt, base);
  if (t < 0) t = 0;
  const float2 *pw = ps + (size_t)t * kCW;
  auto ww = [&](int i) {
    const float2 p = __ldcg(pw + i);
    return p.x != -CUDART_INF_F ? p.y * ex2((p.x - M) * c) : 0.f;
  };
  float base2 = 0.f;
  int w = warp_prefix_cross(kCW, target - base, ww, base2);
  if (w < 0) w = 0;
  const int x0 = t * TA + w * SLICE;
  const int n = min(SLICE, V - x0);
  float v[PER];
  lane_chunk_load<DT, PER>(row + x0, n, -CUDART_INF_F, v);
#pragma unroll
  for (int k = 0; k < PER; ++k) v[k] = ex2((v[k] - M) * c);
  return x0 + warp_rescan_regs<PER>(v, base + base2, target);
}

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

}  // namespace sv
