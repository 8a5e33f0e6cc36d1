// Small calls in one launch: one thread-block cluster per batch row (chains)
// or per tree, with no workspace and no global atomics.
//
// CTA r of a cluster owns the vocabulary slice [r S, (r + 1) S) of every
// row its batch row needs.  It reduces its slice of each row to a partial,
// the partials of the cluster's CTAs are merged through distributed shared
// memory (DSMEM) after a cluster barrier, and every CTA makes the row's
// decision from the merged statistics.
//
// Chains ("論文解説: Speculative Sampling", §技術的詳細 ステップ3 and
// §修正付き棄却サンプリング; greedy rows: "投機的デコーディングとは？"
// §ドラフト生成と並列検証の仕組み): a chain CTA keeps its slices of the rows in
// shared memory, so the accept tests, the residual max(0, p_j - q_j) and the
// draws read no logit twice from global memory.  After the decision each
// warp sums the draw's weights over its part of the slice; a second cluster
// barrier makes those sums visible, every CTA locates the part holding the
// crossing of u R, and the warp that owns it rescans its part from shared
// memory and writes the row's outputs.
//
// Trees (SpecInfer explainer, §推論方法): a tree CTA streams its slices of
// the node rows (argmax only), and CTA 0 merges the node rows through DSMEM
// and walks the tree.
//
// A last cluster barrier keeps every CTA resident until no other CTA can
// still read its shared memory.  Every CTA passes every barrier, whatever
// its rows hold.
#pragma once

#include "sv_pass_decide.cuh"

namespace sv {

constexpr int kClusterMax = 8;        // largest cluster: the portable size
constexpr int kClThreads = 512;       // chain CTAs: 16 warps, one per kept row at a time
constexpr int kClWarps = kClThreads / 32;
constexpr int kClParts = kClusterMax * kClWarps;  // draw parts of a cluster: at most 128
constexpr int kClusterSmemMax = 128 * 1024;  // kept row slices and draw weights per chain CTA

struct ClusterParams {
  const void *target;  // chain: [B, gamma+1, V]; tree: [B*N, V]
  const void *draft;   // [B, gamma, V] logits or fp32 probabilities
  const int32_t *draft_tokens;
  const float *temps;
  const float *unif;
  const int32_t *parent;
  const int32_t *node_tokens;
  int B, gamma, V, N, max_depth;
  int S;        // slice elements per CTA (a multiple of 8)
  int rstride;  // bytes of one kept row slice in shared memory (a multiple of 16)
  int32_t *out_tokens, *out_nacc, *out_status, *out_path;
  float *out_diag;
};

__device__ __forceinline__ unsigned smem_u32(const void *p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_size() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to DSMEM reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of shared variable p in CTA `rank` of the cluster.
__device__ __forceinline__ unsigned dsmem_addr(const void *p, unsigned rank) {
  unsigned r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_dsmem_f2(unsigned a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_dsmem_f32(unsigned a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// Element i of a kept slice (raw element type DT in shared memory).
template <int DT>
__device__ __forceinline__ float slice_elt(const unsigned char *row, int i) {
  if constexpr (DT == SV_F32) {
    return reinterpret_cast<const float *>(row)[i];
  } else {
    const unsigned short h = reinterpret_cast<const unsigned short *>(row)[i];
    if constexpr (DT == SV_BF16) return __uint_as_float((unsigned)h << 16);
    else return __half2float(__ushort_as_half(h));
  }
}

// Starts copying n elements of DT from global src into shared dst, thread t
// of nt: 16-byte asynchronous copies (cp.async, no register staging, all in
// flight at once) when src starts on a 16-byte boundary; otherwise eight
// elements per thread at a time through registers.  The caller commits and
// waits for the asynchronous copies.
template <int DT>
__device__ __forceinline__ void slice_copy(unsigned char *dst, const typename Elt<DT>::T *src,
                                           int n, int t, int nt) {
  using T = typename Elt<DT>::T;
  constexpr int ES = (int)sizeof(T), VEC = 16 / ES;
  T *d = reinterpret_cast<T *>(dst);
  if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
    const int nv = n / VEC;
    for (int v = t; v < nv; v += nt) cp_async<16>(dst + 16 * v, src + (size_t)v * VEC);
    for (int i = nv * VEC + t; i < n; i += nt) d[i] = src[i];
  } else {
    for (int i0 = 8 * t; i0 < n; i0 += 8 * nt) {
      T e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (i0 + k < n) e[k] = src[i0 + k];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (i0 + k < n) d[i0 + k] = e[k];
    }
  }
}

// Softmax partial (max, sum of 2^((x - max) c)) of a kept slice of n
// elements, by one warp: lanes take 16-byte vectors of the slice in turn (the
// chunk maximum on packed words, then the sum with four accumulators); the
// last partial vector is read element by element.  NaN anywhere gives NaN.
template <int DT>
__device__ __forceinline__ float2 slice_softmax(const unsigned char *row, int n, float c) {
  constexpr int VEC = Elt<DT>::kVec;
  const int lane = lane_id(), nv = n / VEC;
  const uint4 *rv = reinterpret_cast<const uint4 *>(row);
  unsigned mw = neg_inf_word<DT>();
#pragma unroll 4
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = rv[v];
    mw = packed_max<DT>(mw, packed_max<DT>(packed_max<DT>(w.x, w.y), packed_max<DT>(w.z, w.w)));
  }
  float m = packed_word_max<DT>(mw);
  for (int i = nv * VEC + lane; i < n; i += 32) m = max_nan(m, slice_elt<DT>(row, i));
  m = warp_max_nan(m);
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  if (m != -CUDART_INF_F) {
#pragma unroll 2
    for (int v = lane; v < nv; v += 32) {
      float f[VEC];
      Elt<DT>::unpack(rv[v], f);
#pragma unroll
      for (int t = 0; t < VEC; ++t) s4[t & 3] += ex2((f[t] - m) * c);
    }
    for (int i = nv * VEC + lane; i < n; i += 32) s4[0] += ex2((slice_elt<DT>(row, i) - m) * c);
  }
  return make_float2(m, warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3])));
}

// Argmax partial (max, lowest global index holding it) of a kept slice
// starting at vocabulary index x0, by one warp (NaN anywhere gives NaN).
template <int DT>
__device__ __forceinline__ float2 slice_argmax(const unsigned char *row, int n, int x0) {
  constexpr int VEC = Elt<DT>::kVec;
  const int lane = lane_id(), nv = n / VEC;
  const uint4 *rv = reinterpret_cast<const uint4 *>(row);
  unsigned mw = neg_inf_word<DT>();
#pragma unroll 4
  for (int v = lane; v < nv; v += 32) {
    const uint4 w = rv[v];
    mw = packed_max<DT>(mw, packed_max<DT>(packed_max<DT>(w.x, w.y), packed_max<DT>(w.z, w.w)));
  }
  float m = packed_word_max<DT>(mw);
  for (int i = nv * VEC + lane; i < n; i += 32) m = max_nan(m, slice_elt<DT>(row, i));
  m = warp_max_nan(m);
  if (isnan(m)) return make_float2(m, __int_as_float(0x7fffffff));
  // the lane's first element equal to the maximum (its vectors in order)
  int idx = 0x7fffffff;
  for (int v = lane; v < nv && idx == 0x7fffffff; v += 32) {
    float f[VEC];
    Elt<DT>::unpack(rv[v], f);
#pragma unroll
    for (int t = VEC - 1; t >= 0; --t)
      if (f[t] == m) idx = v * VEC + t;
  }
  for (int i = nv * VEC + lane; i < n && idx == 0x7fffffff; i += 32)
    if (slice_elt<DT>(row, i) == m) idx = i;
  idx = warp_min_int(idx);
  return make_float2(m, __int_as_float(idx == 0x7fffffff ? idx : x0 + idx));
}

// Draw weights of slice element i: the residual max(0, p_j - q_j) of the
// kept pair (prow, qrow) when `resid`, else the unnormalised probability
// 2^((l - M) c) of row prow.
template <int TDT, int DDT, bool PROBS>
__device__ __forceinline__ float draw_weight(bool resid, const unsigned char *prow,
                                             const unsigned char *qrow, int i,
                                             const ResidCoef &rk, float M) {
  const float lp = slice_elt<TDT>(prow, i);
  if (!resid) return ex2((lp - M) * rk.c);
  const float p = ex2(fmaf(lp - rk.Mp, rk.c, -rk.lzp));
  const float q = PROBS ? slice_elt<SV_F32>(qrow, i)
                        : ex2(fmaf(slice_elt<DDT>(qrow, i) - rk.Mq, rk.c, -rk.lzq));
  return max_nan(0.f, p - q);
}

// An invalid chain row: every token -1, no draft accepted.
__device__ __forceinline__ void cluster_error_row(const ClusterParams &P, int b, int status,
                                                  int width) {
  int32_t *ot = P.out_tokens + (size_t)b * width;
  for (int s = lane_id(); s < width; s += 32) ot[s] = -1;
  if (lane_id() == 0) {
    P.out_nacc[b] = 0;
    if (P.out_status) P.out_status[b] = status;
  }
}

// The draw chosen by every CTA's warp 0 from the cluster's part weights.
struct ClusterDraw {
  int bad;       // the weights are not finite (or hold no mass): an invalid row
  int alt;       // 1: the residual has no mass, so the draw takes p_j instead
  int part;      // the part (CTA rank * warps + warp) holding the crossing
  float base;    // the mass before that part
  float target;  // u R (+inf: rounding left no crossing, take the last positive element)
  float R;       // the residual mass (the diagnostics' fourth column)
};

template <int MODE, int TDT, int DDT, bool PROBS>
__global__ void __launch_bounds__(kClThreads, 1) sv_cluster_chain_kernel(const ClusterParams P) {
  extern __shared__ __align__(16) unsigned char cl_rows[];  // kept row slices
  __shared__ float2 cl_part[kMaxRows];  // this CTA's partial of each row
  __shared__ float rowM[kMaxRows], rowZ[kMaxRows];
  __shared__ int rowI[kMaxRows];
  __shared__ float cl_w[2][kClWarps];  // this CTA's per-warp draw weights
  __shared__ float cl_lsum[kClWarps][32];  // ... per lane (the draw's own weights)
  __shared__ int cl_lpos[kClWarps][32];    // each lane's last element of positive weight
  __shared__ int cl_j, cl_kind;
  __shared__ int cl_x[32];  // the draft tokens, for the row's outputs
  __shared__ ResidCoef cl_rk;
  __shared__ ClusterDraw cl_draw;
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  grid_dependents_launch();
  grid_dependency_wait();  // the inputs written by earlier work in the stream are visible
  const unsigned CS = cluster_size(), rank = cluster_rank();
  const int b = blockIdx.x / CS;
  const int g = P.gamma, G1 = g + 1, V = P.V;
  const int lane = lane_id(), warp = warp_id();
  const int x_lo = (int)rank * P.S;
  const int n = max(0, min(V, x_lo + P.S) - x_lo);
  const float T = MODE == MODE_CHAIN ? __ldg(P.temps + b) : 0.f;
  const bool badT = bad_temperature(T);
  const bool greedy = !badT && T <= 0.f;
  const float c = kLog2e / T;
  // kept rows: target 0..gamma, then (stochastic rows) draft 0..gamma-1
  const int nkeep = badT ? 0 : (greedy ? G1 : G1 + g);
  const TT *tgt = reinterpret_cast<const TT *>(P.target) + (size_t)b * G1 * V;
  const DTy *drf = MODE == MODE_CHAIN ? reinterpret_cast<const DTy *>(P.draft) + (size_t)b * g * V
                                      : nullptr;
  // 1. this CTA's slices into shared memory (every thread takes part in
  // every row, so every copy is in flight at once)
  for (int k = 0; k < nkeep; ++k) {
    unsigned char *dst = cl_rows + (size_t)k * P.rstride;
    if (k < G1) slice_copy<TDT>(dst, tgt + (size_t)k * V + x_lo, n, threadIdx.x, kClThreads);
    else slice_copy<DDT>(dst, drf + (size_t)(k - G1) * V + x_lo, n, threadIdx.x, kClThreads);
  }
  cp_async_commit();
  // 0. the draft tokens and the uniforms (one lane per position), issued
  // while the copies are in flight; the logits at the tokens are gathered
  // after the copies (below), so no warp waits for the dependent load
  const bool act = warp == 0 && lane < g;
  int x = 0;
  bool tok_ok = false;
  float lp = 0.f, lq = 0.f, ui = 0.f;
  if (act && !badT) {
    x = __ldg(P.draft_tokens + (size_t)b * g + lane);
    if (!greedy) ui = __ldg(P.unif + (size_t)b * G1 + lane);
  }
  const float ug = (!badT && !greedy) ? __ldg(P.unif + (size_t)b * G1 + g) : 0.f;
  cp_async_wait_all();
  __syncthreads();
  if (act && !badT) {
    cl_x[lane] = x;
    tok_ok = x >= 0 && x < V;
    if (!greedy && tok_ok) {  // used by the accept tests, after the row statistics
      lp = Elt<TDT>::load1(tgt + (size_t)lane * V + x);
      lq = Elt<DDT>::load1(drf + (size_t)lane * V + x);
    }
  }
  // 2. slice partials: softmax rows (argmax for greedy rows); probability
  // drafts need none
  const int npart = greedy ? G1 : (PROBS ? G1 : G1 + g);
  for (int k = warp; k < npart; k += kClWarps) {
    const unsigned char *row = cl_rows + (size_t)k * P.rstride;
    float2 pt;
    if (greedy) pt = slice_argmax<TDT>(row, n, x_lo);
    else if (k < G1) pt = slice_softmax<TDT>(row, n, c);
    else pt = slice_softmax<DDT>(row, n, c);
    if (lane == 0) cl_part[k] = pt;
  }
  cluster_sync();  // 1: every CTA's partials are written
  // 3. merge every row over the cluster: lane l of a warp reads CTA l % CS's
  // partial of row l / CS of the warp's group of 32 / CS rows (one DSMEM
  // round trip per group), and the CS lanes of a row reduce by shuffles
  const int rpw = 32 / (int)CS;
  for (int k0 = warp * rpw; k0 < npart; k0 += kClWarps * rpw) {
    const int k = k0 + lane / (int)CS, q = lane % (int)CS;
    float2 pt = make_float2(-CUDART_INF_F, greedy ? __int_as_float(0x7fffffff) : 0.f);
    if (k < npart) pt = ld_dsmem_f2(dsmem_addr(&cl_part[k], (unsigned)q));
    float M = pt.x;
    for (int o = 1; o < (int)CS; o <<= 1) M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (greedy) {
      int nan = isnan(pt.x) ? 1 : 0;
      int I = pt.x == M ? __float_as_int(pt.y) : 0x7fffffff;
      for (int o = 1; o < (int)CS; o <<= 1) {
        nan |= __shfl_xor_sync(0xffffffffu, nan, o);
        I = min(I, __shfl_xor_sync(0xffffffffu, I, o));
      }
      if (q == 0 && k < npart) {
        rowM[k] = nan ? CUDART_NAN_F : M;
        rowI[k] = I;
      }
    } else {
      float z = (pt.x == -CUDART_INF_F) ? 0.f : pt.y * ex2((pt.x - M) * c);
      for (int o = 1; o < (int)CS; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      if (q == 0 && k < npart) {
        rowM[k] = M;
        rowZ[k] = z;
      }
    }
  }
  __syncthreads();
  // 4. the decision (warp 0 of every CTA; CTA 0 writes the diagnostics and
  // the rows that need no draw)
  if (warp == 0) {
    const unsigned gmask = (g >= 32) ? 0xffffffffu : ((1u << g) - 1u);
    int status = 0, j = g, kind = -1;
    float p = 0.f, q = 0.f;
    if (badT) {
      status = SV_ROW_BAD_TEMPERATURE;
    } else if (greedy) {
      bool nf = false;
      for (int r = lane; r < G1; r += 32) nf |= isnan(rowM[r]);
      const bool match = act && tok_ok && x == rowI[lane];
      const unsigned mm = __ballot_sync(0xffffffffu, match) & gmask;
      const unsigned badtok = __ballot_sync(0xffffffffu, act && !tok_ok);
      j = (~mm & gmask) ? __ffs(~mm & gmask) - 1 : g;
      status = (badtok ? SV_ROW_BAD_TOKEN : 0) | (__any_sync(0xffffffffu, nf) ? SV_ROW_NONFINITE : 0);
    } else {
      bool acc = false, nf = false;
      if (act && tok_ok) {
        p = ex2((lp - rowM[lane]) * c) / rowZ[lane];
        q = PROBS ? lq : ex2((lq - rowM[G1 + lane]) * c) / rowZ[G1 + lane];
        acc = ui * q < p;
      }
      for (int r = lane; r < npart; r += 32) {
        const float Z = rowZ[r];
        nf |= !(Z > 0.f && Z <= 3.0e38f);
      }
      if (PROBS) nf |= act && tok_ok && !isfinite(q);
      const unsigned am = __ballot_sync(0xffffffffu, acc) & gmask;
      const unsigned badtok = __ballot_sync(0xffffffffu, act && !tok_ok);
      j = (~am & gmask) ? __ffs(~am & gmask) - 1 : g;
      status = (badtok ? SV_ROW_BAD_TOKEN : 0) | (__any_sync(0xffffffffu, nf) ? SV_ROW_NONFINITE : 0);
      if (!status) kind = j < g ? 0 : 1;
    }
    if (rank == 0 && P.out_diag && act) {
      float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!badT && !greedy) {
        const float ap = (q > 0.f) ? fminf(1.f, p / q) : (p > 0.f ? 1.f : 0.f);
        d = make_float4(p, q, ap, 0.f);
      }
      reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + lane] = d;
    }
    if (rank == 0 && kind < 0) {
      // no draw: an invalid row, or a greedy row (the argmax of row j)
      if (status) {
        cluster_error_row(P, b, status, G1);
      } else {
        int32_t *ot = P.out_tokens + (size_t)b * G1;
        const int tj = rowI[j];
        for (int s = lane; s < G1; s += 32) ot[s] = s < j ? x : (s == j ? tj : -1);
        if (lane == 0) {
          P.out_nacc[b] = j;
          if (P.out_status) P.out_status[b] = 0;
        }
      }
    }
    if (lane == 0) {
      cl_j = j;
      cl_kind = kind;
      ResidCoef rk;
      rk.c = c;
      rk.Mp = kind >= 0 ? rowM[j] : 0.f;
      rk.lzp = kind >= 0 ? log2f(rowZ[j]) : 0.f;
      rk.Mq = (kind == 0 && !PROBS) ? rowM[G1 + j] : 0.f;
      rk.lzq = (kind == 0 && !PROBS) ? log2f(rowZ[G1 + j]) : 0.f;
      cl_rk = rk;
    }
  }
  __syncthreads();
  // 5. the draw's weights over this CTA's slice.  Warp w owns the part
  // [w L, (w + 1) L) of the slice, lane l the elements l PER .. l PER + PER - 1
  // of it.  kind 0 (a rejected pair): the residual, and p_j for the case of
  // a residual without mass; kind 1 (every draft accepted): the bonus row.
  const int kind = cl_kind, j = cl_j;
  const int PER = (n + kClThreads - 1) / kClThreads;
  const int L = 32 * PER;
  const ResidCoef rk = cl_rk;
  const unsigned char *prow = cl_rows + (size_t)(kind == 1 ? g : j) * P.rstride;
  const unsigned char *qrow = cl_rows + (size_t)(G1 + j) * P.rstride;
  const float Mw = kind == 1 ? rowM[g] : rk.Mp;  // the row whose probabilities weigh
  const int i0 = warp * L + lane * PER;
  // the draw's own weights (the residual, or the bonus row) are kept in
  // shared memory after the row slices, with each lane's sum and last
  // positive element, so the rescan below reads them back
  float *wbuf = reinterpret_cast<float *>(cl_rows + (size_t)(G1 + g) * P.rstride);
  float ws0 = 0.f, ws1 = 0.f;
  if (kind >= 0) {
    int lpos = -1;
    for (int t = 0; t < PER; ++t) {
      if (i0 + t >= n) break;
      const float w = draw_weight<TDT, DDT, PROBS>(kind == 0, prow, qrow, i0 + t, rk, Mw);
      wbuf[i0 + t] = w;
      ws0 += w;
      if (w > 0.f) lpos = i0 + t;
      if (kind == 0) ws1 += draw_weight<TDT, DDT, PROBS>(false, prow, qrow, i0 + t, rk, Mw);
    }
    cl_lsum[warp][lane] = ws0;
    cl_lpos[warp][lane] = lpos;
    ws0 = warp_sum(ws0);
    ws1 = warp_sum(ws1);
  }
  if (lane == 0) {
    cl_w[0][warp] = ws0;
    cl_w[1][warp] = ws1;
  }
  cluster_sync();  // 2: every CTA's weights are written
  // 6. every CTA's warp 0 reads the cluster's part weights (in vocabulary
  // order: CTA rank, then warp; lane l holds parts l, l + 32, l + 64, ...)
  // and locates the crossing of u R
  if (kind >= 0 && warp == 0) {
    constexpr int G = kClParts / 32;
    const int parts = (int)CS * kClWarps;
    float a[G], w[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int pt = lane + 32 * i;
      a[i] = w[i] = 0.f;
      if (pt < parts) {
        const unsigned q = (unsigned)(pt / kClWarps);
        a[i] = ld_dsmem_f32(dsmem_addr(&cl_w[0][pt % kClWarps], q));
        w[i] = ld_dsmem_f32(dsmem_addr(&cl_w[1][pt % kClWarps], q));
      }
    }
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      s0 += a[i];
      s1 += w[i];
    }
    const float R0 = warp_sum(s0), R1 = warp_sum(s1);
    ClusterDraw d;
    d.R = R0;
    d.alt = kind == 0 && !isnan(R0) && !isinf(R0) && !(R0 > 0.f);
    const float R = d.alt ? R1 : R0;
    if (!d.alt) {
#pragma unroll
      for (int i = 0; i < G; ++i) w[i] = a[i];
    }
    d.bad = isnan(R) || isinf(R) || !(R > 0.f);
    d.part = -1;
    d.base = 0.f;
    d.target = ug * R;
    if (!d.bad) {
      // inclusive prefix over the parts in order, group by group
      float incl[G], carry = 0.f;
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float v = w[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += y;
        }
        incl[i] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      int found = -1, lastpos = -1;
      float base_found = 0.f, base_last = 0.f;
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const bool in = lane + 32 * i < parts;
        const unsigned h = __ballot_sync(0xffffffffu, in && incl[i] > d.target);
        const float before = __shfl_sync(0xffffffffu, incl[i] - w[i], h ? __ffs(h) - 1 : 0);
        if (found < 0 && h) {
          found = 32 * i + __ffs(h) - 1;
          base_found = before;
        }
        const unsigned pm = __ballot_sync(0xffffffffu, in && w[i] > 0.f);
        const float lb = __shfl_sync(0xffffffffu, incl[i] - w[i], pm ? 31 - __clz(pm) : 0);
        if (pm) {
          lastpos = 32 * i + 31 - __clz(pm);
          base_last = lb;
        }
      }
      if (found >= 0) {
        d.part = found;
        d.base = base_found;
      } else {
        // rounding left no crossing: the last element of positive weight,
        // in the last part that holds one
        d.part = lastpos;
        d.base = base_last;
        d.target = CUDART_INF_F;
      }
    }
    if (lane == 0) cl_draw = d;
    if (d.bad && rank == 0) cluster_error_row(P, b, SV_ROW_NONFINITE, G1);
  }
  __syncthreads();
  // 7. the part's owner rescans it from shared memory and writes the row
  const ClusterDraw d = cl_draw;
  if (kind >= 0 && !d.bad && d.part / kClWarps == (int)rank && warp == d.part % kClWarps) {
    // the draw's own weights were kept; p_j (a residual without mass) is
    // weighed again
    float tsum = 0.f;
    int lastpos = -1;
    if (!d.alt) {
      tsum = cl_lsum[warp][lane];
      lastpos = cl_lpos[warp][lane];
    } else {
      for (int t = 0; t < PER; ++t) {
        if (i0 + t >= n) break;
        const float w = draw_weight<TDT, DDT, PROBS>(false, prow, qrow, i0 + t, rk, Mw);
        tsum += w;
        if (w > 0.f) lastpos = i0 + t;
      }
    }
    float incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float start = d.base + incl - tsum;
    const unsigned hit = __ballot_sync(0xffffffffu, start + tsum > d.target);
    int k;
    if (hit) {
      const int l = __ffs(hit) - 1;
      int kk = -1;
      if (lane == l) {
        float acc = start;
        for (int t = 0; t < PER && kk < 0; ++t) {
          if (i0 + t >= n) break;
          acc += d.alt ? draw_weight<TDT, DDT, PROBS>(false, prow, qrow, i0 + t, rk, Mw)
                       : wbuf[i0 + t];
          if (acc > d.target) kk = i0 + t;
        }
        if (kk < 0) kk = lastpos >= 0 ? lastpos : i0;
      }
      k = __shfl_sync(0xffffffffu, kk, l);
    } else {
      const int lp2 = warp_max_int(lastpos);
      k = lp2 >= 0 ? lp2 : warp * L;
    }
    k += x_lo;
    int32_t *ot = P.out_tokens + (size_t)b * G1;
    for (int s = lane; s < G1; s += 32) ot[s] = s < j ? cl_x[s] : (s == j ? k : -1);
    if (lane == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
      if (P.out_diag && kind == 0) P.out_diag[((size_t)b * g + j) * 4 + 3] = d.R;
    }
  }
  // 3: no CTA leaves while another may read its shared memory.  Every DSMEM
  // read of this kernel has returned its value before its warp arrives, so
  // the arrival needs no release (the row's global writes need none either:
  // the kernel's end makes them visible)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
               "barrier.cluster.wait.aligned;" ::: "memory");
}

// Trees: CTA r of tree b's cluster streams its slice of every node row.
// The slice is cut into 4 KB units (row k, unit c); warp w takes units w,
// w + 8, ... of the CTA's list, keeping the next unit's eight 16-byte loads
// per lane in flight while it reduces the current one to (max, lowest
// index).  The units of a row merge in shared memory, the CTAs' rows merge
// in CTA 0 through DSMEM, and CTA 0 validates the tree and walks it.  Rows
// start on 16-byte boundaries on this path, and S is a multiple of the
// vector width.
template <int DT>
__device__ __forceinline__ float2 tree_unit_argmax(const uint4 (&buf)[kChunkVecs], int n) {
  constexpr int VEC = Elt<DT>::kVec;
  const int lane = lane_id();
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
  int idx = 0x7fffffff;
#pragma unroll
  for (int u = kChunkVecs - 1; u >= 0; --u) {
    float f[VEC];
    Elt<DT>::unpack(buf[u], f);
#pragma unroll
    for (int t = VEC - 1; t >= 0; --t) {
      const int e = (lane + 32 * u) * VEC + t;
      if (f[t] == m && e < n) idx = e;  // descending: keeps the lowest
    }
  }
  return make_float2(m, __int_as_float(warp_min_int(idx)));
}

template <int DT>
__global__ void __launch_bounds__(kPassThreads, 2) sv_cluster_tree_kernel(const ClusterParams P) {
  extern __shared__ __align__(16) float2 tu[];  // [N][units per row]: unit partials
  __shared__ float2 tp[SV_MAX_TREE_NODES];      // this CTA's (max, lowest index) per node row
  __shared__ TreeSmem tsm;
  using TT = typename Elt<DT>::T;
  constexpr int VEC = Elt<DT>::kVec, E = Chunk<DT>::kElems;
  grid_dependents_launch();
  grid_dependency_wait();
  const unsigned CS = cluster_size(), rank = cluster_rank();
  const int b = blockIdx.x / CS;
  const int N = P.N, V = P.V;
  const int lane = lane_id(), warp = warp_id();
  const int x_lo = (int)rank * P.S;
  const int n = max(0, min(V, x_lo + P.S) - x_lo);
  const int cps = (n + E - 1) / E;  // units per row slice
  const int units = N * cps;
  const TT *base = reinterpret_cast<const TT *>(P.target) + (size_t)b * N * V + x_lo;
  const unsigned ni = neg_inf_word<DT>();
  auto issue = [&](int k, uint4 (&buf)[kChunkVecs]) {
    const int row = k / cps, c = k - row * cps;
    const TT *src = base + (size_t)row * V + (size_t)c * E;
    const int nu = min(E, n - c * E);
#pragma unroll
    for (int u = 0; u < kChunkVecs; ++u) {
      const int e = (lane + 32 * u) * VEC;
      buf[u] = e < nu ? ld_nc16(src + e) : make_uint4(ni, ni, ni, ni);
    }
  };
  auto finish = [&](int k, const uint4 (&buf)[kChunkVecs]) {
    const int row = k / cps, c = k - row * cps;
    const int nu = min(E, n - c * E);
    float2 pt = tree_unit_argmax<DT>(buf, nu);
    if (__float_as_int(pt.y) != 0x7fffffff) pt.y = __int_as_float(__float_as_int(pt.y) + c * E);
    if (lane == 0) tu[k] = pt;
  };
  uint4 b0[kChunkVecs], b1[kChunkVecs];
  int ka = warp;
  if (ka < units) issue(ka, b0);
  while (ka < units) {
    const int kb = ka + kPassWarps;
    if (kb < units) issue(kb, b1);
    finish(ka, b0);
    if (kb >= units) break;
    ka = kb + kPassWarps;
    if (ka < units) issue(ka, b0);
    finish(kb, b1);
  }
  __syncthreads();
  // the units of each row: the largest value (NaN if any), the lowest index
  for (int row = threadIdx.x; row < N; row += kPassThreads) {
    float M = -CUDART_INF_F;
    int I = 0x7fffffff;
    bool nan = false;
    for (int c = 0; c < cps; ++c) {
      const float2 pt = tu[row * cps + c];
      const int ic = __float_as_int(pt.y);
      nan |= isnan(pt.x);
      if (pt.x > M || (pt.x == M && ic < I)) {
        M = pt.x;
        I = ic;
      }
    }
    tp[row] = make_float2(nan ? CUDART_NAN_F : M, __int_as_float(I == 0x7fffffff ? I : x_lo + I));
  }
  if (threadIdx.x == 0) tsm.flags = 0;
  cluster_sync();  // 1: every CTA's row partials are written
  int flags = 0;
  if (rank == 0) {
    for (int k = warp; k < N; k += kPassWarps) {
      float2 pt = make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
      if (lane < (int)CS) pt = ld_dsmem_f2(dsmem_addr(&tp[k], lane));
      if (__any_sync(0xffffffffu, isnan(pt.x))) flags |= SV_ROW_NONFINITE;
      const float M = warp_max_nan(pt.x);
      const int I = warp_min_int(pt.x == M ? __float_as_int(pt.y) : 0x7fffffff);
      if (lane == 0) tsm.a[k] = I;
    }
  }
  cluster_sync();  // 2: CTA 0 has read every CTA's partials
  if (rank != 0) return;
  for (int k = threadIdx.x; k < N; k += kPassThreads) {
    const int par = __ldg(P.parent + (size_t)b * N + k);
    const int tok = __ldg(P.node_tokens + (size_t)b * N + k);
    tsm.par[k] = par;
    tsm.tok[k] = tok;
    if (k == 0 ? par != -1 : (par < 0 || par >= k)) flags |= SV_ROW_BAD_TREE;
    if (k > 0 && (tok < 0 || tok >= V)) flags |= SV_ROW_BAD_TOKEN;
  }
  if (flags) atomicOr(&tsm.flags, flags);
  __syncthreads();
  if (warp != 0) return;
  flags = tsm.flags;
  const int D = P.max_depth, W = D + 1;
  int32_t *op = P.out_path + (size_t)b * W;
  int32_t *ot = P.out_tokens + (size_t)b * W;
  if (flags) {
    for (int s = lane; s < W; s += 32) {
      ot[s] = -1;
      op[s] = -1;
    }
    if (lane == 0) {
      P.out_nacc[b] = 0;
      if (P.out_status) P.out_status[b] = flags;
    }
    return;
  }
  int cur = 0, d = 0;
  while (d < D) {
    const int a = tsm.a[cur];
    int found = -1;
    for (int c0 = cur + 1; c0 < N && found < 0; c0 += 32) {
      const int ci = c0 + lane;
      const bool m = ci < N && tsm.par[ci] == cur && tsm.tok[ci] == a;
      const unsigned bm = __ballot_sync(0xffffffffu, m);
      if (bm) found = c0 + __ffs(bm) - 1;
    }
    if (found < 0) break;
    if (lane == 0) tsm.path[d] = found;
    cur = found;
    ++d;
  }
  __syncwarp();
  if (lane < W) {
    op[lane] = lane < d ? tsm.path[lane] : -1;
    ot[lane] = lane < d ? tsm.tok[tsm.path[lane]] : (lane == d ? tsm.a[cur] : -1);
  }
  if (lane == 0) {
    P.out_nacc[b] = d;
    if (P.out_status) P.out_status[b] = 0;
  }
}

}  // namespace sv
