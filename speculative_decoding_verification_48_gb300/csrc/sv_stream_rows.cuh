// Row decisions of the streaming kernel, run by the decider warp.
//
// Chain rows ("論文解説: Speculative Sampling", §技術的詳細 ステップ3: accept iff
// u * q(x) < p(x), in order, stop at the first rejection;
// §修正付き棄却サンプリング: draw from norm(max(0, p - q)); §期待される高速化:
// gamma + 1 tokens, so all-accepted rows draw a bonus token from p_gamma);
// greedy rows ("投機的デコーディングとは？" §ドラフト生成と並列検証の仕組み);
// token trees (SpecInfer explainer §推論方法: walk from the root along
// children whose token is the parent's top token).
#pragma once

#include "sv_stream_decide.cuh"

namespace sv {

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
  const size_t row_stride = (size_t)P.tilesMax;
  const float2 *tbase = P.partT + (size_t)b * P.rows * row_stride;

  // 1. merge every row read, one lane per row
  if (!badT) {
    for (int r = lane; r < nrows; r += 32) {
      const int tiles = r < G1 ? P.tilesT : P.tilesD;
      const float2 *pp = tbase + (size_t)r * row_stride;
      if (greedy) {
        const float2 mi = lane_merge_argmax(pp, tiles);
        sm.rowM[r] = mi.x;
        sm.rowI[r] = __float_as_int(mi.y);
      } else {
        const float2 mz = lane_merge_softmax(pp, tiles, c);
        sm.rowM[r] = mz.x;
        sm.rowZ[r] = mz.y;
      }
    }
  }
  __syncwarp();

  // 2. accept tests, one lane per draft position, and the first-reject scan
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
      float lq = 0.f;
      if (PROBS) {
        q = __ldg(reinterpret_cast<const float *>(P.draft) + ((size_t)b * g + i) * V + x);
      } else {
        lq = Elt<DDT>::load1(reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + i) * V + x);
      }
      const float ui = __ldg(P.unif + (size_t)b * G1 + i);
      p = ex2((lp - sm.rowM[i]) * c) / sm.rowZ[i];
      if (!PROBS) q = ex2((lq - sm.rowM[G1 + i]) * c) / sm.rowZ[G1 + i];
      acc = ui * q < p;
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

  // 3. outputs; bonus draw from p_gamma straight from its partials
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
        const size_t ro = ((size_t)b * P.rows + g) * row_stride;
        const int k = warp_sample_row<TDT>(tgt + (size_t)g * V, P.partT + ro, P.partA + ro * kCW,
                                           P.tilesT, V, sm.rowM[g], c,
                                           __ldg(P.unif + (size_t)b * G1 + g));
        if (lane == 0) ot[g] = k;
      } else {
        residual = true;
      }
    }
  }
  __syncwarp();

  // 4. publish: the residual row's Phase-B tiles, or mark the row done
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
      const unsigned base = atomicAdd(&P.hdr->q_reserved, (unsigned)P.tilesB);
      fence_acq_rel_gpu();  // the decision record before the queue items
      for (int t = 0; t < P.tilesB; ++t)
        st_relaxed_u32(P.qitems + base + t, pack_item(b, t, P.tilesB, j));
    } else {
      P.row_done[b] = 1;
    }
    fence_acq_rel_gpu();  // items / done flag before the decision count
    atomicAdd(&P.hdr->decisions_done, 1u);
  }
  __syncwarp();
}

// After the last Phase-B tile of a rejected row: crossing tile of u * R, its
// crossing warp slice, and a rescan of that slice.
template <int TDT, int DDT, bool PROBS>
__device__ void stream_finalize(const SParams &P, int b) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  using TBk = TileB<TDT, DDT>;
  constexpr int SLICE = TBk::kSlice, PER = SLICE / 32;
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
  const float *pt = P.partBT + (size_t)b * P.tilesB;
  auto wt = [&](int i) { return __ldcg(pt + i); };
  float R = 0.f;
  for (int i = lane; i < P.tilesB; i += 32) R += wt(i);
  R = warp_sum(R);
  const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)b * G1 + j) * V;
  int32_t *ot = P.out_tokens + (size_t)b * G1;
  if (isnan(R) || isinf(R)) {
    warp_error_row(P, b, SV_ROW_NONFINITE, G1, ot, nullptr);
  } else {
    int k;
    if (!(R > 0.f)) {
      // zero residual mass: draw from p_j
      const size_t ro = ((size_t)b * P.rows + j) * (size_t)P.tilesMax;
      k = warp_sample_row<TDT>(prow, P.partT + ro, P.partA + ro * kCW, P.tilesT, V, d.Mp, d.c,
                               d.u);
    } else {
      const float target = d.u * R;
      float base = 0.f;
      int t = warp_prefix_cross(P.tilesB, target, wt, base);
      if (t < 0) t = 0;
      const float *pw = P.partB + ((size_t)b * P.tilesB + t) * kCW;
      float base2 = 0.f;
      int w = warp_prefix_cross(kCW, target - base, [&](int i) { return __ldcg(pw + i); }, base2);
      if (w < 0) w = 0;
      const int x0 = t * TBk::kElems + w * SLICE;
      const int n = min(SLICE, V - x0);
      float a[PER], q[PER];
      lane_chunk_load<TDT, PER>(prow + x0, n, -CUDART_INF_F, a);
      lane_chunk_load<DDT, PER>(reinterpret_cast<const DTy *>(P.draft) +
                                    ((size_t)b * g + j) * V + x0,
                                n, PROBS ? 0.f : -CUDART_INF_F, q);
#pragma unroll
      for (int e = 0; e < PER; ++e) a[e] = residual_term<PROBS>(a[e], q[e], d);
      k = x0 + warp_rescan_regs<PER>(a, base + base2, target);
    }
    if (lane == 0) {
      ot[j] = k;
      if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
    }
  }
  __syncwarp();
  if (lane == 0) {
    fence_acq_rel_gpu();
    P.row_done[b] = 1;
  }
}

template <int DT>
__device__ void stream_decide_tree(const SParams &P, int b, StreamSmem &sm) {
  const int N = P.N, V = P.V, D = P.max_depth;
  const int lane = lane_id();
  const float2 *tbase = P.partT + (size_t)b * P.rows * P.tilesMax;
  int flags = 0;
  for (int r = lane; r < N; r += 32) {
    const float2 mi = lane_merge_argmax(tbase + (size_t)r * P.tilesMax, P.tilesT);
    sm.a[r] = __float_as_int(mi.y);
    if (isnan(mi.x)) flags |= SV_ROW_NONFINITE;
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
    fence_acq_rel_gpu();
    P.row_done[b] = 1;
    atomicAdd(&P.hdr->decisions_done, 1u);
  }
  __syncwarp();
}

}  // namespace sv
