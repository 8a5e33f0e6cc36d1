// Decision pass: one group of H CTAs per batch row (one CTA per tree).
//
// Chain rows ("論文解説: Speculative Sampling", §技術的詳細 ステップ3: accept
// draft i iff u_i q_i(x_i) < p_i(x_i), in order, stop at the first
// rejection; §修正付き棄却サンプリング: the replacement is drawn from
// norm(max(0, p_j - q_j)); §期待される高速化: gamma + 1 tokens per round, so a
// row whose drafts all pass draws a bonus token from p_gamma).  Greedy rows
// ("投機的デコーディングとは？" §ドラフト生成と並列検証の仕組み) accept while the
// draft is the target's top token and emit the top token at the first
// mismatch.  Trees (SpecInfer explainer, §技術の仕組み › 基本アイデア and
// §推論方法) walk from the root along the child whose token is the current
// node's top token.
#pragma once

#include "sv_pass_stats.cuh"

namespace sv {

struct DecideSmem {
  float rowM[kMaxRows], rowZ[kMaxRows];
  int rowI[kMaxRows];
  int j, status, last;
  float tot[kPassWarps];  // the rescan: each warp's share of the crossing chunk's mass
  int lastp[kPassWarps];  // ... and its last index of positive mass (-1: none)
  int k;                  // the drawn token
  // per warp: the p and q halves of one residual chunk, copied in by cp.async
  // (q may take one 16-byte block more: its vectors rebuilt from blocks of
  // its own grid)
  alignas(16) unsigned char stage[kPassWarps][2 * kResidBytes + 16];
};

struct TreeSmem {
  int a[SV_MAX_TREE_NODES], par[SV_MAX_TREE_NODES], tok[SV_MAX_TREE_NODES];
  int path[32];
  int flags;
};

// Writes an invalid row: every token (and path entry) -1, no draft accepted.
// Out of line, like the other paths a verifying row rarely takes: the decide
// kernel's common path then lies in fewer instruction-cache lines, which
// matters because each call's logit stream evicts its code from L2.
static __device__ __noinline__ void pass_error_row(const PassParams &P, int b, int status, int width,
                                               int32_t *tok, int32_t *path) {
  for (int s = lane_id(); s < width; s += 32) {
    tok[s] = -1;
    if (path) path[s] = -1;
  }
  if (lane_id() == 0) {
    P.out_nacc[b] = 0;
    if (P.out_status) P.out_status[b] = status;
  }
}

// The bytes [s, s + 16) of the 32-byte concatenation (lo, hi), s an even
// byte offset below 16 (uniform across the warp).
__device__ __forceinline__ uint4 bytes_at(const uint4 &lo, const uint4 &hi, int s) {
  const unsigned c[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const unsigned r = (unsigned)(s & 3) * 8u;
  unsigned o[4];
  switch (s >> 2) {
#define SV_BYTES_AT(W)                                                            \
  case W:                                                                          \
    _Pragma("unroll") for (int i = 0; i < 4; ++i)                                  \
      o[i] = r ? __funnelshift_r(c[W + i], c[W + i + 1], r) : c[W + i];             \
    break;
    SV_BYTES_AT(0)
    SV_BYTES_AT(1)
    SV_BYTES_AT(2)
    default:
      _Pragma("unroll") for (int i = 0; i < 4; ++i)
        o[i] = r ? __funnelshift_r(c[3 + i], c[3 + i + 1], r) : c[3 + i];
      break;
#undef SV_BYTES_AT
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// The same for 8-byte vectors: bytes [s, s + 8) of (lo, hi), s even, < 8.
__device__ __forceinline__ uint2 bytes_at(const uint2 &lo, const uint2 &hi, int s) {
  const unsigned r = (unsigned)(s & 3) * 8u;
  if (s < 4) return r ? make_uint2(__funnelshift_r(lo.x, lo.y, r), __funnelshift_r(lo.y, hi.x, r))
                      : lo;
  return r ? make_uint2(__funnelshift_r(lo.y, hi.x, r), __funnelshift_r(hi.x, hi.y, r))
           : make_uint2(lo.y, hi.x);
}
__device__ __forceinline__ uint4 shfl_vec(const uint4 &v, int src) {
  return make_uint4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                    __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}
__device__ __forceinline__ uint2 shfl_vec(const uint2 &v, int src) {
  return make_uint2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}
__device__ __forceinline__ uint4 shfl_down_vec(const uint4 &v) {
  return make_uint4(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1),
                    __shfl_down_sync(0xffffffffu, v.z, 1), __shfl_down_sync(0xffffffffu, v.w, 1));
}
__device__ __forceinline__ uint2 shfl_down_vec(const uint2 &v) {
  return make_uint2(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1));
}

// The lanes' vectors of a row whose own vector grid is shifted by mq bytes
// (0 < mq < the vector width) from the grid they are read on: vector i of
// the warp (i = lane + 32 u) starts at byte `a0 + i * kB`.  Each lane loads
// the aligned block under its vector's first byte; the block after it is the
// next lane's (the next group's lane 0 for lane 31, and one more load after
// the last group), so each vector costs one aligned load and two shuffles
// of its words.  Blocks that hold no byte of [lo, hi) are not loaded (their
// slots are masked by the caller).
template <class R, int KVECS>
__device__ __forceinline__ void load_realigned(const char *a0, int mq, const char *lo,
                                               const char *hi, R (&out)[KVECS]) {
  constexpr int kB = (int)sizeof(R);
  const int lane = lane_id();
  R blk[KVECS];
#pragma unroll
  for (int u = 0; u < KVECS; ++u) {
    const char *bq = a0 + (ptrdiff_t)(lane + 32 * u) * kB - mq;
    if (bq + kB > lo && bq < hi) {
      if constexpr (kB == 16) blk[u] = ld_nc16(bq);
      else blk[u] = ld_nc8(bq);
    } else {
      blk[u] = R{};
    }
  }
  R ext = R{};
  {
    const char *bq = a0 + (ptrdiff_t)(32 * KVECS) * kB - mq;
    if (lane == 31 && bq + kB > lo && bq < hi) {
      if constexpr (kB == 16) ext = ld_nc16(bq);
      else ext = ld_nc8(bq);
    }
  }
#pragma unroll
  for (int u = 0; u < KVECS; ++u) {
    R nb = shfl_down_vec(blk[u]);
    const R first_next = shfl_vec(u + 1 < KVECS ? blk[(u + 1) % KVECS] : ext, u + 1 < KVECS ? 0 : 31);
    if (lane == 31) nb = first_next;
    out[u] = bytes_at(blk[u], nb, mq);
  }
}

// Chain rows.  Every CTA of the row merges the partials it needs and makes
// the decision (cheap, from L2); CTA h = 0 writes the diagnostics and, for
// greedy, bonus and invalid rows, the outputs.  A rejected row's residual
// sweep is split over the H CTAs; the last to finish draws the token.  Every
// step issues all of its loads at once, so the row costs a handful of
// dependent round trips: gathers (before the wait on the stats kernel),
// partials, sweep, arrival, residual sums, rescan.
template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
__device__ void decide_chain_row(const PassParams &P, int b, int h, DecideSmem &sm) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int g = P.gamma, G1 = g + 1, V = P.V;
  const int lane = lane_id(), warp = warp_id();
  int32_t *ot = P.out_tokens + (size_t)b * G1;
  const TT *tgt = reinterpret_cast<const TT *>(P.target) + (size_t)b * G1 * V;
  // 0. inputs only (none is written by the stats kernel): issued before the
  // wait so their latency overlaps the stats kernel's tail
  const float T = (MODE == MODE_CHAIN) ? __ldg(P.temps + b) : 0.f;
  const bool badT = bad_temperature(T);
  const bool greedy = T <= 0.f;
  const float c = kLog2e / T;
  if ((badT || greedy) && h != 0) return;  // nothing to sweep
  const int i = lane;
  const bool act = warp == 0 && i < g;
  int x = 0;
  bool tok_ok = false;
  float lp = 0.f, lq = 0.f, qp = 0.f, ui = 0.f;
  // the categorical draw, used by every warp of whichever CTA draws the token
  const float ug = (!badT && !greedy) ? __ldg(P.unif + (size_t)b * G1 + g) : 0.f;
  if (act) {
    x = __ldg(P.draft_tokens + (size_t)b * g + i);
    tok_ok = x >= 0 && x < V;
    if (!badT && !greedy && tok_ok) {
      lp = Elt<TDT>::load1(tgt + (size_t)i * V + x);
      if (PROBS) qp = __ldg(reinterpret_cast<const float *>(P.draft) + ((size_t)b * g + i) * V + x);
      else lq = Elt<DDT>::load1(reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + i) * V + x);
      ui = __ldg(P.unif + (size_t)b * G1 + i);
    }
  }
  // 1a. Softmax rows of at most 64 chunks are merged as their partials
  // arrive, without waiting for the whole stats grid: every partial of the
  // row pair must carry this call's tag (bounded polling; if the bound runs
  // out, the block falls back to the wait and merges again).  A tagged
  // partial was written after the stats kernel's own wait, so the work
  // before this call is complete; the fence orders this kernel's later
  // writes after that observation.
  const int nrows = greedy ? G1 : (PROBS ? G1 : 2 * g + 1);
  const Part *pb = P.part + (size_t)b * P.rows * P.cMax;
  bool polled = false;
  if (P.poll && !badT && !greedy && P.cT <= 64 && (PROBS || P.cD <= 64)) {
    bool ok = true;
    for (int r = warp; r < nrows; r += 2 * kPassWarps) {
      const int r2 = r + kPassWarps;
      const int ca = r < G1 ? P.cT : P.cD, cb = r2 < G1 ? P.cT : P.cD;
      float2 za, zb = make_float2(0.f, 0.f);
      ok = warp_rows_softmax2_poll(pb + (size_t)r * P.cMax, ca,
                                   r2 < nrows ? pb + (size_t)r2 * P.cMax : nullptr, cb, c,
                                   P.part_tag, kPollSpins, za, zb);
      if (!ok) break;
      if (lane == 0) {
        sm.rowM[r] = za.x; sm.rowZ[r] = za.y;
        if (r2 < nrows) { sm.rowM[r2] = zb.x; sm.rowZ[r2] = zb.y; }
      }
    }
    polled = __syncthreads_and(ok);
    if (polled) asm volatile("fence.acq_rel.gpu;" ::: "memory");
  }
  bool claim_err = false;
  if (!polled) {
    grid_dependency_wait();
    if (warp == 0) claim_err = __ldcg(P.claim_err) == __ldcg(P.epoch_cur);
  }
  if (badT) {
    if (warp == 0) {
      pass_error_row(P, b, SV_ROW_BAD_TEMPERATURE, G1, ot, nullptr);
      if (MODE == MODE_CHAIN && P.out_diag)
        for (int k = lane; k < g; k += 32)
          reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  // 1b. otherwise, after the wait: each warp takes rows warp, warp + 8, ...
  // two at a time
  for (int r = warp; !polled && r < nrows; r += 2 * kPassWarps) {
    const int r2 = r + kPassWarps;
    const int ca = r < G1 ? P.cT : P.cD, cb = r2 < G1 ? P.cT : P.cD;
    if (greedy) {
      const float2 ma = warp_row_argmax(pb + (size_t)r * P.cMax, ca);
      float2 mb = make_float2(0.f, 0.f);
      if (r2 < nrows) mb = warp_row_argmax(pb + (size_t)r2 * P.cMax, cb);
      if (lane == 0) {
        sm.rowM[r] = ma.x; sm.rowI[r] = __float_as_int(ma.y);
        if (r2 < nrows) { sm.rowM[r2] = mb.x; sm.rowI[r2] = __float_as_int(mb.y); }
      }
    } else {
      float2 za, zb = make_float2(0.f, 0.f);
      if (ca <= 256 && cb <= 256) {
        warp_rows_softmax2(pb + (size_t)r * P.cMax, ca,
                           r2 < nrows ? pb + (size_t)r2 * P.cMax : nullptr, cb, c, za, zb);
      } else {
        za = warp_row_softmax(pb + (size_t)r * P.cMax, ca, c);
        if (r2 < nrows) zb = warp_row_softmax(pb + (size_t)r2 * P.cMax, cb, c);
      }
      if (lane == 0) {
        sm.rowM[r] = za.x; sm.rowZ[r] = za.y;
        if (r2 < nrows) { sm.rowM[r2] = zb.x; sm.rowZ[r2] = zb.y; }
      }
    }
  }
  __syncthreads();
  // 2. accept tests (one lane per draft) and the first-reject scan
  if (warp == 0) {
    const unsigned gmask = (g >= 32) ? 0xffffffffu : ((1u << g) - 1u);
    int status, j;
    bool nf = false;
    if (greedy) {
      for (int r = lane; r < G1; r += 32) nf |= isnan(sm.rowM[r]);
      const bool match = act && tok_ok && x == sm.rowI[i];
      const unsigned mm = __ballot_sync(0xffffffffu, match) & gmask;
      const unsigned badtok = __ballot_sync(0xffffffffu, act && !tok_ok);
      const unsigned nfm = __ballot_sync(0xffffffffu, nf);
      j = (~mm & gmask) ? __ffs(~mm & gmask) - 1 : g;
      status = (badtok ? SV_ROW_BAD_TOKEN : 0) | (nfm ? SV_ROW_NONFINITE : 0);
      if (MODE == MODE_CHAIN && act && P.out_diag)
        reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      float p = 0.f, q = 0.f;
      bool acc = false;
      if (act && tok_ok) {
        p = ex2((lp - sm.rowM[i]) * c) / sm.rowZ[i];
        q = PROBS ? qp : ex2((lq - sm.rowM[G1 + i]) * c) / sm.rowZ[G1 + i];
        acc = ui * q < p;
      }
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
      if (h == 0 && act && P.out_diag) {
        const float ap = (q > 0.f) ? fminf(1.f, p / q) : (p > 0.f ? 1.f : 0.f);
        reinterpret_cast<float4 *>(P.out_diag)[(size_t)b * g + i] = make_float4(p, q, ap, 0.f);
      }
    }
    // a stats kernel that could not finish its claims leaves partials unset
    if (claim_err) status = SV_ROW_TIMEOUT;
    if (lane == 0) { sm.j = j; sm.status = status; }
  }
  __syncthreads();
  const int j = sm.j, status = sm.status;
  // 3. rows finished by CTA 0 alone: invalid, greedy, bonus
  const bool sweep = !status && !greedy && j < g;
  if (!sweep) {
    if (h != 0 || warp != 0) return;
    if (status) {
      pass_error_row(P, b, status, G1, ot, nullptr);
      return;
    }
    int tok_j = 0;
    if (greedy) {
      tok_j = sm.rowI[j];
    } else {
      const Part *pr = pb + (size_t)g * P.cMax;
      const TT *brow = tgt + (size_t)g * V;
      tok_j = warp_sample_softmax_row<TDT>(brow, pr, P.cT, V, sm.rowM[g], c, ug,
                                           P.unaligned ? row_offset16<TDT>(brow) : 0);
    }
    for (int s = lane; s < G1; s += 32)
      ot[s] = s < j ? x : (s == j ? tok_j : -1);  // lane s holds draft token s
    if (lane == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
    }
    return;
  }
  // 4-5.  Rows on the 16-byte grid take the first form (no offsets, no
  // masks); rows off it the second.
  if constexpr (!UNAL) {
    // 4. residual sweep of the row pair (p_j, q_j), chunks [c0, c1) of this CTA
    using PC = PairChunk<TDT, DDT>;
    ResidCoef rk;
    rk.c = c;
    rk.Mp = sm.rowM[j];
    rk.lzp = log2f(sm.rowZ[j]);
    rk.Mq = PROBS ? 0.f : sm.rowM[G1 + j];
    rk.lzq = PROBS ? 0.f : log2f(sm.rowZ[G1 + j]);
    const float Mp = sm.rowM[j];
    const TT *prow = tgt + (size_t)j * V;
    const DTy *qrow = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + j) * V;
    float *rs = P.resid + (size_t)b * P.cR;
    const int c0 = (int)((long long)h * P.cR / P.H), c1 = (int)((long long)(h + 1) * P.cR / P.H);
    // Each warp takes chunk pairs (ch, ch + 8), ch = c0 + warp + 16 i: the
    // first chunk is loaded into registers, the second is copied into this
    // warp's shared-memory stage by cp.async, and both are in flight before the
    // first residual term (one memory round trip per pair).  Every lane reads
    // back only the vectors it copied itself, so its own wait suffices.
    using RA = RawVec<TDT, PC::kVec>;
    using RQ = RawVec<DDT, PC::kVec>;
    typename RA::R *sa = reinterpret_cast<typename RA::R *>(sm.stage[warp]);
    typename RQ::R *sq = reinterpret_cast<typename RQ::R *>(sm.stage[warp] + kResidBytes);
    RA ra[PC::kVecs];
    RQ rq[PC::kVecs];
    auto chunk_sum = [&](int n) {
      unsigned long long s2 = 0ull;  // (+0, +0)
  #pragma unroll
      for (int u = 0; u < PC::kVecs; ++u) {
        const int e = (lane + 32 * u) * PC::kVec;
        if (e < n) {
          float a[PC::kVec], q[PC::kVec];
          ra[u].unpack(a);
          rq[u].unpack(q);
  #pragma unroll
          for (int t = 0; t < PC::kVec; t += 2) {
            const float2 r = resid_pair<PROBS>(a[t], a[t + 1], q[t], q[t + 1], rk);
            s2 = f2_add(s2, f2_pack(r.x, r.y));
          }
        }
      }
      const float2 sp = f2_unpack(s2);
      return warp_sum(sp.x + sp.y);
    };
    // 8-byte vectors (a 16-bit target beside fp32 draft rows) measured slower
    // staged than one register-held chunk at a time, so only pairs of 16-byte
    // vectors take the stage
    constexpr bool kStage = RA::kB == 16 && RQ::kB == 16;
    for (int ch = c0 + warp; ch < c1; ch += (kStage ? 2 : 1) * kPassWarps) {
      const int chB = ch + kPassWarps;
      const int nB = kStage && chB < c1 ? min(PC::kElems, V - chB * PC::kElems) : 0;
      if (nB > 0) {
        const int xB = chB * PC::kElems;
  #pragma unroll
        for (int u = 0; u < PC::kVecs; ++u) {
          const int e = (lane + 32 * u) * PC::kVec;
          if (e < nB) {
            cp_async<RA::kB>(sa + lane + 32 * u, prow + xB + e);
            cp_async<RQ::kB>(sq + lane + 32 * u, qrow + xB + e);
          }
        }
        cp_async_commit();
      }
      const int x0 = ch * PC::kElems;
      const int n = min(PC::kElems, V - x0);
  #pragma unroll
      for (int u = 0; u < PC::kVecs; ++u) {
        const int e = (lane + 32 * u) * PC::kVec;
        if (e < n) {
          ra[u].load(prow + x0 + e);
          rq[u].load(qrow + x0 + e);
        }
      }
      const float s = chunk_sum(n);
      if (lane == 0) rs[ch] = s;
      if (nB > 0) {
        cp_async_wait_all();
  #pragma unroll
        for (int u = 0; u < PC::kVecs; ++u) {
          if ((lane + 32 * u) * PC::kVec < nB) {
            ra[u].r = sa[lane + 32 * u];
            rq[u].r = sq[lane + 32 * u];
          }
        }
        const float sB = chunk_sum(nB);
        if (lane == 0) rs[chB] = sB;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // a block that merged by polling waits here: the stats kernel zeroes
      // done[] before its first partial, and the stats grid has long finished
      // by now, so this returns at once
      if (polled) grid_dependency_wait();
      // one acquire-release add: it publishes this CTA's chunk sums (ordered
      // before it by the barrier above) and, in the last CTA, acquires the
      // other CTAs' sums
      unsigned prev;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                   : "=r"(prev) : "l"(P.done + b) : "memory");
      sm.last = (prev == (unsigned)P.H - 1u);
    }
    __syncthreads();
    if (!sm.last) return;
    // 5. the last CTA.  Every warp locates the crossing chunk of u * R from
    // the same chunk sums; the chunk is rescanned by all eight warps, each
    // over its eighth, and a prefix over the eight shares picks the warp that
    // holds the crossing.  Warp 0, whose lanes hold the draft tokens, writes
    // the row's outputs.
    const float u = ug;
    float R = 0.f, base = 0.f;
    const int t = warp_chunk_cross(P.cR, [&](int k) { return __ldcg(rs + k); }, u, R, base);
    if (isnan(R) || isinf(R) || !(R > 0.f)) {
      if (warp != 0) return;
      if (!(R > 0.f) && !isnan(R)) {
        // no residual mass (p_j == q_j up to rounding): draw from p_j
        const int k = warp_sample_softmax_row<TDT>(prow, pb + (size_t)j * P.cMax, P.cT, V, Mp, c, u);
        for (int s = lane; s < G1; s += 32)
          ot[s] = s < j ? x : (s == j ? k : -1);  // lane s holds draft token s
        if (lane == 0) {
          P.out_nacc[b] = j;
          if (P.out_status) P.out_status[b] = 0;
          if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
        }
      } else {
        pass_error_row(P, b, SV_ROW_NONFINITE, G1, ot, nullptr);
      }
      return;
    }
    const float target = u * R;
    constexpr int SUB = PC::kElems / kPassWarps, SPER = SUB / 32;
    static_assert(SPER % 2 == 0, "pairs of elements per lane");
    const int xs = t * PC::kElems + warp * SUB;
    float a[SPER], qv[SPER];
    lane_row_load<TDT, SPER>(prow, xs, V, -CUDART_INF_F, a);
    lane_row_load<DDT, SPER>(qrow, xs, V, PROBS ? 0.f : -CUDART_INF_F, qv);
    float ls = 0.f;
    int lpos = -1;
  #pragma unroll
    for (int e = 0; e < SPER; e += 2) {
      const float2 r = resid_pair<PROBS>(a[e], a[e + 1], qv[e], qv[e + 1], rk);
      a[e] = r.x;
      a[e + 1] = r.y;
    }
  #pragma unroll
    for (int e = 0; e < SPER; ++e) {
      ls += a[e];
      if (a[e] > 0.f) lpos = lane * SPER + e;
    }
    const float wt = warp_sum(ls);
    const int wl = warp_max_int(lpos);
    if (lane == 0) {
      sm.tot[warp] = wt;
      sm.lastp[warp] = wl >= 0 ? xs + wl : -1;
    }
    __syncthreads();
    float bw = base;
    int hw = -1;
    for (int w = 0; w < kPassWarps && hw < 0; ++w) {
      if (bw + sm.tot[w] > target) hw = w;
      else bw += sm.tot[w];
    }
    if (warp == hw) {
      const int kl = warp_rescan<SPER>(a, bw, target);
      if (lane == 0) sm.k = xs + kl;
    } else if (hw < 0 && warp == 0 && lane == 0) {
      // rounding left no crossing: the last element of positive mass
      int kk = t * PC::kElems;
      for (int w = 0; w < kPassWarps; ++w)
        if (sm.lastp[w] >= 0) kk = sm.lastp[w];
      sm.k = kk;
    }
    __syncthreads();
    if (warp != 0) return;
    const int k = sm.k;
    for (int s = lane; s < G1; s += 32)
      ot[s] = s < j ? x : (s == j ? k : -1);  // lane s holds draft token s
    if (lane == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
      if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
    }
  } else {
    // 4. residual sweep of the row pair (p_j, q_j), chunks [c0, c1) of this CTA.
    // Chunk ch covers vocabulary indices [ch kElems - off, (ch + 1) kElems -
    // off), off being the target row's elements before its first vector
    // boundary (0 when rows start on 16-byte boundaries), so the target row's
    // vectors are aligned; the draft row's are too when its own offset agrees,
    // else its elements are read one at a time.  Slots outside the row are
    // masked: p = 0 there, so they add no mass.
    using PC = PairChunk<TDT, DDT>;
    using RA = RawVec<TDT, PC::kVec>;
    using RQ = RawVec<DDT, PC::kVec>;
    ResidCoef rk;
    rk.c = c;
    rk.Mp = sm.rowM[j];
    rk.lzp = log2f(sm.rowZ[j]);
    rk.Mq = PROBS ? 0.f : sm.rowM[G1 + j];
    rk.lzq = PROBS ? 0.f : log2f(sm.rowZ[G1 + j]);
    const float Mp = sm.rowM[j];
    const TT *prow = tgt + (size_t)j * V;
    const DTy *qrow = reinterpret_cast<const DTy *>(P.draft) + ((size_t)b * g + j) * V;
    const int off = UNAL ? (int)((reinterpret_cast<uintptr_t>(prow) & (RA::kB - 1)) / sizeof(TT))
                         : 0;
    const int mq = (int)(reinterpret_cast<uintptr_t>(qrow - off) & (RQ::kB - 1));  // bytes
    const bool qa = !UNAL || mq == 0;
    float *rs = P.resid + (size_t)b * P.cR;
    const int c0 = (int)((long long)h * P.cR / P.H), c1 = (int)((long long)(h + 1) * P.cR / P.H);
    // Each warp takes chunk pairs (ch, ch + 8), ch = c0 + warp + 16 i: the
    // first chunk is loaded into registers, the second is copied into this
    // warp's shared-memory stage by cp.async, and both are in flight before the
    // first residual term (one memory round trip per pair).  Every lane reads
    // back only the vectors it copied itself, so its own wait suffices.
    typename RA::R *sa = reinterpret_cast<typename RA::R *>(sm.stage[warp]);
    typename RQ::R *sq = reinterpret_cast<typename RQ::R *>(sm.stage[warp] + kResidBytes);
    RA ra[PC::kVecs];
    RQ rq[PC::kVecs];
    auto chunk_sum = [&](int x0) {
      unsigned long long s2 = 0ull;  // (+0, +0)
  #pragma unroll
      for (int u = 0; u < PC::kVecs; ++u) {
        const int x = x0 + (lane + 32 * u) * PC::kVec;
        if (x < V && (!UNAL || x + PC::kVec > 0)) {
          float a[PC::kVec], q[PC::kVec];
          ra[u].unpack(a);
          rq[u].unpack(q);
          if (UNAL && (x < 0 || x + PC::kVec > V)) {
  #pragma unroll
            for (int t = 0; t < PC::kVec; ++t)
              if (x + t < 0 || x + t >= V) {
                a[t] = -CUDART_INF_F;  // p = 0: no mass
                q[t] = PROBS ? 0.f : -CUDART_INF_F;  // a neighbour's NaN stays out
              }
          }
  #pragma unroll
          for (int t = 0; t < PC::kVec; t += 2) {
            const float2 r = resid_pair<PROBS>(a[t], a[t + 1], q[t], q[t + 1], rk);
            s2 = f2_add(s2, f2_pack(r.x, r.y));
          }
        }
      }
      const float2 sp = f2_unpack(s2);
      return warp_sum(sp.x + sp.y);
    };
    // 8-byte vectors (a 16-bit target beside fp32 draft rows) measured slower
    // staged than one register-held chunk at a time, so only pairs of 16-byte
    // vectors take the stage
    const bool stage = RA::kB == 16 && RQ::kB == 16;
    const int stride = (stage ? 2 : 1) * kPassWarps;
    for (int ch = c0 + warp; ch < c1; ch += stride) {
      const int chB = ch + kPassWarps;
      const bool useB = stage && chB < c1;
      if (useB) {
        const int xB = chB * PC::kElems - off;
  #pragma unroll
        for (int u = 0; u < PC::kVecs; ++u) {
          const int x = xB + (lane + 32 * u) * PC::kVec;
          if (x < V && (!UNAL || x + PC::kVec > 0)) {
            cp_async<RA::kB>(sa + lane + 32 * u, prow + x);
            if (qa) cp_async<RQ::kB>(sq + lane + 32 * u, qrow + x);
          }
        }
        if (!qa) {
          // the draft row's aligned blocks under the vectors, one more after
          // them (blocks that hold no byte of the row are not copied: the
          // slots they would fill are masked)
          const char *q0 = reinterpret_cast<const char *>(qrow + xB) - mq;
          const char *qlo = reinterpret_cast<const char *>(qrow);
          const char *qhi = reinterpret_cast<const char *>(qrow + V);
          for (int i = lane; i <= 32 * PC::kVecs; i += 32) {
            const char *bq = q0 + (ptrdiff_t)i * RQ::kB;
            if (bq + RQ::kB > qlo && bq < qhi) cp_async<RQ::kB>(sq + i, bq);
          }
        }
        cp_async_commit();
      }
      const int x0 = ch * PC::kElems - off;
      if (!qa) {
        // the draft row's vectors are shifted from the target row's grid
        typename RQ::R qv[PC::kVecs];
        load_realigned<typename RQ::R, PC::kVecs>(
            reinterpret_cast<const char *>(qrow + x0), mq, reinterpret_cast<const char *>(qrow),
            reinterpret_cast<const char *>(qrow + V), qv);
  #pragma unroll
        for (int u = 0; u < PC::kVecs; ++u) rq[u].r = qv[u];
      }
  #pragma unroll
      for (int u = 0; u < PC::kVecs; ++u) {
        const int x = x0 + (lane + 32 * u) * PC::kVec;
        if (x < V && (!UNAL || x + PC::kVec > 0)) {
          ra[u].load(prow + x);
          if (qa) rq[u].load(qrow + x);
        }
      }
      const float s = chunk_sum(x0);
      if (lane == 0) rs[ch] = s;
      if (useB) {
        cp_async_wait_all();
        if (!qa) __syncwarp();  // a vector's second block was copied by the next lane
        const int xB = chB * PC::kElems - off;
  #pragma unroll
        for (int u = 0; u < PC::kVecs; ++u) {
          const int x = xB + (lane + 32 * u) * PC::kVec;
          if (x < V && (!UNAL || x + PC::kVec > 0)) {
            ra[u].r = sa[lane + 32 * u];
            rq[u].r = qa ? sq[lane + 32 * u]
                         : bytes_at(sq[lane + 32 * u], sq[lane + 32 * u + 1], mq);
          }
        }
        const float sB = chunk_sum(xB);
        if (lane == 0) rs[chB] = sB;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // a block that merged by polling waits here: the stats kernel zeroes
      // done[] before its first partial, and the stats grid has long finished
      // by now, so this returns at once
      if (polled) grid_dependency_wait();
      // one acquire-release add: it publishes this CTA's chunk sums (ordered
      // before it by the barrier above) and, in the last CTA, acquires the
      // other CTAs' sums
      unsigned prev;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                   : "=r"(prev) : "l"(P.done + b) : "memory");
      sm.last = (prev == (unsigned)P.H - 1u);
    }
    __syncthreads();
    if (!sm.last) return;
    // 5. the last CTA.  Every warp locates the crossing chunk of u * R from
    // the same chunk sums; the chunk is rescanned by all eight warps, each
    // over its eighth, and a prefix over the eight shares picks the warp that
    // holds the crossing.  Warp 0, whose lanes hold the draft tokens, writes
    // the row's outputs.
    const float u = ug;
    float R = 0.f, base = 0.f;
    const int t = warp_chunk_cross(P.cR, [&](int k) { return __ldcg(rs + k); }, u, R, base);
    if (isnan(R) || isinf(R) || !(R > 0.f)) {
      if (warp != 0) return;
      if (!(R > 0.f) && !isnan(R)) {
        // no residual mass (p_j == q_j up to rounding): draw from p_j
        const int k = warp_sample_softmax_row<TDT>(prow, pb + (size_t)j * P.cMax, P.cT, V, Mp, c, u,
                                                   P.unaligned ? row_offset16<TDT>(prow) : 0);
        for (int s = lane; s < G1; s += 32)
          ot[s] = s < j ? x : (s == j ? k : -1);  // lane s holds draft token s
        if (lane == 0) {
          P.out_nacc[b] = j;
          if (P.out_status) P.out_status[b] = 0;
          if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
        }
      } else {
        pass_error_row(P, b, SV_ROW_NONFINITE, G1, ot, nullptr);
      }
      return;
    }
    const float target = u * R;
    constexpr int SUB = PC::kElems / kPassWarps, SPER = SUB / 32;
    static_assert(SPER % 2 == 0, "pairs of elements per lane");
    const int xs = t * PC::kElems - off + warp * SUB;
    float a[SPER], qv[SPER];
    lane_row_load<TDT, SPER>(prow, xs, V, -CUDART_INF_F, a);
    lane_row_load<DDT, SPER>(qrow, xs, V, PROBS ? 0.f : -CUDART_INF_F, qv);
    float ls = 0.f;
    int lpos = -1;
  #pragma unroll
    for (int e = 0; e < SPER; e += 2) {
      const float2 r = resid_pair<PROBS>(a[e], a[e + 1], qv[e], qv[e + 1], rk);
      a[e] = r.x;
      a[e + 1] = r.y;
    }
  #pragma unroll
    for (int e = 0; e < SPER; ++e) {
      ls += a[e];
      if (a[e] > 0.f) lpos = lane * SPER + e;
    }
    const float wt = warp_sum(ls);
    const int wl = warp_max_int(lpos);
    if (lane == 0) {
      sm.tot[warp] = wt;
      sm.lastp[warp] = wl >= 0 ? xs + wl : -1;
    }
    __syncthreads();
    float bw = base;
    int hw = -1;
    for (int w = 0; w < kPassWarps && hw < 0; ++w) {
      if (bw + sm.tot[w] > target) hw = w;
      else bw += sm.tot[w];
    }
    if (warp == hw) {
      const int kl = warp_rescan<SPER>(a, bw, target);
      if (lane == 0) sm.k = xs + kl;
    } else if (hw < 0 && warp == 0 && lane == 0) {
      // rounding left no crossing: the last element of positive mass
      int kk = t * PC::kElems;
      for (int w = 0; w < kPassWarps; ++w)
        if (sm.lastp[w] >= 0) kk = sm.lastp[w];
      sm.k = kk;
    }
    __syncthreads();
    if (warp != 0) return;
    const int k = sm.k;
    for (int s = lane; s < G1; s += 32)
      ot[s] = s < j ? x : (s == j ? k : -1);  // lane s holds draft token s
    if (lane == 0) {
      P.out_nacc[b] = j;
      if (P.out_status) P.out_status[b] = 0;
      if (P.out_diag) P.out_diag[((size_t)b * g + j) * 4 + 3] = R;
    }
  }
}

// One tree per CTA: argmax of every node row, validation, then the walk.
template <int DT>
__device__ void decide_tree(const PassParams &P, int b, TreeSmem &sm) {
  const int N = P.N, V = P.V, D = P.max_depth;
  const int lane = lane_id(), warp = warp_id();
  if (threadIdx.x == 0) sm.flags = 0;
  __syncthreads();
  int flags = 0;
  const Part *pb = P.part + (size_t)b * N * P.cMax;
  // The tree arrays are inputs (the stats kernel writes neither): each
  // thread's first node is loaded before the merge, which hides its latency.
  const int n0 = threadIdx.x;
  int par0 = 0, tok0 = 0;
  if (n0 < N) {
    par0 = __ldg(P.parent + (size_t)b * N + n0);
    tok0 = __ldg(P.node_tokens + (size_t)b * N + n0);
  }
  // On polling calls the partials are merged as they arrive: every partial
  // a lane holds must carry this call's tag (bounded; if the bound runs out
  // anywhere in the CTA, the CTA takes the dependency wait and merges again).
  bool polled = false;
  if (P.poll && P.cT <= 32) {
    bool ok = true;
    for (int r0 = warp * 8; ok && r0 < N; r0 += kPassWarps * 8) {
      unsigned long long w[8][2];
      bool need[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        need[k] = r0 + k < N && lane < P.cT;
        w[k][0] = w[k][1] = 0ull;
      }
      for (int it = 0;; ++it) {
        bool pending = false;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (need[k]) part_poll(pb + (size_t)(r0 + k) * P.cMax + lane, w[k][0], w[k][1]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          need[k] = need[k] && !part_tagged(w[k][0], w[k][1], P.part_tag);
          pending |= need[k];
        }
        if (!__any_sync(0xffffffffu, pending)) break;
        if (it >= kPollSpins) {
          ok = false;
          break;
        }
        __nanosleep(128);
      }
      if (!ok) break;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = r0 + k;  // warp-uniform
        if (r < N) {
          const float v = lane < P.cT ? __uint_as_float((unsigned)w[k][0]) : -CUDART_INF_F;
          const int i = lane < P.cT ? (int)(unsigned)w[k][1] : 0x7fffffff;
          if (__any_sync(0xffffffffu, isnan(v))) flags |= SV_ROW_NONFINITE;
          const float M = warp_max_nan(v);
          const int I = warp_min_int(v == M ? i : 0x7fffffff);
          if (lane == 0) sm.a[r] = I;
        }
      }
    }
    polled = __syncthreads_and(ok);
    if (polled) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    else flags = 0;
  }
  if (!polled) {
    grid_dependency_wait();  // the stats kernel's partials are complete
    if (P.cT <= 32) {
      // Rows of at most 32 chunks: each lane holds one chunk partial of each
      // of 8 rows, all loaded at once, so a warp's group of 8 rows costs one
      // memory round trip.  The merge is that of warp_row_argmax: the largest
      // value, the lowest index among chunks holding it, NaN flags the row.
      for (int r0 = warp * 8; r0 < N; r0 += kPassWarps * 8) {
        float2 pt[8];
  #pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = r0 + k;
          pt[k] = (r < N && lane < P.cT)
                      ? part_value(pb + (size_t)r * P.cMax + lane)
                      : make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
        }
  #pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = r0 + k;  // warp-uniform
          if (r < N) {
            if (__any_sync(0xffffffffu, isnan(pt[k].x))) flags |= SV_ROW_NONFINITE;
            const float M = warp_max_nan(pt[k].x);
            const int I = warp_min_int(pt[k].x == M ? __float_as_int(pt[k].y) : 0x7fffffff);
            if (lane == 0) sm.a[r] = I;
          }
        }
      }
    } else {
      for (int r = warp; r < N; r += kPassWarps) {
        const float2 mi = warp_row_argmax(pb + (size_t)r * P.cMax, P.cT);
        if (lane == 0) sm.a[r] = __float_as_int(mi.y);
        if (isnan(mi.x)) flags |= SV_ROW_NONFINITE;
      }
    }
  }
  for (int n = n0; n < N; n += kPassThreads) {
    const int par = n == n0 ? par0 : __ldg(P.parent + (size_t)b * N + n);
    const int tok = n == n0 ? tok0 : __ldg(P.node_tokens + (size_t)b * N + n);
    sm.par[n] = par;
    sm.tok[n] = tok;
    if (n == 0 ? par != -1 : (par < 0 || par >= n)) flags |= SV_ROW_BAD_TREE;
    if (n > 0 && (tok < 0 || tok >= V)) flags |= SV_ROW_BAD_TOKEN;
  }
  // (a polled merge saw every partial of this call: no claim ran out)
  if (!polled && threadIdx.x == 0 && __ldcg(P.claim_err) == __ldcg(P.epoch_cur))
    flags |= SV_ROW_TIMEOUT;
  if (flags) atomicOr(&sm.flags, flags);
  __syncthreads();
  if (warp != 0) return;
  flags = sm.flags;
  const int W = D + 1;
  int32_t *op = P.out_path + (size_t)b * W;
  int32_t *ot = P.out_tokens + (size_t)b * W;
  if (flags) {
    pass_error_row(P, b, flags, W, ot, op);
    return;
  }
  int cur = 0, d = 0;
  while (d < D) {
    const int a = sm.a[cur];
    int found = -1;
    for (int base = cur + 1; base < N && found < 0; base += 32) {
      const int ci = base + lane;
      const bool m = ci < N && sm.par[ci] == cur && sm.tok[ci] == a;
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

// Draft-side draw, one warp per row ("論文解説: Speculative Sampling",
// §アルゴリズム Step 1: the draft token is drawn from softmax(draft logits / T);
// the draw is the inverse CDF in vocabulary order with the row's uniform,
// and T <= 0 takes the first argmax).  out_diag carries q(token).
template <int DT>
__device__ void decide_draft_row(const PassParams &P, int b) {
  using TT = typename Elt<DT>::T;
  const int lane = lane_id(), V = P.V;
  const float T = __ldg(P.temps + b);
  const TT *row = reinterpret_cast<const TT *>(P.target) + (size_t)b * V;
  const Part *pr = P.part + (size_t)b * P.cMax;
  int status = 0, tok = -1;
  float prob = 0.f;
  if (bad_temperature(T)) {
    status = SV_ROW_BAD_TEMPERATURE;
  } else if (T <= 0.f) {
    const float2 mi = warp_row_argmax(pr, P.cT);
    if (isnan(mi.x)) status = SV_ROW_NONFINITE;
    else tok = __float_as_int(mi.y);
  } else {
    const float c = kLog2e / T;
    const float2 mz = warp_row_softmax(pr, P.cT, c);
    if (!(mz.y > 0.f && mz.y <= 3.0e38f)) {
      status = SV_ROW_NONFINITE;
    } else {
      tok = warp_sample_softmax_row<DT>(row, pr, P.cT, V, mz.x, c, __ldg(P.unif + b),
                                        P.unaligned ? row_offset16<DT>(row) : 0);
      prob = ex2((Elt<DT>::load1(row + tok) - mz.x) * c) / mz.y;
    }
  }
  if (__ldcg(P.claim_err) == __ldcg(P.epoch_cur)) status = SV_ROW_TIMEOUT;
  if (lane == 0) {
    P.out_tokens[b] = status ? -1 : tok;
    if (P.out_diag) P.out_diag[b] = status ? 0.f : prob;
    if (P.out_status) P.out_status[b] = status;
  }
}

template <int MODE, int TDT, int DDT, bool PROBS, bool UNAL>
__global__ void __launch_bounds__(kPassThreads, UNAL ? 3 : 4) sv_decide_kernel(const PassParams P) {
  const int b = blockIdx.x / P.H, h = blockIdx.x - b * P.H;
  if (MODE == MODE_DRAFT) {
    grid_dependency_wait();  // the stats kernel's partials are complete
    const int r = blockIdx.x * kPassWarps + warp_id();  // one warp per row
    if (r < P.B) decide_draft_row<TDT>(P, r);
  } else if (MODE == MODE_TREE) {
    __shared__ TreeSmem sm;
    decide_tree<TDT>(P, b, sm);  // it polls the partials or waits for the stats kernel
  } else {
    __shared__ DecideSmem sm;
    decide_chain_row<MODE, TDT, DDT, PROBS, UNAL>(P, b, h, sm);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // After CTA 0's own row: the stats kernel has finished with its claim
    // counters (a polling CTA 0 waits for it only here, so its row is not
    // held up by the wait): leave them zeroed, record this call's epoch and
    // stamp the counters valid for the next call on this workspace (which
    // reads them after this grid ends).
    grid_dependency_wait();
    for (int s = 0; s < kClaimStripes; ++s) P.claim[s * kClaimStride] = 0u;
    *P.epoch_base = __ldcg(P.epoch_cur);
    __threadfence();
    st_release_u64(P.claim_stamp, kStampValid);
  }
}

}  // namespace sv
