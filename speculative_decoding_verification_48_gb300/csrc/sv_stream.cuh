// Streaming verification kernel for sm_103a: one persistent CTA per SM with a
// shared-memory ring filled by TMA bulk copies.
//
// Warp roles of a CTA:
//   warp 3  scheduler   picks the unit sequence — a Phase-B ticket when tiles
//                       are queued, else the next Phase-A units of a
//                       device-wide counter — and writes unit descriptors to a
//                       shared-memory ring; every global round trip of
//                       scheduling happens here;
//   warp 0  producer    turns descriptors into cp.async.bulk copies of the
//                       unit's tile(s) into a ring stage (full barrier);
//   warps 4..19 consumers  each reduces its 1/16 slice of a stage to a warp
//                       partial — softmax (max, sum exp2), argmax (max, first
//                       index) or residual mass — releases the stage (empty
//                       barrier) and puts the partial in a shared-memory
//                       partial ring;
//   warp 1  bookkeeper  drains the partial ring: stores the slice partials
//                       and their merged tile partial, and counts the units
//                       into their batch rows, one fence per batch of units;
//                       the unit that completes a row queues the row for the
//                       decider;
//   warp 2  decider     merges the row's tile partials (one lane per row),
//                       runs the accept tests / greedy match / tree walk,
//                       draws the bonus token, or queues the row's Phase-B
//                       tiles device-wide; after the row's last Phase-B tile
//                       it finds the crossing tile and slice of u * R and
//                       rescans that slice.
//
// Rows must start on 16-byte boundaries (V * element size a multiple of 16,
// 16-byte aligned bases); other shapes use the register-tile kernels.
#pragma once

#include "sv_stream_rows.cuh"

namespace sv {

// Scheduler (a whole warp): decides the unit sequence and writes one
// descriptor per unit into a shared-memory ring, up to kSchedBatch units per
// step with one lane per unit, published with one fence per step.  It owns
// every global round trip of scheduling, so the producer's stage-barrier
// arrivals never wait on loads.
//   Phase B: the device-wide queue is split round-robin, CTA c owning slots
//   c, c + G, c + 2G, ...; lanes poll the next owned slots together and the
//   published prefix becomes descriptors (decision record loaded per lane).
//   Phase A: claims of up to kClaim consecutive units from a device-wide
//   counter while many remain (single units near the end), two claims in
//   flight so a batch's temperatures are requested a batch ahead.
template <int MODE, int TDT, int DDT, bool PROBS>
__device__ void stream_scheduler(const SParams &P, StreamSmem &sm) {
  const int lane = lane_id();
  const int G1 = P.gamma + 1;
  const unsigned totalA = (unsigned)P.totalA;
  const long long qcap = (long long)P.B * P.tilesB;
  const unsigned grid = gridDim.x;
  const unsigned unitsA = (unsigned)P.unitsA;
  const unsigned kmax = (unsigned)min(kClaim, P.unitsA);
  // claim size shrinks with the work left per CTA: about half of each CTA's
  // remaining share, between 1 and kmax units
  auto claim_size = [&](unsigned at) {
    const unsigned left = at < totalA ? totalA - at : 0u;
    return max(1u, min(kmax, left / (2u * grid)));
  };
  // Phase-A units a row reads: all of them for a sampled row, the target
  // rows' tiles for a greedy row, one no-op unit for an invalid temperature
  const unsigned tgt_units = (unsigned)(G1 * P.tilesT);
  auto row_units = [&](float T) -> unsigned {
    if (MODE != MODE_CHAIN) return unitsA;
    if (bad_temperature(T)) return 1u;
    return T > 0.f ? unitsA : tgt_units;
  };
  // claims: lane 0 issues, every lane keeps the values (broadcast on use)
  unsigned n1_s = 0, n1_k = kmax, n2_s = 0, n2_k = kmax;
  if (lane == 0) {
    n1_s = atomicAdd(&P.hdr->a_next, kmax);
    n2_s = atomicAdd(&P.hdr->a_next, kmax);
  }
  n1_s = __shfl_sync(0xffffffffu, n1_s, 0);
  float n1_lo = 0.f, n1_hi = 0.f;
  if (MODE == MODE_CHAIN && n1_s < totalA) {
    n1_lo = __ldg(P.temps + n1_s / unitsA);
    n1_hi = __ldg(P.temps + (min(n1_s + n1_k, totalA) - 1u) / unitsA);
  }
  unsigned cur = 0, cur_end = 0;  // current Phase-A batch
  float Tlo = 0.f, Thi = 0.f;
  unsigned blo = 0;
  long long bnext = blockIdx.x;   // next owned Phase-B queue slot
  int tail = 0;                   // descriptors written
  bool stop = false, timed_out = false;
  long long t0 = clock64();
  while (!stop) {
    // room for a full step in the ring
    const long long tw = clock64();
    while (tail + kSchedBatch - sm.ring_head > kRing) {
      if (clock64() - tw > kStreamWait) { timed_out = true; break; }
    }
    if (timed_out) break;
    int written = 0;
    // ---- Phase B: published prefix of the next owned slots
    if constexpr (MODE == MODE_CHAIN) {
      const long long slot = bnext + (long long)lane * grid;
      unsigned w = 0;
      if (lane < kSchedBatch && slot < qcap) w = ld_relaxed_u32(P.qitems + slot);
      const unsigned pub = __ballot_sync(0xffffffffu, w != 0);
      const int nb = __ffs(~pub) - 1;  // leading published slots
      if (nb > 0) {
        fence_acq_rel_gpu();  // acquire: decision records published before the items
        if (lane < nb) {
          const unsigned v = w - 1u;
          const int j = (int)(v & 31u), bt = (int)(v >> 5);
          const int bb = bt / P.tilesB, tt = bt % P.tilesB;
          StageMeta &mt = sm.ring[(tail + lane) % kRing];
          mt.target = 0;
          if (bb < P.B && j < P.gamma) {
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
            mt.n = min(P.TB, P.V - tt * P.TB);
            mt.kind = U_RESID;
          } else {
            atomicOr(&P.hdr->error, 2u);  // a malformed item: never copy from it
            mt.kind = U_SKIP;
            mt.b = 0;
          }
        }
        written = nb;
        bnext += (long long)nb * grid;
      }
    }
    // ---- Phase A: the rest of the step from the current batch.  Units a
    // row does not read are not emitted: a greedy row reads only its target
    // rows, a row with an invalid temperature reads nothing and gets one
    // no-op unit; every emitted unit carries its row's unit count.
    bool moved = written > 0, promoted = false;
    while (written < kSchedBatch) {
      if (cur >= cur_end) {
        // a second promotion in one step would wait on the claim and the
        // temperature loads just issued: publish what the step has first
        if (promoted && written > 0) break;
        n1_s = __shfl_sync(0xffffffffu, n1_s, 0);
        if (n1_s >= totalA) break;
        promoted = true;
        // promote n1; n2 becomes n1 (fetch its temperatures); claim a new n2
        cur = n1_s;
        cur_end = min(n1_s + n1_k, totalA);
        blo = cur / unitsA;
        Tlo = n1_lo;
        Thi = n1_hi;
        n1_s = __shfl_sync(0xffffffffu, n2_s, 0);
        n1_k = __shfl_sync(0xffffffffu, n2_k, 0);
        if (MODE == MODE_CHAIN && n1_s < totalA) {
          n1_lo = __ldg(P.temps + n1_s / unitsA);
          n1_hi = __ldg(P.temps + (min(n1_s + n1_k, totalA) - 1u) / unitsA);
        }
        if (lane == 0) {
          n2_k = claim_size(max(cur_end, n1_s + n1_k));
          n2_s = atomicAdd(&P.hdr->a_next, n2_k);
        }
      }
      moved = true;
      {
        // jump over the unread tail of the row at cur (warp-uniform)
        const unsigned bb = cur / unitsA, ri = cur % unitsA;
        if (ri >= row_units(bb == blo ? Tlo : Thi)) {
          cur = min(cur_end, (bb + 1u) * unitsA);
          continue;
        }
      }
      const int na = (int)min((unsigned)(kSchedBatch - written), cur_end - cur);
      const unsigned ua = cur + (unsigned)lane;
      const int bb = (int)(ua / unitsA), ri = (int)(ua % unitsA);
      const float T = ((unsigned)bb == blo) ? Tlo : Thi;
      const unsigned target = row_units(T);
      const bool keep = lane < na && (unsigned)ri < target;
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) {
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
        int k = U_ARGMAX;
        float c = 0.f;
        if constexpr (MODE == MODE_CHAIN) {
          if (bad_temperature(T)) k = U_NOOP;
          else if (T > 0.f) { k = U_SOFTMAX; c = kLog2e / T; }
        }
        const int TA = isdraft ? P.TA_D : P.TA_T;
        const int pos = __popc(km & ((1u << lane) - 1u));
        StageMeta &mt = sm.ring[(tail + written + pos) % kRing];
        mt.kind = k;
        mt.b = bb;
        mt.row = row;
        mt.tile = tile;
        mt.isdraft = isdraft;
        mt.c = c;
        mt.n = min(TA, P.V - tile * TA);
        mt.target = (int)target;
      }
      cur += (unsigned)na;
      written += __popc(km);
    }
    if (!moved) {
      // nothing to hand out: the end of Phase A
      if (MODE != MODE_CHAIN) {
        stop = true;
      } else {
        unsigned dd = 0, qr = 0;
        if (lane == 0) {
          dd = ld_acquire(&P.hdr->decisions_done);
          qr = ld_volatile_u32(&P.hdr->q_reserved);
        }
        dd = __shfl_sync(0xffffffffu, dd, 0);
        qr = __shfl_sync(0xffffffffu, qr, 0);
        // every row decided and every owned slot below the final count taken
        if (dd >= (unsigned)P.B && bnext >= (long long)qr) stop = true;
        else {
          __nanosleep(200);
          if (clock64() - t0 > kStreamWait) { timed_out = true; break; }
        }
      }
      if (stop) {
        if (lane == 0) sm.ring[tail % kRing].kind = U_STOP;
        written = 1;
      }
    }
    __syncwarp();
    if (written > 0 && lane == 0) {
      __threadfence_block();
      sm.ring_tail = tail + written;
    }
    tail += written;
    if (moved) t0 = clock64();  // the end-phase bound counts idle time only
  }
  if (timed_out && lane == 0) {
    // hand the producer a STOP so the consumers finish
    const long long tw = clock64();
    while (tail + 1 - sm.ring_head > kRing && clock64() - tw < kStreamWait) {}
    sm.ring[tail % kRing].kind = U_STOP;
    __threadfence_block();
    sm.ring_tail = tail + 1;
    atomicOr(&P.hdr->error, 1u);
    for (int b = 0; b < P.B; ++b)
      if (ld_volatile_u32(P.row_done + b) == 0 && P.out_status) P.out_status[b] = SV_ROW_TIMEOUT;
  }
}

// Producer (one thread): takes descriptors from the ring and issues the
// bulk copies of each unit into the next free stage.  Its only global-memory
// operations are the asynchronous copies, so arriving on the stage barrier
// never waits on a load.
template <int MODE, int TDT, int DDT, bool PROBS>
__device__ void stream_producer(const SParams &P, StreamSmem &sm, unsigned char *stages) {
  using TT = typename Elt<TDT>::T;
  using DTy = typename Elt<DDT>::T;
  const int G1 = P.gamma + 1;
  int last_data_stage = -1;
  unsigned last_data_phase = 0;
  bool timed_out = false;
  for (int it = 0;; ++it) {
    const int s = it % kStages;
    const unsigned ph = (unsigned)(it / kStages) & 1u;
    if (it >= kStages && !mbar_wait(&sm.empty[s], ph ^ 1u, clock64())) timed_out = true;
    const long long tw = clock64();
    while (!timed_out && sm.ring_tail <= it) {
      if (clock64() - tw > kStreamWait) timed_out = true;
    }
    StageMeta &mt = sm.meta[s];
    if (timed_out) {
      mt.kind = U_STOP;
    } else {
      __threadfence_block();  // acquire: the slot was written before the tail
      const volatile StageMeta &d = sm.ring[it % kRing];
      mt.kind = d.kind; mt.b = d.b; mt.row = d.row; mt.tile = d.tile; mt.n = d.n;
      mt.isdraft = d.isdraft; mt.j = d.j; mt.c = d.c; mt.Mp = d.Mp; mt.invZp = d.invZp;
      mt.Mq = d.Mq; mt.invZq = d.invZq; mt.target = d.target;
      __threadfence_block();
      sm.ring_head = it + 1;
    }
    unsigned char *dst = stages + (size_t)s * kStageBytes;
    {
      // never issue a copy from a descriptor outside the arrays
      bool ok = mt.b >= 0 && mt.b < P.B && mt.n > 0;
      if (mt.kind == U_SOFTMAX || mt.kind == U_ARGMAX) {
        const int tiles = mt.isdraft ? P.tilesD : P.tilesT;
        const int TA = mt.isdraft ? P.TA_D : P.TA_T;
        ok = ok && mt.row >= 0 && mt.row < P.rows && mt.tile >= 0 && mt.tile < tiles &&
             mt.n <= TA && mt.tile * TA + mt.n <= P.V;
      } else if (mt.kind == U_RESID) {
        ok = ok && mt.j >= 0 && mt.j < P.gamma && mt.tile >= 0 && mt.tile < P.tilesB &&
             mt.n <= P.TB && mt.tile * P.TB + mt.n <= P.V;
      } else {
        ok = true;
      }
      if (mt.kind == U_SKIP) ok = true;
      if (!ok) {
        atomicOr(&P.hdr->error, 4u);
        mt.kind = U_SKIP;
      }
    }
    if (mt.kind == U_SOFTMAX || mt.kind == U_ARGMAX) {
      const int TA = mt.isdraft ? P.TA_D : P.TA_T;
      const int x0 = mt.tile * TA;
      const char *src;
      unsigned bytes;
      if (mt.isdraft) {
        src = reinterpret_cast<const char *>(reinterpret_cast<const DTy *>(P.draft) +
                                             ((size_t)mt.b * P.gamma + (mt.row - G1)) * P.V + x0);
        bytes = (unsigned)(mt.n * sizeof(DTy));
      } else {
        const int rows_per = (MODE == MODE_TREE) ? P.N : G1;
        src = reinterpret_cast<const char *>(reinterpret_cast<const TT *>(P.target) +
                                             ((size_t)mt.b * rows_per + mt.row) * P.V + x0);
        bytes = (unsigned)(mt.n * sizeof(TT));
      }
      mbar_expect_tx(&sm.full[s], bytes);
      bulk_g2s(dst, src, bytes, &sm.full[s]);
      last_data_stage = s;
      last_data_phase = ph;
    } else if (mt.kind == U_RESID) {
      const int x0 = mt.tile * P.TB;
      const TT *prow = reinterpret_cast<const TT *>(P.target) + ((size_t)mt.b * G1 + mt.j) * P.V + x0;
      const DTy *qrow =
          reinterpret_cast<const DTy *>(P.draft) + ((size_t)mt.b * P.gamma + mt.j) * P.V + x0;
      const unsigned pbytes = (unsigned)(mt.n * sizeof(TT));
      const unsigned qbytes = (unsigned)(mt.n * sizeof(DTy));
      mbar_expect_tx(&sm.full[s], pbytes + qbytes);
      bulk_g2s(dst, prow, pbytes, &sm.full[s]);
      bulk_g2s(dst + (size_t)P.TB * sizeof(TT), qrow, qbytes, &sm.full[s]);
      last_data_stage = s;
      last_data_phase = ph;
    }
    const bool stop = mt.kind == U_STOP;
    mbar_arrive(&sm.full[s]);
    if (stop) break;
  }
  if (timed_out) {
    atomicOr(&P.hdr->error, 1u);
    // let the copies still in flight land before the CTA can exit
    if (last_data_stage >= 0) mbar_wait(&sm.full[last_data_stage], last_data_phase, clock64());
  }
}

// Bookkeeper: the tile partial of one unit from its kCW = 16 slice partials,
// held by the 16 lanes of a half-warp (the two halves merge two units at
// once).  Branch-free so both halves run the same shuffles whatever their
// unit kinds: softmax (M, sum s 2^((m - M) c)), argmax (max, lowest index
// holding it), residual (sum of masses, in .y).
__device__ __forceinline__ float2 half_merge(int kind, float2 v, float c) {
  float mx = v.x;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
  if (kind == U_SOFTMAX) z = (v.x == -CUDART_INF_F) ? v.y : v.y * ex2((v.x - mx) * c);
  else if (kind == U_RESID) z = v.x;
  int idx = (kind == U_ARGMAX && v.x == mx) ? __float_as_int(v.y) : 0x7fffffff;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    z += __shfl_xor_sync(0xffffffffu, z, o);
    idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
  }
  return make_float2(mx, kind == U_ARGMAX ? __int_as_float(idx) : z);
}

template <int MODE, int TDT, int DDT, bool PROBS>
__global__ void __launch_bounds__(kStreamThreads, 1) sv_stream_kernel(const SParams P) {
  extern __shared__ unsigned char smem_raw[];
  StreamSmem &sm = *reinterpret_cast<StreamSmem *>(smem_raw);
  unsigned char *stages = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(StreamSmem) + 127) & ~uintptr_t(127));
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
    }
    for (int s = 0; s < kPR; ++s) {
      mbar_init(&sm.pdone[s], kCW);
      mbar_init(&sm.pfree[s], 1);
    }
    sm.dq_push = 0;
    sm.dq_pop = 0;
    sm.ctl_done = 0;
    sm.ring_head = 0;
    sm.ring_tail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) stream_producer<MODE, TDT, DDT, PROBS>(P, sm, stages);
    return;
  }

  if (warp == 3) {
    // ------------------------------------------------------------ scheduler
    stream_scheduler<MODE, TDT, DDT, PROBS>(P, sm);
    return;
  }

  if (warp >= 4) {
    // ------------------------------------------------------------ consumers
    // Each consumer warp releases the stage itself once its slice is reduced,
    // then hands the slice partial to the bookkeeper through a ring of kPR
    // partial slots (slot it % kPR for unit it).
    const int cw = warp - 4;
    for (int it = 0;; ++it) {
      const int s = it % kStages;
      const unsigned ph = (unsigned)(it / kStages) & 1u;
      if (!mbar_wait(&sm.full[s], ph, clock64())) {
        if (lane == 0) atomicOr(&P.hdr->error, 1u);
        return;
      }
      const StageMeta mt = sm.meta[s];
      const unsigned char *st = stages + (size_t)s * kStageBytes;
      float2 part = make_float2(0.f, 0.f);
      if (mt.kind == U_SOFTMAX) {
        if (mt.isdraft) part = warp_softmax_slice<DDT>(st, mt.n, cw, mt.c);
        else part = warp_softmax_slice<TDT>(st, mt.n, cw, mt.c);
      } else if (mt.kind == U_ARGMAX) {
        part = warp_argmax_slice<TDT>(st, mt.n, cw, mt.tile * P.TA_T);
      } else if (mt.kind == U_RESID) {
        if constexpr (MODE == MODE_CHAIN) part.x = warp_resid_slice<TDT, DDT, PROBS>(st, mt.n, cw, mt);
      }
      __syncwarp();  // every lane is done with the stage
      const int ps = it % kPR;
      bool ok = true;
      if (lane == 0) {
        if (mt.kind != U_STOP) mbar_arrive(&sm.empty[s]);
        if (it >= kPR) ok = mbar_wait(&sm.pfree[ps], ((unsigned)(it / kPR) & 1u) ^ 1u, clock64());
        if (ok) {
          sm.wpart[ps][cw] = part;
          if (cw == 0) sm.pmeta[ps] = mt;
          mbar_arrive(&sm.pdone[ps]);
        } else {
          atomicOr(&P.hdr->error, 1u);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || mt.kind == U_STOP) break;
    }
    return;
  }

  if (warp == 1) {
    // ------------------------------------------------------------ bookkeeper
    // Drains the partial ring in batches of up to kBookBatch units: stores
    // the slice partials and tile partials (two units per pass, one per
    // half-warp), fences once, then adds each batch row's units to its
    // counter with one atomic per row, issued by one leader lane per row.
    const int half = lane >> 4, hl = lane & 15;
    bool stop = false;
    for (int it = 0; !stop;) {
      int nb = 1;
      if (lane == 0) {
        if (!mbar_wait(&sm.pdone[it % kPR], (unsigned)(it / kPR) & 1u, clock64())) {
          atomicOr(&P.hdr->error, 1u);
          nb = 0;
        }
        while (nb > 0 && nb < kBookBatch &&
               mbar_test(&sm.pdone[(it + nb) % kPR], (unsigned)((it + nb) / kPR) & 1u))
          ++nb;
      }
      nb = __shfl_sync(0xffffffffu, nb, 0);
      if (nb == 0) break;
      // lane l < nb: unit it + l's row key, for the counting below
      int kl = U_SKIP, bl = 0, tl = 0;
      if (lane < nb) {
        const StageMeta &m = sm.pmeta[(it + lane) % kPR];
        kl = m.kind;
        bl = m.b;
        tl = (kl == U_RESID) ? P.tilesB : m.target;
      }
      const unsigned sm_stop = __ballot_sync(0xffffffffu, lane < nb && kl == U_STOP);
      const int used = sm_stop ? __ffs(sm_stop) - 1 : nb;
      stop = sm_stop != 0;
      // partial stores and tile merges, two units per pass
      for (int k0 = 0; k0 < used; k0 += 2) {
        const int k = k0 + half;
        int kind = U_SKIP, b = 0, ro = 0;
        float c = 0.f;
        float2 wp = make_float2(0.f, 0.f);
        if (k < used) {
          const StageMeta &m = sm.pmeta[(it + k) % kPR];
          kind = m.kind;
          b = m.b;
          ro = (kind == U_RESID) ? m.tile : m.row * P.tilesMax + m.tile;
          c = m.c;
          wp = sm.wpart[(it + k) % kPR][hl];
        }
        const float2 tp = half_merge(kind, wp, c);
        if (kind == U_SOFTMAX || kind == U_ARGMAX) {
          const size_t r = (size_t)b * P.rows * P.tilesMax + ro;
          P.partA[r * kCW + hl] = wp;
          if (hl == 0) P.partT[r] = tp;
        } else if (kind == U_RESID) {
          const size_t r = (size_t)b * P.tilesB + ro;
          P.partB[r * kCW + hl] = wp.x;
          if (hl == 0) P.partBT[r] = tp.y;
        }
      }
      __syncwarp();
      fence_acq_rel_gpu();  // the partials above before the counts below
      // one leader lane per (counter, row) adds that row's units of the batch
      const bool counted = lane < used && kl != U_SKIP;
      const unsigned key = counted ? ((kl == U_RESID ? 0x80000000u : 0u) | (unsigned)bl)
                                   : (0x40000000u | (unsigned)lane);
      const unsigned grp = __match_any_sync(0xffffffffu, key);
      bool last = false;
      if (counted && (__ffs(grp) - 1) == lane) {
        const unsigned n = (unsigned)__popc(grp);
        const unsigned prev = atomicAdd((kl == U_RESID ? P.b_count : P.a_count) + bl, n);
        last = prev + n == (unsigned)tl;
      }
      const unsigned lm = __ballot_sync(0xffffffffu, last);
      if (lane == 0)
        for (int k = 0; k < used; ++k) mbar_arrive(&sm.pfree[(it + k) % kPR]);
      if (lm) {
        fence_acq_rel_gpu();  // acquire: other CTAs' partials of the completed rows
        for (unsigned mm = lm; mm; mm &= mm - 1) {
          const int l = __ffs(mm) - 1;
          const int kind = __shfl_sync(0xffffffffu, kl, l);
          const int b = __shfl_sync(0xffffffffu, bl, l);
          if (lane == 0) {
            const int item = kind == U_RESID ? D_FINAL : (MODE == MODE_TREE ? D_TREE : D_CHAIN);
            const long long tq = clock64();
            while (sm.dq_push - sm.dq_pop >= kDQ && clock64() - tq < kStreamWait) __nanosleep(64);
            reinterpret_cast<volatile int *>(sm.dq)[sm.dq_push % kDQ] = (item << 28) | b;
            __threadfence_block();
            sm.dq_push = sm.dq_push + 1;
          }
        }
      }
      __syncwarp();
      it += used;
    }
    if (lane == 0) {
      __threadfence_block();
      sm.ctl_done = 1;
    }
    return;
  }

  // -------------------------------------------------------------- decider
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
      fence_acq_rel_gpu();
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

// Workspace layout of the streaming kernel; every call zeroes the control
// block [0, ctrl).
struct StreamLayout {
  size_t a_count, b_count, row_done, qitems, ctrl, dec, partA, partT, partB, partBT, total;
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
  L.partT = off;    off = align_up(off + (size_t)B * rows * L.tilesMax * sizeof(float2), 256);
  L.partB = off;    off = align_up(off + (size_t)B * L.tilesB * kCW * sizeof(float), 256);
  L.partBT = off;   off = align_up(off + (size_t)B * L.tilesB * sizeof(float), 256);
  L.total = off;
  return L;
}

}  // namespace sv
