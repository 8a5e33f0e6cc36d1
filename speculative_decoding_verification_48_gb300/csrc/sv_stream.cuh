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
//                       index) or residual mass — and arrives on done;
//   warp 1  bookkeeper  releases finished stages (empty barrier), stores the
//                       slice partials and their merged tile partial, and
//                       counts the units into their batch rows, one fence per
//                       batch of stages; the unit that completes a row queues
//                       the row for the decider;
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

// Scheduler (one thread of its own warp): decides the unit sequence and
// writes one descriptor per unit into a shared-memory ring.  All global
// round trips of scheduling (Phase-A claims, temperatures, Phase-B tickets
// and decision records) happen here, off the thread that arrives on the
// stage barriers, and none of their results is needed in the iteration that
// requests it.  Phase-A claims take batches of up to kClaim consecutive
// units while many remain (single units near the end); a batch is decoded
// once and then walked with increments.
template <int MODE, int TDT, int DDT, bool PROBS>
__device__ void stream_scheduler(const SParams &P, StreamSmem &sm) {
  const int G1 = P.gamma + 1;
  const unsigned totalA = (unsigned)P.totalA;
  const unsigned qcap = (unsigned)(P.B * P.tilesB);
  const unsigned grid = gridDim.x;
  const unsigned unitsA = (unsigned)P.unitsA;
  const unsigned kmax = (unsigned)min(kClaim, P.unitsA);
  const int rowsA = (MODE == MODE_CHAIN) ? (PROBS ? G1 : G1 + P.gamma) : P.rows;
  auto claim_size = [&](unsigned at) { return (at + 4u * kmax * grid < totalA) ? kmax : 1u; };
  // Two claims in flight: n1 (next batch, temperatures being fetched) and
  // n2 (its atomic still returning).
  unsigned n1_s = atomicAdd(&P.hdr->a_next, kmax), n1_k = kmax;
  unsigned n2_s = atomicAdd(&P.hdr->a_next, kmax), n2_k = kmax;
  float n1_lo = 0.f, n1_hi = 0.f;
  if (MODE == MODE_CHAIN && n1_s < totalA) {
    n1_lo = __ldg(P.temps + n1_s / unitsA);
    n1_hi = __ldg(P.temps + (min(n1_s + n1_k, totalA) - 1u) / unitsA);
  }
  // current batch: remaining count and the walking position (b, row, tile)
  unsigned left = 0;
  int cb = 0, crow = 0, ctile = 0, blo = -1;
  float Tlo = 0.f, Thi = 0.f;
  // queue counters in use / loads in flight, pending ticket and its item
  unsigned qh = 0, qr = 0, qh_n = 0, qr_n = 0;
  long long ticket = -1;
  unsigned tw_seen = 0, tw_n = 0;
  bool tw_fresh = false;
  bool timed_out = false;
  for (int it = 0;; ++it) {
    const long long tw = clock64();
    while (it - sm.ring_head >= kRing) {
      if (clock64() - tw > kStreamWait) { timed_out = true; break; }
    }
    StageMeta &mt = sm.ring[it % kRing];
    int kind = U_STOP;
    const bool poll = (it % kPoll) == 0;
    const long long t0 = clock64();
    while (!timed_out) {
      if constexpr (MODE == MODE_CHAIN) {
        // Phase-B tiles first: they are L2-hot and unblock finalisation.
        if (poll || left == 0) {
          if (ticket < 0 && qh < qr) {
            ticket = atomicAdd(&P.hdr->q_head, 1u);
            if (ticket >= (long long)qcap) ticket = -1;  // can never be published
            qh = qr;
            tw_seen = 0;
            tw_fresh = false;
          } else if (ticket >= 0 && tw_seen == 0) {
            {
              // use the value loaded at the previous poll; start the next load
              if (tw_fresh) tw_seen = tw_n;
              tw_n = ld_relaxed_u32(P.qitems + ticket);
              tw_fresh = true;
            }
          }
        }
        if (ticket >= 0 && tw_seen != 0) {
          fence_acq_rel_gpu();  // acquire: the decision record published before the item
          const unsigned v = tw_seen - 1u;
          ticket = -1;
          tw_seen = 0;
          tw_fresh = false;
          const int j = (int)(v & 31u), bt = (int)(v >> 5);
          const int bb = bt / P.tilesB, tt = bt % P.tilesB;
          if (bb >= P.B || j >= P.gamma) {
            // a malformed item: never copy from it
            atomicOr(&P.hdr->error, 2u);
            continue;
          }
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
          kind = U_RESID;
          break;
        }
      }
      if (left == 0 && n1_s < totalA) {
        // promote n1 (decode its first unit once); n2 becomes n1; claim n2
        const unsigned s0 = n1_s;
        left = min(n1_s + n1_k, totalA) - s0;
        cb = (int)(s0 / unitsA);
        const int ri = (int)(s0 % unitsA);
        if (MODE != MODE_CHAIN || ri < G1 * P.tilesT) {
          crow = ri / P.tilesT;
          ctile = ri % P.tilesT;
        } else {
          const int rd = ri - G1 * P.tilesT;
          crow = G1 + rd / P.tilesD;
          ctile = rd % P.tilesD;
        }
        blo = cb;
        Tlo = n1_lo;
        Thi = n1_hi;
        n1_s = n2_s;
        n1_k = n2_k;
        if (MODE == MODE_CHAIN && n1_s < totalA) {
          n1_lo = __ldg(P.temps + n1_s / unitsA);
          n1_hi = __ldg(P.temps + (min(n1_s + n1_k, totalA) - 1u) / unitsA);
        }
        n2_k = claim_size(max(s0 + left, n1_s + n1_k));
        n2_s = atomicAdd(&P.hdr->a_next, n2_k);
      }
      if (left > 0) {
        const int isdraft = (MODE == MODE_CHAIN && crow >= G1) ? 1 : 0;
        const float T = (cb == blo) ? Tlo : Thi;
        int k = U_ARGMAX;
        float c = 0.f;
        if constexpr (MODE == MODE_CHAIN) {
          if (bad_temperature(T) || (isdraft && T <= 0.f)) k = U_NOOP;
          else if (T > 0.f) { k = U_SOFTMAX; c = kLog2e / T; }
        }
        const int TA = isdraft ? P.TA_D : P.TA_T;
        mt.b = cb;
        mt.row = crow;
        mt.tile = ctile;
        mt.isdraft = isdraft;
        mt.c = c;
        mt.n = min(TA, P.V - ctile * TA);
        kind = k;
        // advance (tile, row, batch row)
        --left;
        if (++ctile == (isdraft ? P.tilesD : P.tilesT)) {
          ctile = 0;
          if (++crow == rowsA) { crow = 0; ++cb; }
        }
        break;
      }
      // Phase A exhausted: wait for queued Phase-B tiles or the end.
      if (MODE != MODE_CHAIN) break;
      const unsigned dd = ld_acquire(&P.hdr->decisions_done);
      qh = ld_volatile_u32(&P.hdr->q_head);
      qr = ld_volatile_u32(&P.hdr->q_reserved);
      if (ticket >= 0 && ticket < (long long)qcap) {
        tw_seen = ld_relaxed_u32(P.qitems + ticket);
        if (tw_seen != 0) continue;
        // every row decided and the ticket beyond the final count: nothing
        // will ever be published there
        if (dd >= (unsigned)P.B && ticket >= (long long)qr) ticket = -1;
      } else {
        if (qh < qr) continue;
        if (dd >= (unsigned)P.B) break;
      }
      __nanosleep(200);
      if (clock64() - t0 > kStreamWait) { timed_out = true; break; }
    }
    if (timed_out) kind = U_STOP;
    mt.kind = kind;
    __threadfence_block();
    sm.ring_tail = it + 1;
    if (kind == U_STOP) break;
    if constexpr (MODE == MODE_CHAIN) {
      if (poll) {
        // use the counters loaded at the previous poll; start the next loads
        qh = qh_n;
        qr = qr_n;
        qh_n = ld_volatile_u32(&P.hdr->q_head);
        qr_n = ld_volatile_u32(&P.hdr->q_reserved);
      }
    }
  }
  if (timed_out) {
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
      const volatile StageMeta &d = sm.ring[it % kRing];
      mt.kind = d.kind; mt.b = d.b; mt.row = d.row; mt.tile = d.tile; mt.n = d.n;
      mt.isdraft = d.isdraft; mt.j = d.j; mt.c = d.c; mt.Mp = d.Mp; mt.invZp = d.invZp;
      mt.Mq = d.Mq; mt.invZq = d.invZq;
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
      if (!ok) {
        atomicOr(&P.hdr->error, 4u);
        mt.kind = U_NOOP;
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

// Bookkeeper: the tile partial merged from the kCW slice partials held by
// lanes 0..kCW-1 (other lanes pass neutral values).  Returns it in lane 0.
__device__ __forceinline__ float2 merge_slices(int kind, float2 v, float c) {
  const bool mine = lane_id() < kCW;
  if (kind == U_SOFTMAX) {
    const float m = mine ? v.x : -CUDART_INF_F;
    const float M = warp_max_nan(m);
    float z = 0.f;
    if (mine) z = (v.x == -CUDART_INF_F) ? v.y : v.y * ex2((v.x - M) * c);
    return make_float2(M, warp_sum(z));
  }
  if (kind == U_ARGMAX) {
    const float m = mine ? v.x : -CUDART_INF_F;
    const float best = warp_max_nan(m);
    const int idx = warp_min_int(mine && v.x == best ? __float_as_int(v.y) : 0x7fffffff);
    return make_float2(best, __int_as_float(idx));
  }
  return make_float2(warp_sum(mine ? v.x : 0.f), 0.f);
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
      mbar_init(&sm.done[s], kCW);
      mbar_init(&sm.empty[s], 1);
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
    if (lane == 0) stream_scheduler<MODE, TDT, DDT, PROBS>(P, sm);
    return;
  }

  if (warp >= 4) {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 4;
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
      // Read the batch's descriptors and slice partials, release the stages,
      // then write the partials out: the release never waits on global stores.
      StageMeta mts[kBookBatch];
      float2 wps[kBookBatch];
      int used = 0;
      for (int k = 0; k < nb; ++k) {
        const int s = (it + k) % kStages;
        mts[k] = sm.meta[s];
        if (mts[k].kind == U_STOP) { stop = true; break; }
        wps[k] = lane < kCW ? sm.wpart[s][lane] : make_float2(0.f, 0.f);
        ++used;
      }
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < used; ++k) mbar_arrive(&sm.empty[(it + k) % kStages]);
      __syncwarp();
      unsigned *cnt[kBookBatch];
      unsigned target[kBookBatch];
      int item[kBookBatch];
      for (int k = 0; k < used; ++k) {
        const StageMeta &mt = mts[k];
        const float2 wp = wps[k];
        if (mt.kind == U_SOFTMAX || mt.kind == U_ARGMAX) {
          const size_t ro = ((size_t)mt.b * P.rows + mt.row) * P.tilesMax + mt.tile;
          if (lane < kCW) P.partA[ro * kCW + lane] = wp;
          const float2 tp = merge_slices(mt.kind, wp, mt.c);
          if (lane == 0) P.partT[ro] = tp;
        } else if (mt.kind == U_RESID) {
          const size_t ro = (size_t)mt.b * P.tilesB + mt.tile;
          if (lane < kCW) P.partB[ro * kCW + lane] = wp.x;
          const float2 tp = merge_slices(U_RESID, wp, 0.f);
          if (lane == 0) P.partBT[ro] = tp.x;
        }
        if (mt.kind == U_RESID) {
          cnt[k] = P.b_count + mt.b;
          target[k] = (unsigned)P.tilesB;
          item[k] = D_FINAL;
        } else {
          cnt[k] = P.a_count + mt.b;
          target[k] = (unsigned)P.unitsA;
          item[k] = (MODE == MODE_TREE) ? D_TREE : D_CHAIN;
        }
      }
      __syncwarp();
      if (lane == 0) {
        fence_acq_rel_gpu();  // the partials above before the arrivals below
        unsigned prev[kBookBatch];
        for (int k = 0; k < used; ++k) prev[k] = atomicAdd(cnt[k], 1u);
        bool any_last = false;
        for (int k = 0; k < used; ++k) any_last |= (prev[k] == target[k] - 1);
        if (any_last) fence_acq_rel_gpu();  // acquire: other CTAs' partials of the row
        for (int k = 0; k < used; ++k) {
          if (prev[k] == target[k] - 1) {
            const long long tq = clock64();
            while (sm.dq_push - sm.dq_pop >= kDQ && clock64() - tq < kStreamWait) __nanosleep(64);
            reinterpret_cast<volatile int *>(sm.dq)[sm.dq_push % kDQ] = (item[k] << 28) | mts[k].b;
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
