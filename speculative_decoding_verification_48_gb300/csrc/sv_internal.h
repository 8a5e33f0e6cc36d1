// Internal definitions shared by the host API and the kernels of the
// verification library: tile geometry, workspace layout, kernel parameters
// and the unit schedule.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// One CTA processes one "unit": a tile of kTile consecutive vocabulary
// entries of one logit row (Phase A), or of one target/draft row pair
// (Phase B).  256 threads x 32 elements per thread.
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 8192;
constexpr int kPer = kTile / kThreads;
constexpr int kMaxRows = 2 * SV_MAX_GAMMA + 1;

enum Mode { MODE_CHAIN = 0, MODE_CHAIN_GREEDY = 1, MODE_TREE = 2, MODE_DRAFT = 3 };
enum DecKind { DEC_DONE = 0, DEC_RESIDUAL = 1 };

// Per-batch-row decision written by the CTA that completes the row's
// Phase A, read by the row's Phase B units.  64 bytes.
struct Decision {
  int kind;    // DecKind
  int j;       // first rejected position
  int pad0, pad1;
  float c;     // log2(e) / T
  float Mp, invZp, Mq, invZq;  // row maxima and 1 / normalisers of rows p_j, q_j
  float u;     // the categorical draw u_gamma
  float pad2[6];
};
static_assert(sizeof(Decision) == 64, "Decision must stay 64 bytes");

struct WsHeader {
  unsigned unit_counter;  // dynamic work counter (reset by the last CTA to exit)
  unsigned exit_counter;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The first kPassHeaderBytes of every workspace hold the two-launch path's
// state between calls (claim counters and their validity stamp); the
// register-tile kernels' layout starts after them and never touches them.
constexpr size_t kPassHeaderBytes = 4096;

// Workspace layout for B batch rows of `rows` logit rows of V entries.  The
// control block [0, ctrl) holds the work counters, per-row arrival counters,
// decision flags and error words; every call zeroes it first (one small
// memset), so a workspace needs no initialisation and may be shared by calls
// of different shapes in stream order.
struct Layout {
  size_t a_count, b_count, flag, err, ctrl, dec, partA, partB, total;
  int tiles;
};

inline Layout make_layout(int B, int rows, int V) {
  Layout L;
  L.tiles = (V + kTile - 1) / kTile;
  size_t off = 256;  // WsHeader
  L.a_count = off; off = align_up(off + (size_t)B * 4, 256);
  L.b_count = off; off = align_up(off + (size_t)B * 4, 256);
  L.flag = off;    off = align_up(off + (size_t)B * 4, 256);
  L.err = off;     off = align_up(off + (size_t)B * 4, 256);
  L.ctrl = off;
  L.dec = off;     off = align_up(off + (size_t)B * sizeof(Decision), 256);
  L.partA = off;   off = align_up(off + (size_t)B * rows * L.tiles * sizeof(float2), 256);
  L.partB = off;   off = align_up(off + (size_t)B * L.tiles * sizeof(float), 256);
  L.total = off;
  return L;
}

// Unit schedule of one launch.  The unit sequence is built from B blocks
// (one per batch row, in batch order): block k holds the A units of batch
// row k followed by the B units of batch row k - L (the lag).  The B units
// of the last L rows follow the last A block.  With Bc = 0 a launch runs A
// units only; with A = 0 and L = 0 it runs B units only.
struct Sched {
  int B, A, Bc, L;
  int total;
};

struct KParams {
  const void *target;         // chain: [B, gamma+1, V]; tree: [B*N, V]
  const void *draft;          // [B, gamma, V] logits or fp32 probabilities
  const int32_t *draft_tokens;
  const float *temps;
  const float *unif;
  const int32_t *parent;
  const int32_t *node_tokens;
  int B, gamma, V, tiles, rows, N, max_depth;
  int phase_b;                // 1 if the call has Phase-B units (publish decisions)
  int use_stream;             // allow the streaming (TMA ring) kernel
  int32_t *out_tokens, *out_nacc, *out_status, *out_path;
  float *out_diag;
  char *ws;                   // workspace base
  WsHeader *hdr;
  unsigned *a_count, *b_count, *flag;
  int *err;                   // per-row SV_ROW_TIMEOUT bits from Phase-B waits
  size_t ctrl_bytes;          // bytes of the control block zeroed per call
  Decision *dec;
  float2 *partA;
  float *partB;
  Sched sched;
};

// Launchers, defined in the kernel translation units (one per target dtype
// for the chain, so they compile in parallel).
sv_status launch_chain_f32(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream);
sv_status launch_chain_bf16(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream);
sv_status launch_chain_f16(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream);
sv_status launch_chain_greedy(const KParams &P, sv_dtype tdt, cudaStream_t stream);
sv_status launch_tree(const KParams &P, sv_dtype dt, cudaStream_t stream);
sv_status launch_draft(const KParams &P, sv_dtype dt, cudaStream_t stream);

// Device properties cached per device (host side).
int sm_count(int device);

// Workspace bytes covering both kernel families for the given shape.
size_t workspace_bytes_any(int B, int rows, int V);

// Identifier of a launched call, unique across every entry point and
// instantiation of this process, never 0.
unsigned long long next_call_id();

}  // namespace sv
