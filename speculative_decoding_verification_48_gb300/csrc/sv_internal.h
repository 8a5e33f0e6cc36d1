// Internal definitions shared by the host API and the kernels of the
// verification library: the verification modes, the parameters of a call
// and the launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

constexpr int kMaxRows = 2 * SV_MAX_GAMMA + 1;

enum Mode { MODE_CHAIN = 0, MODE_CHAIN_GREEDY = 1, MODE_TREE = 2, MODE_DRAFT = 3 };

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The first kPassHeaderBytes of every workspace hold state kept valid from
// call to call (claim counters, error, ready, stamp and epoch words).
constexpr size_t kPassHeaderBytes = 4096;

// One call, as the entry points receive it.
struct KParams {
  const void *target;         // chain: [B, gamma+1, V]; tree: [B*N, V]; draft: [B, V]
  const void *draft;          // [B, gamma, V] logits or fp32 probabilities
  const int32_t *draft_tokens;
  const float *temps;
  const float *unif;
  const int32_t *parent;
  const int32_t *node_tokens;
  int B, gamma, V, rows, N, max_depth;
  int32_t *out_tokens, *out_nacc, *out_status, *out_path;
  float *out_diag;
  char *ws;                   // workspace base
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

// Diagnostics: every call takes the two-launch streaming path (set by
// spec_verify_force_stream_path).
bool force_stream_path();

// Workspace bytes covering every call shape with B batch rows of at most
// `rows` logit rows of V elements.
size_t workspace_bytes_any(int B, int rows, int V);

// Identifier of a launched call, unique across every entry point and
// instantiation of this process, never 0.
unsigned long long next_call_id();

}  // namespace sv
