// C ABI of the verification library: argument validation, workspace layout,
// parameter packing and dispatch.  Every check that can fail happens before
// the first CUDA call, so an invalid call touches no GPU state.
#include <atomic>

#include "sv_pass_common.cuh"

namespace sv {

int sm_count(int device) {
  static std::atomic<int> cache[64];
  if (device < 0 || device >= 64) return 0;
  int v = cache[device].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cache[device].store(v, std::memory_order_relaxed);
  }
  return v;
}

size_t workspace_bytes_any(int B, int rows, int V) {
  // fp32 rows off the 16-byte grid give the most warp-chunks and residual
  // chunks
  return make_pass_layout(B, rows, V, 4, 4, true, true).total;
}

static bool valid_dtype(int d) { return d == SV_F32 || d == SV_BF16 || d == SV_F16; }

static size_t dtype_size(int d) { return d == SV_F32 ? 4 : 2; }

// Natural alignment of a (nullable) pointer.
static bool aligned_to(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

static std::atomic<unsigned long long> g_calls{0};
static std::atomic<int> g_force_stream{0};

bool force_stream_path() { return g_force_stream.load(std::memory_order_relaxed) != 0; }

unsigned long long next_call_id() {
  return g_calls.fetch_add(1, std::memory_order_relaxed) + 1;
}

}  // namespace sv

using namespace sv;

extern "C" {

SV_API size_t spec_verify_workspace_bytes(int B, int rows_per_batch, int V, sv_dtype dt) {
  (void)dt;
  if (B <= 0 || rows_per_batch <= 0 || V <= 0 || V > SV_MAX_VOCAB) return 0;
  return workspace_bytes_any(B, rows_per_batch, V);
}

SV_API sv_status spec_verify_chain(const void *target_logits, sv_dtype tdt, const void *draft,
                                   sv_dtype ddt, int draft_is_probs, const int32_t *draft_tokens,
                                   const float *temperatures, const float *uniforms, int B,
                                   int gamma, int V, int32_t *out_tokens,
                                   int32_t *out_num_accepted, float *out_diag,
                                   int32_t *out_row_status, void *workspace,
                                   size_t workspace_bytes, sv_stream_t stream) {
  if (!target_logits || !draft || !draft_tokens || !temperatures || !uniforms || !out_tokens ||
      !out_num_accepted || !workspace)
    return SV_ERR_INVALID_ARG;
  if (B < 1 || gamma < 1 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
    return SV_ERR_INVALID_ARG;
  if (!valid_dtype(tdt) || !valid_dtype(ddt)) return SV_ERR_INVALID_ARG;
  const bool probs = draft_is_probs != 0;
  if (probs && ddt != SV_F32) return SV_ERR_UNSUPPORTED;
  if (!aligned_to(target_logits, dtype_size(tdt)) || !aligned_to(draft, dtype_size(ddt)) ||
      !aligned_to(draft_tokens, 4) || !aligned_to(temperatures, 4) || !aligned_to(uniforms, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) ||
      !aligned_to(out_row_status, 4) || !aligned_to(out_diag, 16))
    return SV_ERR_INVALID_ARG;
  const int rows = (gamma + 1) + (probs ? 0 : gamma);
  if (workspace_bytes < workspace_bytes_any(B, rows, V) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15))
    return SV_ERR_INVALID_ARG;

  KParams P{};
  P.target = target_logits;
  P.draft = draft;
  P.draft_tokens = draft_tokens;
  P.temps = temperatures;
  P.unif = uniforms;
  P.B = B;
  P.gamma = gamma;
  P.V = V;
  P.rows = rows;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.out_diag = out_diag;
  P.out_status = out_row_status;
  P.ws = static_cast<char *>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (tdt) {
    case SV_F32: return launch_chain_f32(P, ddt, probs, s);
    case SV_BF16: return launch_chain_bf16(P, ddt, probs, s);
    case SV_F16: return launch_chain_f16(P, ddt, probs, s);
  }
  return SV_ERR_UNSUPPORTED;
}

SV_API sv_status spec_verify_chain_greedy(const void *target_logits, sv_dtype tdt,
                                          const int32_t *draft_tokens, int B, int gamma, int V,
                                          int32_t *out_tokens, int32_t *out_num_accepted,
                                          int32_t *out_row_status, void *workspace,
                                          size_t workspace_bytes, sv_stream_t stream) {
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted || !workspace)
    return SV_ERR_INVALID_ARG;
  if (B < 1 || gamma < 1 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
    return SV_ERR_INVALID_ARG;
  if (!valid_dtype(tdt)) return SV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, dtype_size(tdt)) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) ||
      !aligned_to(out_row_status, 4))
    return SV_ERR_INVALID_ARG;
  const int rows = gamma + 1;
  if (workspace_bytes < workspace_bytes_any(B, rows, V) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15))
    return SV_ERR_INVALID_ARG;

  KParams P{};
  P.target = target_logits;
  P.draft_tokens = draft_tokens;
  P.B = B;
  P.gamma = gamma;
  P.V = V;
  P.rows = rows;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.out_status = out_row_status;
  P.ws = static_cast<char *>(workspace);
  return launch_chain_greedy(P, tdt, reinterpret_cast<cudaStream_t>(stream));
}

SV_API sv_status spec_verify_tree_greedy(const void *node_logits, sv_dtype dt,
                                         const int32_t *parent, const int32_t *node_tokens, int B,
                                         int N, int V, int max_depth, int32_t *out_path,
                                         int32_t *out_tokens, int32_t *out_num_accepted,
                                         int32_t *out_row_status, void *workspace,
                                         size_t workspace_bytes, sv_stream_t stream) {
  if (!node_logits || !parent || !node_tokens || !out_path || !out_tokens || !out_num_accepted ||
      !workspace)
    return SV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_VOCAB || max_depth < 0 ||
      max_depth > SV_MAX_TREE_DEPTH)
    return SV_ERR_INVALID_ARG;
  if (!valid_dtype(dt)) return SV_ERR_INVALID_ARG;
  if (!aligned_to(node_logits, dtype_size(dt)) || !aligned_to(parent, 4) ||
      !aligned_to(node_tokens, 4) || !aligned_to(out_path, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_num_accepted, 4) || !aligned_to(out_row_status, 4))
    return SV_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_any(B, N, V) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15))
    return SV_ERR_INVALID_ARG;

  KParams P{};
  P.target = node_logits;
  P.parent = parent;
  P.node_tokens = node_tokens;
  P.B = B;
  P.N = N;
  P.V = V;
  P.rows = N;
  P.max_depth = max_depth;
  P.out_path = out_path;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.out_status = out_row_status;
  P.ws = static_cast<char *>(workspace);
  return launch_tree(P, dt, reinterpret_cast<cudaStream_t>(stream));
}

SV_API sv_status spec_draft_sample(const void *logits, sv_dtype dt, const float *temperatures,
                                   const float *uniforms, int B, int V, int32_t *out_tokens,
                                   float *out_probs, int32_t *out_row_status, void *workspace,
                                   size_t workspace_bytes, sv_stream_t stream) {
  if (!logits || !temperatures || !uniforms || !out_tokens || !workspace)
    return SV_ERR_INVALID_ARG;
  if (B < 1 || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_INVALID_ARG;
  if (!valid_dtype(dt)) return SV_ERR_INVALID_ARG;
  if (!aligned_to(temperatures, 4) || !aligned_to(uniforms, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_probs, 4) || !aligned_to(out_row_status, 4))
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(logits, dtype_size(dt))) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_any(B, 1, V) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15))
    return SV_ERR_INVALID_ARG;
  KParams P{};
  P.target = logits;
  P.temps = temperatures;
  P.unif = uniforms;
  P.B = B;
  P.N = 1;
  P.V = V;
  P.rows = 1;
  P.out_tokens = out_tokens;
  P.out_diag = out_probs;
  P.out_status = out_row_status;
  P.ws = static_cast<char *>(workspace);
  return launch_draft(P, dt, reinterpret_cast<cudaStream_t>(stream));
}

SV_API int spec_verify_force_stream_path(int on) {
  return g_force_stream.exchange(on ? 1 : 0, std::memory_order_relaxed);
}

SV_API unsigned long long spec_verify_set_call_counter(unsigned long long calls) {
  return g_calls.exchange(calls, std::memory_order_relaxed);
}

SV_API const char *spec_verify_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK: success";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: null pointer, size out of range or workspace too small";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: dtype combination or size not supported";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA call or kernel launch failed";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a device-side wait ran out";
  }
  return "unknown sv_status";
}

}  // extern "C"
