/*
 * spec_verify.h — C ABI of the GB300 (sm_103a) speculative-sampling
 * verification library.
 *
 * The library runs the verification step of speculative decoding on one GPU:
 *
 *   - chain speculative sampling ("Speculative Sampling", Chen et al.,
 *     arXiv:2302.01318, as explained on "論文解説: Speculative Sampling —
 *     ドラフトモデルによるLLMデコード高速化", §技術的詳細 ステップ3 and
 *     §修正付き棄却サンプリング): temperature softmax of target and draft rows,
 *     accept test min(1, p/q) against a supplied uniform, stop at the first
 *     rejection, draw the replacement from norm(max(0, p - q)), or a bonus
 *     token from p at position gamma+1 when every draft is accepted;
 *   - greedy chain verification ("投機的デコーディングとは？LLMの回答を高速化
 *     する仕組み", §ドラフト生成と並列検証の仕組み and the worked example in
 *     §候補の採用と棄却を具体例で見る);
 *   - SpecInfer-style token-tree greedy verification (SpecInfer explainer,
 *     §技術の仕組み › 基本アイデア and §推論方法): argmax per tree node, then a
 *     walk from the root along children whose token matches.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array pointers are DEVICE pointers owned by the caller.  Arrays are
 *    dense and row-major: a logit row is V contiguous elements, row stride V.
 *    The library never allocates and never synchronises the host; work is
 *    enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - `workspace` is caller-owned device memory of at least
 *    spec_verify_workspace_bytes(...) bytes, 16-byte aligned.  Its first
 *    4096 bytes hold library state between calls: work-claim counters, left
 *    zeroed by every call and stamped valid (a call that finds no valid
 *    stamp resets them itself), and a call epoch that the kernels advance
 *    by one per call, CUDA graph replays included.  Those 4096 bytes must
 *    be zero before the first call on the memory, and again whenever the
 *    caller has used that memory for anything else in between: recycled
 *    memory can hold a stale valid stamp above non-zero counters, which the
 *    library cannot tell from its own state.  The rest of the workspace
 *    needs no initialisation.  Calls that may overlap on the GPU need
 *    distinct workspaces; calls in stream order may share one, whatever
 *    their shapes.
 *  - Each call enqueues its kernels as programmatic dependents
 *    (programmatic dependent launch) of the work before them in `stream`:
 *    the first kernel waits on the device for that work to complete before
 *    it reads the inputs or touches the workspace, and only then lets the
 *    call's second kernel start, so stream order is kept even after work
 *    that lets its own dependents start early.
 *  - Calls may be captured into a CUDA graph.  Each replay verifies the
 *    inputs found in the captured buffers at replay time.
 *  - Row alignment is the caller's job: target row i scores draft i (the
 *    distribution conditioned on the context and drafts 0..i-1); row gamma is
 *    the bonus row.
 *  - Host-detectable argument errors return a status synchronously and
 *    enqueue nothing.  Errors in the DATA (bad token ids, NaN rows, malformed
 *    trees) are reported per row in `out_row_status` (bit mask SV_ROW_*); such
 *    a row gets num_accepted = 0 and every token -1.
 *  - Every pointer must be aligned to its element type (out_diag to 16
 *    bytes); otherwise the call returns SV_ERR_INVALID_ARG.  Any V >= 1 and
 *    any row alignment are accepted.  Rows are streamed on each row's own
 *    16-byte grid (whole aligned 16-byte blocks); the bytes of a block that
 *    lie outside the row are masked, never used.
 *  - No function throws; all are thread-safe given distinct workspaces.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, workspace too small */
  SV_ERR_UNSUPPORTED = 2,   /* dtype combination or size the library does not handle */
  SV_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  SV_ERR_TIMEOUT = 4        /* reserved: device-side timeouts are reported per row */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1, SV_F16 = 2 } sv_dtype;

/* Per-row data-error bits written to out_row_status. */
#define SV_ROW_OK 0
#define SV_ROW_BAD_TOKEN 1        /* a draft / node token outside [0, V) */
#define SV_ROW_NONFINITE 2        /* NaN (or +inf / all -inf) in a softmax row, NaN in an argmax row,
                                     a non-finite draft probability read, or a non-finite residual */
#define SV_ROW_BAD_TREE 4         /* parent[0] != -1 or parent[n] outside [0, n) */
#define SV_ROW_TIMEOUT 8          /* a bounded device-side wait ran out (about one second) */
#define SV_ROW_BAD_TEMPERATURE 16 /* temperature NaN or in (0, 1e-20) */

/* Size limits checked on the host. */
#define SV_MAX_GAMMA 31           /* gamma + 1 <= 32: one warp lane per position */
#define SV_MAX_TREE_NODES 1024
#define SV_MAX_TREE_DEPTH 31
#define SV_MAX_VOCAB (1 << 26)

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *sv_stream_t;

/*
 * Workspace bytes for B batch rows (chains or trees) of at most
 * `rows_per_batch` logit rows of V elements each.  rows_per_batch is
 * 2*gamma+1 for spec_verify_chain with draft logits, gamma+1 for
 * spec_verify_chain with draft probabilities and for
 * spec_verify_chain_greedy, N for spec_verify_tree_greedy, and 1 for
 * spec_draft_sample.  `dt` is the
 * logit dtype.  Returns 0 for non-positive sizes.
 */
SV_API size_t spec_verify_workspace_bytes(int B, int rows_per_batch, int V, sv_dtype dt);

/*
 * Chain speculative sampling, one verification step per batch row.
 * ("論文解説: Speculative Sampling", §技術的詳細 ステップ3: accept equation;
 *  §修正付き棄却サンプリング: residual equation; §期待される高速化: gamma+1
 *  tokens per round, hence the bonus draw.)
 *
 *  target_logits  [B, gamma+1, V] of dtype tdt.
 *  draft          [B, gamma, V]: logits of dtype ddt, or, if draft_is_probs,
 *                 fp32 probabilities (ddt must be SV_F32) used as given — no
 *                 temperature, no renormalisation; only q(x_i) and the row at
 *                 a rejected position are read.
 *  draft_tokens   int32 [B, gamma].
 *  temperatures   fp32 [B].  T <= 0: greedy row (target argmax, draft row and
 *                 uniforms unused).  T > 0: p = softmax(target/T) and, for
 *                 draft logits, q = softmax(draft/T).
 *  uniforms       fp32 [B, gamma+1] in [0, 1): column i < gamma is the accept
 *                 draw of draft i, column gamma the single categorical draw.
 *  Per row: accept draft i iff u_i * q_i(x_i) < p_i(x_i), in order; j = first
 *  rejection (else gamma); the token at slot j is the smallest k with
 *  sum_{x<=k} w(x) > u_gamma * sum_x w(x), w = max(0, p_j - q_j) if j < gamma
 *  (w = p_j if that mass is zero), w = p_gamma if j == gamma.
 *  out_tokens       int32 [B, gamma+1]: drafts 0..j-1, the drawn token, then -1.
 *  out_num_accepted int32 [B]: j.
 *  out_diag         nullable fp32 [B, gamma, 4]: per draft i, (p_i(x_i),
 *                   q_i(x_i), min(1, p/q), residual mass sum max(0, p_j - q_j)
 *                   at i == j of a rejected row, else 0).  Zero for greedy rows.
 *  out_row_status   nullable int32 [B]: SV_ROW_* bits, 0 when the row is valid.
 *  Limits: B >= 1, 1 <= gamma <= SV_MAX_GAMMA, 1 <= V <= SV_MAX_VOCAB.
 */
SV_API sv_status spec_verify_chain(const void *target_logits, sv_dtype tdt,
                                   const void *draft, sv_dtype ddt, int draft_is_probs,
                                   const int32_t *draft_tokens, const float *temperatures,
                                   const float *uniforms, int B, int gamma, int V,
                                   int32_t *out_tokens, int32_t *out_num_accepted,
                                   float *out_diag, int32_t *out_row_status,
                                   void *workspace, size_t workspace_bytes, sv_stream_t stream);

/*
 * Greedy chain verification ("投機的デコーディングとは？", §ドラフト生成と並列検証の
 * 仕組み; worked example §候補の採用と棄却を具体例で見る).
 *  a_i = argmax of target row i (lowest index among equal maxima, -0 == +0);
 *  accept while x_i == a_i; at the first mismatch j (or j = gamma) emit a_j.
 *  target_logits [B, gamma+1, V] of dtype tdt; draft_tokens int32 [B, gamma];
 *  out_tokens int32 [B, gamma+1]; out_num_accepted int32 [B];
 *  out_row_status nullable int32 [B].  Same results as spec_verify_chain with
 *  every temperature <= 0.
 */
SV_API sv_status spec_verify_chain_greedy(const void *target_logits, sv_dtype tdt,
                                          const int32_t *draft_tokens, int B, int gamma, int V,
                                          int32_t *out_tokens, int32_t *out_num_accepted,
                                          int32_t *out_row_status, void *workspace,
                                          size_t workspace_bytes, sv_stream_t stream);

/*
 * Token-tree greedy verification (SpecInfer explainer, §技術の仕組み › 基本アイデア,
 * §推論方法).
 *  node_logits [B*N, V] of dtype dt: row b*N + n scores what follows node n of
 *  tree b.  parent int32 [B, N]: parent[0] = -1, 0 <= parent[n] < n (node 0
 *  is the root, the context's last token; it is never verified).
 *  node_tokens int32 [B, N].
 *  Walk: cur = 0; while depth < max_depth: take the lowest-index child c of
 *  cur with node_tokens[c] == argmax(row cur); stop if none.  The argmax of
 *  the last node reached is appended as the correction / bonus token.
 *  out_path   int32 [B, max_depth+1]: accepted node ids, then -1.
 *  out_tokens int32 [B, max_depth+1]: accepted node tokens, the appended
 *             token, then -1.
 *  out_num_accepted int32 [B]: accepted depth.  out_row_status nullable [B].
 *  Limits: 1 <= N <= SV_MAX_TREE_NODES, 0 <= max_depth <= SV_MAX_TREE_DEPTH.
 */
SV_API sv_status spec_verify_tree_greedy(const void *node_logits, sv_dtype dt,
                                         const int32_t *parent, const int32_t *node_tokens,
                                         int B, int N, int V, int max_depth,
                                         int32_t *out_path, int32_t *out_tokens,
                                         int32_t *out_num_accepted, int32_t *out_row_status,
                                         void *workspace, size_t workspace_bytes,
                                         sv_stream_t stream);

/*
 * Draft-side categorical draw, one per row: the draft step that produces
 * the tokens verified above ("論文解説: Speculative Sampling", §アルゴリズム
 * Step 1: each draft token is drawn from softmax(draft logits / T)).
 *  logits       [B, V] of dtype dt (the draft model's next-token rows).
 *  temperatures fp32 [B]; T <= 0 takes the first argmax (lowest index).
 *  uniforms     fp32 [B] in [0, 1): the draw is the inverse CDF in
 *               ascending vocabulary order, the smallest k with
 *               sum_{x<=k} q(x) > u * sum_x q(x), q = softmax(logits / T).
 *  out_tokens   int32 [B]: the drawn token (-1 for an invalid row).
 *  out_probs    nullable fp32 [B]: q(token) (0 for greedy and invalid rows).
 *  out_row_status nullable int32 [B]: SV_ROW_* bits.
 *  workspace: spec_verify_workspace_bytes(B, 1, V, dt) bytes.
 *  Any V >= 1 and any row alignment (the pointer aligned to its element
 *  type) are accepted.
 */
SV_API sv_status spec_draft_sample(const void *logits, sv_dtype dt, const float *temperatures,
                                   const float *uniforms, int B, int V, int32_t *out_tokens,
                                   float *out_probs, int32_t *out_row_status, void *workspace,
                                   size_t workspace_bytes, sv_stream_t stream);

/*
 * Token-tree attention mask (SpecInfer explainer, §技術の仕組み › 基本アイデア and
 * §推論方法: all tree nodes are scored in one target pass, each node seeing
 * itself and its ancestors only).
 *  parent       int32 [B, N]: parent[0] = -1, 0 <= parent[n] < n.
 *  out_mask     uint64 [B, N, W], W = ceil(N / 64): row n has bit m (bit
 *               m % 64 of word m / 64) set iff m == n or m is an ancestor of n.
 *  out_depth    nullable int32 [B, N]: edges from the root.
 *  out_row_status nullable int32 [B]: SV_ROW_BAD_TREE for a malformed tree,
 *               whose mask is all zero and depths 0.
 *  Limits: 1 <= N <= SV_MAX_TREE_NODES.  No workspace.
 */
SV_API sv_status spec_tree_mask(const int32_t *parent, int B, int N, uint64_t *out_mask,
                                int32_t *out_depth, int32_t *out_row_status, sv_stream_t stream);

/*
 * KV-cache compaction after token-tree verification ("論文解説: Speculative
 * Sampling", §実装のポイント: the KV entries of rejected tokens are dropped;
 * SpecInfer explainer, §推論方法: all tree nodes were scored in one pass, so
 * their KV rows lie in node order after the context).  Tree node n >= 1 of
 * tree b was written at slot base[b] + n - 1; the accepted path nodes
 * path[b, 0..d-1] (d = num_accepted[b], the output of
 * spec_verify_tree_greedy) move to slots base[b] + 0..d-1 in path order, in
 * place, and the cache length becomes base[b] + d.  Other slots keep their
 * bytes.
 *  kv           device, [B, S] rows of row_bytes bytes each (any element
 *               type: rows are moved as bytes), updated in place.  16-byte
 *               aligned; row_bytes a positive multiple of 16.
 *  base         int32 [B]: slot of tree node 1 (the first slot after the
 *               context).
 *  path         int32 [B, path_width], 1 <= path_width <= SV_MAX_TREE_DEPTH + 1.
 *  num_accepted int32 [B].
 *  out_length   nullable int32 [B]: base[b] + d, or base[b] for a bad row.
 *  out_row_status nullable int32 [B]: SV_ROW_BAD_TREE when d is outside
 *               [0, path_width], base[b] < 0, or a path entry is below i + 1,
 *               not above the previous entry, or names a slot >= S; such a
 *               row moves nothing.
 *  All pointers are device pointers owned by the caller.  No workspace; the
 *  call is asynchronous on `stream`.  Returns SV_ERR_INVALID_ARG for null
 *  required pointers, bad sizes or misaligned buffers.
 */
SV_API sv_status spec_tree_kv_compact(void *kv, size_t row_bytes, int B, int S,
                                      const int32_t *base, const int32_t *path, int path_width,
                                      const int32_t *num_accepted, int32_t *out_length,
                                      int32_t *out_row_status, sv_stream_t stream);

/*
 * Diagnostics.  Runs one of the library's bounded device-side waits on a flag
 * that nothing sets, so that a caller can check that the wait gives up after
 * its bound and reports instead of hanging (the verification calls report the
 * same event as SV_ROW_TIMEOUT in out_row_status).
 *  which        0: the stats kernel's wait for its claim counters to be reset
 *               (a spin bound, about a second);
 *               1: the decide kernel's poll of a row's chunk partials for
 *               the call's tag (a bound of 512 polling rounds, after which
 *               the decide kernel waits for the stats kernel instead).
 *  scratch      device memory of at least 64 bytes, 16-byte aligned; the call
 *               zeroes and uses it.
 *  out_status   device int32 [1]: SV_ROW_TIMEOUT when the wait ran out, the
 *               expected result; SV_ROW_OK if the flag was seen.
 * Takes about a second of GPU time.  The context stays usable afterwards.
 */
SV_API sv_status spec_verify_wait_selftest(int which, void *scratch, int32_t *out_status,
                                           sv_stream_t stream);

/*
 * Diagnostics.  Small calls (chains whose kept row slices fit the shared
 * memory of one cluster of at most 8 CTAs per batch row; trees of at most
 * 1 MB of node-row slices per CTA; every cluster resident at once) run on
 * the cluster path: one launch, no workspace use.
 * Every other call runs the two-launch streaming path.  With on != 0 every
 * call takes the streaming path (tests use this to check both paths on the
 * same shapes); returns the previous setting.  Process-wide.
 */
SV_API int spec_verify_force_stream_path(int on);

/*
 * Diagnostics.  Sets the process-wide call counter that numbers the
 * library's calls and returns its previous value.  The next call gets
 * number calls + 1.  A call's number tags the partial results its first
 * kernel hands to its second; only calls numbered below 2^31 let the second
 * kernel merge tagged partials as they arrive (the tags of those calls are
 * all distinct), later calls wait for the first kernel to finish.  Tests use
 * this to reach that limit.  Moving the counter backwards can repeat tags of
 * earlier calls and is not supported.
 */
SV_API unsigned long long spec_verify_set_call_counter(unsigned long long calls);

/* Static description of a status code; never NULL. */
SV_API const char *spec_verify_status_string(sv_status s);

/*
 * Bytes of the fixed scratch array behind spec_verify_chain_no_alloc.
 */
#define SV_NO_ALLOC_SCRATCH_BYTES (8 << 20)

/*
 * spec_verify_chain without a caller-provided workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory — for example a plugin inside a serving engine that has
 * already reserved the whole GPU for its own pool, or a decode loop that must
 * not call cudaMalloc because cudaMalloc can synchronise the device.  Inputs
 * and outputs are the caller's device arrays, exactly as for
 * spec_verify_chain (same arguments, same results); only the scratch memory
 * differs.  It is one fixed array of SV_NO_ALLOC_SCRATCH_BYTES (8 MiB) in the
 * library's device image, which every GPU that loads the library holds until
 * the process exits.  This function allocates nothing and calls no
 * allocating library routine.
 *
 *  - Sizes whose workspace (spec_verify_workspace_bytes with rows_per_batch
 *    2*gamma+1, or gamma+1 with draft_is_probs) exceeds
 *    SV_NO_ALLOC_SCRATCH_BYTES return SV_ERR_UNSUPPORTED and enqueue nothing.
 *    B=64, gamma=7, V=128256 needs about 2 MB.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  A failed lookup returns SV_ERR_CUDA.  The
 *    address is kept for the life of the process and belongs to the
 *    device's primary context: do not use this function after
 *    cudaDeviceReset, nor under a context made current through the driver
 *    API.
 *  - Every call on a device shares the one array.  Calls that may overlap
 *    on the GPU (different streams, or different host threads without
 *    ordering) race on it and give wrong results: keep them in one stream
 *    order.  What an earlier call left in the array does no harm: every
 *    call either finds its state valid or resets it.
 */
SV_API sv_status spec_verify_chain_no_alloc(const void *target_logits, sv_dtype tdt,
                                            const void *draft, sv_dtype ddt, int draft_is_probs,
                                            const int32_t *draft_tokens,
                                            const float *temperatures, const float *uniforms,
                                            int B, int gamma, int V, int32_t *out_tokens,
                                            int32_t *out_num_accepted, float *out_diag,
                                            int32_t *out_row_status, sv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H_ */
