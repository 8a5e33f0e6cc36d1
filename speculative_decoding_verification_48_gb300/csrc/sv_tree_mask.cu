// Token-tree attention mask from the parent array (SpecInfer explainer,
// §技術の仕組み › 基本アイデア and §推論方法: every tree node is scored in one
// target pass, which needs a mask letting each node see itself and its
// ancestors only).  Mask row n of a tree has bit m set iff m == n or m is an
// ancestor of n; rows are N bits stored as W = ceil(N / 64) little-endian
// 64-bit words (bit m % 64 of word m / 64).
#include "sv_internal.h"

namespace sv {

// One CTA per tree.  The parents are staged in shared memory and checked
// (parent[0] == -1, 0 <= parent[n] < n); each thread then walks its node's
// ancestor chain once.  Ancestors have strictly decreasing indices, so the
// walk ends within n + 1 steps and visits the row's words from high to low:
// each word is written once, words the walk skips are written as zero.
__global__ void __launch_bounds__(1024) sv_tree_mask_kernel(const int32_t *parent, int N, int W,
                                                            unsigned long long *out_mask,
                                                            int32_t *out_depth,
                                                            int32_t *out_status) {
  __shared__ int par[SV_MAX_TREE_NODES];
  __shared__ int bad;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const int p = parent[(size_t)b * N + n];
    par[n] = p;
    if (n == 0 ? p != -1 : (p < 0 || p >= n)) bad = 1;
  }
  __syncthreads();
  const bool ok = bad == 0;
  unsigned long long *rows = out_mask + (size_t)b * N * W;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    unsigned long long *row = rows + (size_t)n * W;
    if (!ok) {
      for (int w = 0; w < W; ++w) row[w] = 0ull;
      if (out_depth) out_depth[(size_t)b * N + n] = 0;
      continue;
    }
    int cw = n >> 6;
    for (int w = cw + 1; w < W; ++w) row[w] = 0ull;
    unsigned long long acc = 0ull;
    int d = 0;
    for (int cur = n; cur >= 0; cur = par[cur]) {
      const int wi = cur >> 6;
      if (wi != cw) {
        row[cw] = acc;
        for (int w = wi + 1; w < cw; ++w) row[w] = 0ull;
        cw = wi;
        acc = 0ull;
      }
      acc |= 1ull << (cur & 63);
      ++d;
    }
    row[cw] = acc;
    for (int w = 0; w < cw; ++w) row[w] = 0ull;
    if (out_depth) out_depth[(size_t)b * N + n] = d - 1;
  }
  if (threadIdx.x == 0 && out_status) out_status[b] = ok ? SV_ROW_OK : SV_ROW_BAD_TREE;
}

}  // namespace sv

extern "C" {

SV_API sv_status spec_tree_mask(const int32_t *parent, int B, int N, uint64_t *out_mask,
                                int32_t *out_depth, int32_t *out_row_status, sv_stream_t stream) {
  if (!parent || !out_mask) return SV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || N > SV_MAX_TREE_NODES) return SV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(parent) & 3) || (reinterpret_cast<uintptr_t>(out_mask) & 7) ||
      (reinterpret_cast<uintptr_t>(out_depth) & 3) ||
      (reinterpret_cast<uintptr_t>(out_row_status) & 3))
    return SV_ERR_INVALID_ARG;
  const int W = (N + 63) / 64;
  const int threads = N >= 1024 ? 1024 : ((N + 31) / 32) * 32;
  sv::sv_tree_mask_kernel<<<B, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      parent, N, W, reinterpret_cast<unsigned long long *>(out_mask), out_depth, out_row_status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
