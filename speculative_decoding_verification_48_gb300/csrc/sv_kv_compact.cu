// KV-cache compaction after token-tree verification ("論文解説: Speculative
// Sampling", §実装のポイント: the KV entries of rejected tokens are discarded;
// SpecInfer explainer, §推論方法: every tree node was scored in one pass, so
// its KV row sits at the node's slot).  Tree node n (n >= 1) was written at
// slot base + n - 1; the accepted path nodes path[0..d-1] move to slots
// base + 0..d-1 in path order and the cache length becomes base + d.
#include "sv_internal.h"

namespace sv {

constexpr int kKvTile = 1024;                 // bytes of each row per CTA
constexpr int kKvRows = SV_MAX_TREE_DEPTH + 1;  // longest accepted path

// Grid (column tiles, trees).  Warp 0 validates the path; then every row's
// tile is read into shared memory before any is written, because a
// destination slot can be another row's source (sources never lie below
// their destinations, and tiles of one tree are disjoint byte ranges).
__global__ void __launch_bounds__(256) sv_kv_compact_kernel(
    unsigned char *kv, size_t row_bytes, int S, const int32_t *base, const int32_t *path,
    int width, const int32_t *num_accepted, int32_t *out_length, int32_t *out_status) {
  __shared__ uint4 tile[kKvRows][kKvTile / 16];
  __shared__ int s_d, s_ok, s_base;
  __shared__ int s_src[kKvRows];
  const int b = blockIdx.y, lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    // the path row is read alongside d and base (width <= 32 lanes), so one
    // memory round trip covers the whole check
    const int p = lane < width ? __ldg(path + (size_t)b * width + lane) : 0;
    const int d = __ldg(num_accepted + b);
    const int bs = __ldg(base + b);
    const bool dok = d >= 0 && d <= width && bs >= 0;
    const int prev = __shfl_up_sync(0xffffffffu, p, 1);
    const bool bad = dok && lane < d &&
                     (p < lane + 1 || (lane > 0 && p <= prev) || (long long)bs + p - 1 >= S);
    const bool ok = dok && !__any_sync(0xffffffffu, bad);
    if (lane < kKvRows) s_src[lane] = ok && lane < d ? bs + p - 1 : 0;
    if (lane == 0) {
      s_d = ok ? d : 0;
      s_ok = ok;
      s_base = bs;
    }
  }
  __syncthreads();
  const int d = s_d;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (out_length) out_length[b] = s_ok ? s_base + d : s_base;
    if (out_status) out_status[b] = s_ok ? SV_ROW_OK : SV_ROW_BAD_TREE;
  }
  if (d == 0) return;
  const size_t col0 = (size_t)blockIdx.x * kKvTile;
  const int units = (int)min((size_t)kKvTile, row_bytes - col0) / 16;
  unsigned char *tree = kv + (size_t)b * S * row_bytes;
  for (int k = threadIdx.x; k < d * units; k += blockDim.x) {
    const int i = k / units, u = k - i * units;
    tile[i][u] = *reinterpret_cast<const uint4 *>(tree + (size_t)s_src[i] * row_bytes + col0 +
                                                  (size_t)u * 16);
  }
  __syncthreads();
  for (int k = threadIdx.x; k < d * units; k += blockDim.x) {
    const int i = k / units, u = k - i * units;
    *reinterpret_cast<uint4 *>(tree + (size_t)(s_base + i) * row_bytes + col0 + (size_t)u * 16) =
        tile[i][u];
  }
}

}  // namespace sv

extern "C" {

SV_API sv_status spec_tree_kv_compact(void *kv, size_t row_bytes, int B, int S,
                                      const int32_t *base, const int32_t *path, int path_width,
                                      const int32_t *num_accepted, int32_t *out_length,
                                      int32_t *out_row_status, sv_stream_t stream) {
  if (!kv || !base || !path || !num_accepted) return SV_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || S < 1 || path_width < 1 || path_width > sv::kKvRows)
    return SV_ERR_INVALID_ARG;
  if (row_bytes < 16 || row_bytes % 16 || (reinterpret_cast<uintptr_t>(kv) & 15) ||
      (reinterpret_cast<uintptr_t>(base) & 3) || (reinterpret_cast<uintptr_t>(path) & 3) ||
      (reinterpret_cast<uintptr_t>(num_accepted) & 3) ||
      (reinterpret_cast<uintptr_t>(out_length) & 3) ||
      (reinterpret_cast<uintptr_t>(out_row_status) & 3))
    return SV_ERR_INVALID_ARG;
  const size_t tiles = (row_bytes + sv::kKvTile - 1) / sv::kKvTile;
  if (tiles > 0x7fffffffu) return SV_ERR_UNSUPPORTED;
  dim3 grid((unsigned)tiles, (unsigned)B);
  sv::sv_kv_compact_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned char *>(kv), row_bytes, S, base, path, path_width, num_accepted,
      out_length, out_row_status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"
