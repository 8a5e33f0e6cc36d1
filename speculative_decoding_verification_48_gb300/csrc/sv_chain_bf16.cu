// Chain speculative-sampling kernels with bf16 target logits.
#include "sv_launch.cuh"

namespace sv {
sv_status launch_chain_bf16(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream) {
  return launch_chain_t<SV_BF16>(P, ddt, probs, stream);
}
}  // namespace sv
