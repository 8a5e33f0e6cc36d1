// Chain speculative-sampling kernels with f16 target logits.
#include "sv_launch.cuh"

namespace sv {
sv_status launch_chain_f16(const KParams &P, sv_dtype ddt, bool probs, cudaStream_t stream) {
  return launch_chain_t<SV_F16>(P, ddt, probs, stream);
}
}  // namespace sv
