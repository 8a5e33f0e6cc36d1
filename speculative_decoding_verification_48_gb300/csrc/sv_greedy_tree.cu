// Greedy chain and token-tree verification kernels.
#include "sv_launch.cuh"

namespace sv {

sv_status launch_chain_greedy(const KParams &P, sv_dtype tdt, cudaStream_t stream) {
  switch (tdt) {
    case SV_F32: return launch_verify<MODE_CHAIN_GREEDY, SV_F32, SV_F32, false>(P, stream);
    case SV_BF16: return launch_verify<MODE_CHAIN_GREEDY, SV_BF16, SV_BF16, false>(P, stream);
    case SV_F16: return launch_verify<MODE_CHAIN_GREEDY, SV_F16, SV_F16, false>(P, stream);
  }
  return SV_ERR_UNSUPPORTED;
}

sv_status launch_tree(const KParams &P, sv_dtype dt, cudaStream_t stream) {
  switch (dt) {
    case SV_F32: return launch_verify<MODE_TREE, SV_F32, SV_F32, false>(P, stream);
    case SV_BF16: return launch_verify<MODE_TREE, SV_BF16, SV_BF16, false>(P, stream);
    case SV_F16: return launch_verify<MODE_TREE, SV_F16, SV_F16, false>(P, stream);
  }
  return SV_ERR_UNSUPPORTED;
}

}  // namespace sv
