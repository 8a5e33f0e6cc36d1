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

// Draft-side draws: the two-launch path, whatever the rows' alignment.
template <int DT>
static sv_status launch_draft_t(const KParams &P, cudaStream_t stream) {
  constexpr int es = (DT == SV_F32) ? 4 : 2;
  const bool unaligned = !rows_aligned(P.target, P.V, es);
  const PassLayout L = make_pass_layout(P.B, 1, P.V, es, es, false, unaligned);
  const long long total = pass_units<MODE_DRAFT, DT, DT, false>(P, L);
  if (total < 0) return SV_ERR_UNSUPPORTED;
  return launch_pass<MODE_DRAFT, DT, DT, false>(P, L, total, unaligned, stream);
}

sv_status launch_draft(const KParams &P, sv_dtype dt, cudaStream_t stream) {
  switch (dt) {
    case SV_F32: return launch_draft_t<SV_F32>(P, stream);
    case SV_BF16: return launch_draft_t<SV_BF16>(P, stream);
    case SV_F16: return launch_draft_t<SV_F16>(P, stream);
  }
  return SV_ERR_UNSUPPORTED;
}

}  // namespace sv
