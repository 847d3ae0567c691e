// Fused backward map instantiations (any weighted sum of logprobs, entropy
// and KL of the same policy logits).
#include "row_bwd.cuh"

namespace vls {

template <int DIR>
cudaError_t launch_bwd_fused_dir(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16)
    return cap ? launch_bwd_t<__nv_bfloat16, kBwdFused, true, DIR>(a, s)
               : launch_bwd_t<__nv_bfloat16, kBwdFused, false, DIR>(a, s);
  return cap ? launch_bwd_t<float, kBwdFused, true, DIR>(a, s) : launch_bwd_t<float, kBwdFused, false, DIR>(a, s);
}

cudaError_t launch_bwd_fused(FusedKl kl, vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  if (kl == kFusedKlReverse) return launch_bwd_fused_dir<kFusedKlReverse>(dt, cap, a, s);
  if (kl == kFusedKlForward) return launch_bwd_fused_dir<kFusedKlForward>(dt, cap, a, s);
  return launch_bwd_fused_dir<kFusedNoKl>(dt, cap, a, s);
}

}  // namespace vls
