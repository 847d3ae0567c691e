// Fused backward map instantiations (any weighted sum of logprobs, entropy
// and KL of the same policy logits).
#include "row_bwd.cuh"

namespace vls {

cudaError_t launch_bwd_fused(FusedKl kl, vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  if (kl == kFusedKlReverse) return launch_bwd_op<kBwdFused, kFusedKlReverse>(dt, cap, a, s);
  if (kl == kFusedKlForward) return launch_bwd_op<kBwdFused, kFusedKlForward>(dt, cap, a, s);
  return launch_bwd_op<kBwdFused, kFusedNoKl>(dt, cap, a, s);
}

}  // namespace vls
