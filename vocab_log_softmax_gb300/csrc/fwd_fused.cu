// Fused forward sweep instantiations (logprobs + entropy + optional KL).
#include "row_fwd.cuh"

namespace vls {

cudaError_t launch_fwd_fused(FusedKl kl, vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  if (kl == kFusedKlReverse) return launch_fwd_op<kFwdFused, kFusedKlReverse>(dt, cap, a, s);
  if (kl == kFusedKlForward) return launch_fwd_op<kFwdFused, kFusedKlForward>(dt, cap, a, s);
  return launch_fwd_op<kFwdFused, kFusedNoKl>(dt, cap, a, s);
}

}  // namespace vls
