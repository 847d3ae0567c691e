// Backward sweep instantiations: logprob gradient.
#include "row_bwd.cuh"

namespace vls {
cudaError_t launch_bwd_logp(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  return launch_bwd_op<kBwdLogp>(dt, cap, a, s);
}
}  // namespace vls
