// Backward sweep instantiations: KL gradients (both directions).
#include "row_bwd.cuh"

namespace vls {
cudaError_t launch_bwd_kl(bool reverse, vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  return reverse ? launch_bwd_op<kBwdKlReverse>(dt, cap, a, s) : launch_bwd_op<kBwdKlForward>(dt, cap, a, s);
}
}  // namespace vls
