// Backward sweep instantiations: entropy gradient.
#include "row_bwd.cuh"

namespace vls {
cudaError_t launch_bwd_entropy(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  return launch_bwd_op<kBwdEntropy>(dt, cap, a, s);
}
}  // namespace vls
