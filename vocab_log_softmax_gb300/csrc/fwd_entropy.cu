// Forward sweep instantiations for the entropy statistic.
#include "row_fwd.cuh"

namespace vls {
cudaError_t launch_fwd_entropy(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  return launch_fwd_op<kFwdEntropy>(dt, cap, a, s);
}
}  // namespace vls
