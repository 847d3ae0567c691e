// Forward sweep instantiations for the logp statistic.
#include "row_fwd.cuh"

namespace vls {
cudaError_t launch_fwd_logp(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  return launch_fwd_op<kFwdLogp>(dt, cap, a, s);
}
}  // namespace vls
