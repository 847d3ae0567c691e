// Forward sweep instantiations for the kl statistic.
#include "row_fwd.cuh"

namespace vls {
cudaError_t launch_fwd_kl(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  return launch_fwd_op<kFwdKl>(dt, cap, a, s);
}
}  // namespace vls
