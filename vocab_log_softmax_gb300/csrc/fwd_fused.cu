// Fused forward sweep instantiations (logprobs + entropy + optional KL).
#include "row_fwd.cuh"

namespace vls {

template <int DIR>
cudaError_t launch_fused_dir(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16)
    return cap ? launch_fwd_t<__nv_bfloat16, kFwdFused, true, DIR>(a, s)
               : launch_fwd_t<__nv_bfloat16, kFwdFused, false, DIR>(a, s);
  return cap ? launch_fwd_t<float, kFwdFused, true, DIR>(a, s) : launch_fwd_t<float, kFwdFused, false, DIR>(a, s);
}

cudaError_t launch_fwd_fused(FusedKl kl, vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  if (kl == kFusedKlReverse) return launch_fused_dir<kFusedKlReverse>(dt, cap, a, s);
  if (kl == kFusedKlForward) return launch_fused_dir<kFusedKlForward>(dt, cap, a, s);
  return launch_fused_dir<kFusedNoKl>(dt, cap, a, s);
}

}  // namespace vls
