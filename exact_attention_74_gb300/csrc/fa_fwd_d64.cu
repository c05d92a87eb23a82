// Forward kernel instances for head dimension 64.
#include "fa_fwd64_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d64(const FwdLaunch& a) { return fwd64::launch_any(a); }
}  // namespace fa
