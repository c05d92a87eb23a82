// Forward kernel instances for head dimension 256.
#include "fa_fwd256_pair_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d256(const FwdLaunch& a) { return fwd256p::launch_any(a); }
}  // namespace fa
