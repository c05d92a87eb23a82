// Forward kernel instances for head dimension 64.
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d64(const FwdLaunch& a) { return fwd::launch_any<64>(a); }
}  // namespace fa
