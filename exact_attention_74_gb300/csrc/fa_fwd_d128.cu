// Forward kernel instances for head dimension 128.
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d128(const FwdLaunch& a) { return fwd::launch_any<128>(a); }
}  // namespace fa
