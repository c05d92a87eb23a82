// Backward kernel instances (head dimensions 64 and 128).
#include "fa_bwd_kernel.cuh"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch& a) { return a.d == 64 ? bwd::launch<64>(a) : bwd::launch<128>(a); }
}  // namespace fa
