// Backward pass (to be filled in): returns "not supported" for now.
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch&) { return cudaErrorNotSupported; }
}  // namespace fa
