// fa_bwd.cu — backward pass (in progress).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd_bf16(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
