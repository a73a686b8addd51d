// varlen_bwd.cu -- placeholder until the backward kernels land.
#include "varlen_internal.h"
namespace varlen {
cudaError_t launch_bwd(const BwdLaunch&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace varlen
