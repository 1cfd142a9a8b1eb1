// bwd_bf16_sm103.cu -- backward pass by recomputation (placeholder until the
// tensor-core kernel lands: reports "not supported").
#include "kernels.h"

namespace fa {

cudaError_t launch_bwd_bf16_tc(const BwdParams&, const BwdMaps&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
