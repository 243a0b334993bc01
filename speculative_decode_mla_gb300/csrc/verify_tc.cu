// tcgen05 split-KV tree-verify kernel (placeholder until the tensor-core path lands).
#include "common.cuh"

namespace mla {
int tc_kernel_supported() { return 0; }
cudaError_t launch_verify_tc(const VerifyArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
