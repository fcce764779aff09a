// Tensor-core (tcgen05) backward kernels -- not written yet.
#include "fa_internal.cuh"
namespace fa {
cudaError_t launch_tc_bwd(const Problem&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
