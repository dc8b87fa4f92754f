#include "common.cuh"
namespace dr {
cudaError_t tc_bwd(const Params&, cudaStream_t, bool) { return cudaErrorNotSupported; }
}
