#include "common.cuh"
namespace dr {
size_t tc_workspace_bytes(const Params&) { return 0; }
cudaError_t tc_fwd(const Params&, cudaStream_t, bool) { return cudaErrorNotSupported; }
cudaError_t tc_bwd(const Params&, cudaStream_t, bool) { return cudaErrorNotSupported; }
}
