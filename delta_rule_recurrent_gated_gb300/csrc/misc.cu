// misc.cu -- small helper kernels.
#include "common.cuh"
#include "tc.cuh"
#include "trace.cuh"

namespace dr {
namespace {
// dst = src (or 0 when src is null): the state of a sequence with no tokens
// passes through unchanged (hT = h0, dh0 = dhT).
__global__ void copy_or_zero(const float* __restrict__ src, float* __restrict__ dst, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : 0.f;
}

// Self-test of the kernels' failure path: thread 0 initialises an mbarrier; with
// `arrive` it completes the barrier's first phase itself, otherwise nothing ever does.
// Every thread then waits on that phase with the same bounded wait (tc::mbar_wait on
// %globaltimer) the tensor-core kernels use, and a wait that runs out records
// kErrTimeout in the workspace error word the way they do.  Nothing is copied and no
// tensor memory is held, so an expired wait leaves nothing in flight.
__global__ void wait_selftest_kernel(int* err, int arrive, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) tc::mbar_arrive_expect_tx(&bar, 0);
    const bool ok = tc::mbar_wait(&bar, 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicExch(err, kErrTimeout);
}
}  // namespace

cudaError_t wait_selftest(int* err, int arrive, unsigned long long limit_ns, cudaStream_t st) {
    TraceScope ts("wait_selftest", st);
    wait_selftest_kernel<<<1, 32, 0, st>>>(err, arrive, limit_ns);
    return cudaGetLastError();
}

cudaError_t state_passthrough(const float* src, float* dst, size_t n, cudaStream_t st) {
    if (n == 0 || !dst) return cudaSuccess;
    const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    TraceScope ts("copy_or_zero", st);
    copy_or_zero<<<blocks, 256, 0, st>>>(src, dst, n);
    return cudaGetLastError();
}
}  // namespace dr
