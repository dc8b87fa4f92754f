// common.cuh -- shared device helpers and the launch-parameter block of the
// kernels of libdr.so.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dr.h"

namespace dr {

// Device-side error word (first 4 bytes of the workspace): nonzero after a
// bounded wait ran out.
constexpr int kErrTimeout = 1;
// Bound on any single wait of a kernel on its own asynchronous copies / MMAs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Everything a kernel may need.  Pointers that a given entry point does not use
// are null.  Token rows are addressed as row = b*T + t (dense) or the packed
// offset (ragged); element (row, head, c) of a [.., H, d] tensor sits at
// (row*H + head)*d + c.
struct Params {
    int B, T, H, dk, dv, C, variant, N;
    int io_dtype, out_dtype, grad_dtype;
    float scale;
    int num_chunks;           // total chunks over all sequences
    int chunks_per_seq;       // dense layout only
    const int32_t* cu;        // [N+1] or null
    const int32_t* ctab;      // [num_chunks][2] (seq, first row) or null
    const int32_t* coff;      // [N+1] first chunk of each sequence or null
    const void *q, *k, *v;
    const float *beta, *g, *h0;
    const float *erase, *write;  // Gated DeltaNet-2 gates: [.., H, dk] and [.., H, dv]
    void* o;
    float* hT;
    void* u;                  // optional: the write u = beta r, [.., H, dv] in out_dtype
    const void* dO;
    const float* dhT;
    const void* dU;           // optional: dL/du of that write, [.., H, dv] in io_dtype
    void *dq, *dk_, *dv_;
    float *dbeta, *dg, *dh0;
    float *derase, *dwrite;      // their gradients (Gated DeltaNet-2)
    int* err;                 // device error word
    uint8_t* ws;              // workspace base
    int prepare;              // tensor-core path: q, k, beta, g are raw (DR_FLAG_PREPARE_INPUTS)
};

// Input preparation of DR_FLAG_PREPARE_INPUTS, as the tensor-core kernels apply it on
// the fly: q_hat = q rsqrt(sum q^2 + eps), beta = sigmoid(b), g = -softplus(x).
constexpr float kPrepEps = 1e-6f;
__device__ __forceinline__ float prep_sigmoid(float b) { return 1.f / (1.f + expf(-b)); }
__device__ __forceinline__ float prep_neg_softplus(float x) {
    return -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
}
// Sum of x over an aligned group of N consecutive lanes (N a power of two, full warp).
template <int N>
__device__ __forceinline__ float lane_group_sum(float x) {
#pragma unroll
    for (int o = N / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// (sequence, first row, length) of global chunk `c`
__device__ __forceinline__ void chunk_info(const Params& p, int c, int& seq, int& row0, int& len) {
    if (p.ctab) {
        seq = p.ctab[2 * c];
        row0 = p.ctab[2 * c + 1];
        const int end = p.cu[seq + 1];
        len = min(p.C, end - row0);
    } else {
        seq = c / p.chunks_per_seq;
        const int t0 = (c % p.chunks_per_seq) * p.C;
        row0 = seq * p.T + t0;
        len = min(p.C, p.T - t0);
    }
}
// first chunk and chunk count of sequence n, and its first row
__device__ __forceinline__ void seq_chunks(const Params& p, int n, int& c0, int& nc, int& row0, int& len) {
    if (p.cu) {
        c0 = p.coff[n];
        nc = p.coff[n + 1] - c0;
        row0 = p.cu[n];
        len = p.cu[n + 1] - row0;
    } else {
        c0 = n * p.chunks_per_seq;
        nc = p.chunks_per_seq;
        row0 = n * p.T;
        len = p.T;
    }
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float ld_any(const void* p, size_t i, int dtype) {
    return dtype == DR_F32 ? static_cast<const float*>(p)[i]
                           : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}
__device__ __forceinline__ void st_any(void* p, size_t i, int dtype, float x) {
    if (dtype == DR_F32)
        static_cast<float*>(p)[i] = x;
    else
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
}

}  // namespace dr

namespace dr {
// Raise a kernel's dynamic shared-memory limit once per device: `done` keeps one bit per
// device ordinal (< 64) on which the attribute is set; safe for concurrent callers.
template <typename K>
inline cudaError_t set_smem_once(K kernel, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

}  // namespace dr
