// simt_util.cuh -- block-wide fp32 helpers of the CUDA-core chunkwise kernels
// (simt.cu, simt_gdn2.cu): a plain matrix product over per-CTA scratch matrices and
// the state load.  Every helper is block-wide and ends with __syncthreads().
#pragma once

#include "common.cuh"

namespace dr {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kBuf = 64 * 64;  // floats per scratch matrix (C, d_k, d_v <= 64)

// C[m x n] = alpha * op(A) op(B) (+ C when acc).  op(A) is m x k.
__device__ void mm(float* Cm, int ldc, const float* A, int lda, bool ta, const float* Bm,
                   int ldb, bool tb, int m, int n, int k, float alpha, bool acc) {
    for (int idx = threadIdx.x; idx < m * n; idx += blockDim.x) {
        const int i = idx / n, j = idx % n;
        float s = 0.f;
        for (int p = 0; p < k; ++p) {
            const float a = ta ? A[p * lda + i] : A[i * lda + p];
            const float b = tb ? Bm[j * ldb + p] : Bm[p * ldb + j];
            s = fmaf(a, b, s);
        }
        Cm[i * ldc + j] = acc ? Cm[i * ldc + j] + alpha * s : alpha * s;
    }
    __syncthreads();
}

// The same product with each thread computing a 2 x 2 block of C (one pass over k
// loads two values of op(A) and two of op(B) for four multiply-adds).  Every output
// sums its k terms in the same order as mm.  Edges of odd m or n are bounds-checked.
__device__ void mm2(float* Cm, int ldc, const float* A, int lda, bool ta, const float* Bm,
                    int ldb, bool tb, int m, int n, int k, float alpha, bool acc) {
    const int mh = (m + 1) / 2, nh = (n + 1) / 2;
    for (int idx = threadIdx.x; idx < mh * nh; idx += blockDim.x) {
        const int i0 = 2 * (idx / nh), j0 = 2 * (idx % nh);
        const bool i1ok = i0 + 1 < m, j1ok = j0 + 1 < n;
        const int i1 = i1ok ? i0 + 1 : i0, j1 = j1ok ? j0 + 1 : j0;
        float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
        for (int p = 0; p < k; ++p) {
            const float a0 = ta ? A[p * lda + i0] : A[i0 * lda + p];
            const float a1 = ta ? A[p * lda + i1] : A[i1 * lda + p];
            const float b0 = tb ? Bm[j0 * ldb + p] : Bm[p * ldb + j0];
            const float b1 = tb ? Bm[j1 * ldb + p] : Bm[p * ldb + j1];
            s00 = fmaf(a0, b0, s00);
            s01 = fmaf(a0, b1, s01);
            s10 = fmaf(a1, b0, s10);
            s11 = fmaf(a1, b1, s11);
        }
        float* c0 = Cm + i0 * ldc;
        c0[j0] = acc ? c0[j0] + alpha * s00 : alpha * s00;
        if (j1ok) c0[j1] = acc ? c0[j1] + alpha * s01 : alpha * s01;
        if (i1ok) {
            float* c1 = Cm + i1 * ldc;
            c1[j0] = acc ? c1[j0] + alpha * s10 : alpha * s10;
            if (j1ok) c1[j1] = acc ? c1[j1] + alpha * s11 : alpha * s11;
        }
    }
    __syncthreads();
}

struct Scratch {
    float* base;
    __device__ float* operator()(int i) const { return base + (size_t)i * kBuf; }
};

__device__ void load_state(float* S, const float* h, int n, int hd, int H, int dk, int dv) {
    for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x)
        S[idx] = h ? h[((size_t)n * H + hd) * dk * dv + idx] : 0.f;
    __syncthreads();
}

}  // namespace
}  // namespace dr
