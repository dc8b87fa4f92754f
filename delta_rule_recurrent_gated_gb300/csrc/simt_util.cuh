// simt_util.cuh -- block-wide fp32 helpers of the CUDA-core chunkwise kernels
// (simt.cu, simt_gdn2.cu): a plain matrix product over per-CTA scratch matrices and
// the state load.  Every helper is block-wide and ends with __syncthreads().
#pragma once

#include "common.cuh"

namespace dr {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kBuf = 64 * 64;  // floats per scratch matrix when C, d_k, d_v <= 64

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
// sums its k terms in the same order as mm.  When the shapes allow (even m and n, k and
// the leading dimensions multiples of 4), four steps of k are loaded at once: float4
// along k for an operand read along its rows, float2 across the 2 x 2 pair for one read
// down its columns; otherwise the scalar loop.  Operands start on 16-byte boundaries.
// A warp covers a patch of 4 x 8 output pairs (rows x columns), so a load of A touches
// at most 4 rows of it and a load of B at most 8.
template <bool TA, bool TB>
__device__ __forceinline__ void mm2_body(float* Cm, int ldc, const float* A, int lda,
                                         const float* Bm, int ldb, int m, int n, int k,
                                         float alpha, bool acc) {
    const int mh = (m + 1) / 2, nh = (n + 1) / 2;
    const bool vec = (m % 2 == 0) && (n % 2 == 0) && (k % 4 == 0) && (lda % 4 == 0) &&
                     (ldb % 4 == 0);
    const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int tm = (mh + 3) / 4, tn = (nh + 7) / 8;
    for (int t = threadIdx.x >> 5; t < tm * tn; t += nwarps) {
        const int pi = (t / tn) * 4 + (lane & 3), pj = (t % tn) * 8 + (lane >> 2);
        if (pi >= mh || pj >= nh) continue;
        const int i0 = 2 * pi, j0 = 2 * pj;
        const bool i1ok = i0 + 1 < m, j1ok = j0 + 1 < n;
        const int i1 = i1ok ? i0 + 1 : i0, j1 = j1ok ? j0 + 1 : j0;
        float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
        int p = 0;
        if (vec) {
            for (; p < k; p += 4) {
                float a0[4], a1[4], b0[4], b1[4];
                if (TA) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 t = *reinterpret_cast<const float2*>(A + (p + q) * lda + i0);
                        a0[q] = t.x;
                        a1[q] = t.y;
                    }
                } else {
                    const float4 t0 = *reinterpret_cast<const float4*>(A + i0 * lda + p);
                    const float4 t1 = *reinterpret_cast<const float4*>(A + i1 * lda + p);
                    a0[0] = t0.x; a0[1] = t0.y; a0[2] = t0.z; a0[3] = t0.w;
                    a1[0] = t1.x; a1[1] = t1.y; a1[2] = t1.z; a1[3] = t1.w;
                }
                if (TB) {
                    const float4 t0 = *reinterpret_cast<const float4*>(Bm + j0 * ldb + p);
                    const float4 t1 = *reinterpret_cast<const float4*>(Bm + j1 * ldb + p);
                    b0[0] = t0.x; b0[1] = t0.y; b0[2] = t0.z; b0[3] = t0.w;
                    b1[0] = t1.x; b1[1] = t1.y; b1[2] = t1.z; b1[3] = t1.w;
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 t = *reinterpret_cast<const float2*>(Bm + (p + q) * ldb + j0);
                        b0[q] = t.x;
                        b1[q] = t.y;
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    s00 = fmaf(a0[q], b0[q], s00);
                    s01 = fmaf(a0[q], b1[q], s01);
                    s10 = fmaf(a1[q], b0[q], s10);
                    s11 = fmaf(a1[q], b1[q], s11);
                }
            }
        }
        for (; p < k; ++p) {
            const float a0 = TA ? A[p * lda + i0] : A[i0 * lda + p];
            const float a1 = TA ? A[p * lda + i1] : A[i1 * lda + p];
            const float b0 = TB ? Bm[j0 * ldb + p] : Bm[p * ldb + j0];
            const float b1 = TB ? Bm[j1 * ldb + p] : Bm[p * ldb + j1];
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
}

__device__ void mm2(float* Cm, int ldc, const float* A, int lda, bool ta, const float* Bm,
                    int ldb, bool tb, int m, int n, int k, float alpha, bool acc) {
    if (ta) {
        if (tb) mm2_body<true, true>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
        else mm2_body<true, false>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
    } else {
        if (tb) mm2_body<false, true>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
        else mm2_body<false, false>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
    }
    __syncthreads();
}

// The same product with 4 x 4 blocks of C per thread, four steps of k per pass (float4
// along k for an operand read along its rows, float4 across the block for one read down
// its columns): two loads per 16 multiply-adds instead of mm2's one per 4.  For shapes
// that are multiples of 4 (m, n, k and the leading dimensions); otherwise mm2.  Each
// output sums its k terms in order, like mm.
template <bool TA, bool TB>
__device__ __forceinline__ void mm4_body(float* Cm, int ldc, const float* A, int lda,
                                         const float* Bm, int ldb, int m, int n, int k,
                                         float alpha, bool acc) {
    const int mt = m / 4, nt = n / 4;
    for (int t = threadIdx.x; t < mt * nt; t += blockDim.x) {
        const int i0 = 4 * (t / nt), j0 = 4 * (t % nt);
        float c[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) c[a][b] = 0.f;
        for (int p = 0; p < k; p += 4) {
            float av[4][4], bv[4][4];  // av[row a][step q], bv[col b][step q]
            if (TA) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(A + (p + q) * lda + i0);
                    av[0][q] = x.x; av[1][q] = x.y; av[2][q] = x.z; av[3][q] = x.w;
                }
            } else {
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float4 x = *reinterpret_cast<const float4*>(A + (i0 + a) * lda + p);
                    av[a][0] = x.x; av[a][1] = x.y; av[a][2] = x.z; av[a][3] = x.w;
                }
            }
            if (TB) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float4 x = *reinterpret_cast<const float4*>(Bm + (j0 + b) * ldb + p);
                    bv[b][0] = x.x; bv[b][1] = x.y; bv[b][2] = x.z; bv[b][3] = x.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(Bm + (p + q) * ldb + j0);
                    bv[0][q] = x.x; bv[1][q] = x.y; bv[2][q] = x.z; bv[3][q] = x.w;
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) c[a][b] = fmaf(av[a][q], bv[b][q], c[a][b]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float* cr = Cm + (i0 + a) * ldc + j0;
#pragma unroll
            for (int b = 0; b < 4; ++b) cr[b] = acc ? cr[b] + alpha * c[a][b] : alpha * c[a][b];
        }
    }
}

__device__ void mm4(float* Cm, int ldc, const float* A, int lda, bool ta, const float* Bm,
                    int ldb, bool tb, int m, int n, int k, float alpha, bool acc) {
    if ((m | n | k | lda | ldb) & 3) {
        mm2(Cm, ldc, A, lda, ta, Bm, ldb, tb, m, n, k, alpha, acc);
        return;
    }
    if (ta) {
        if (tb) mm4_body<true, true>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
        else mm4_body<true, false>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
    } else {
        if (tb) mm4_body<false, true>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
        else mm4_body<false, false>(Cm, ldc, A, lda, Bm, ldb, m, n, k, alpha, acc);
    }
    __syncthreads();
}

// Matrix i of a CTA's scratch slice; `buf` floats per matrix.
struct Scratch {
    float* base;
    int buf;
    __device__ float* operator()(int i) const { return base + (size_t)i * buf; }
};

__device__ void load_state(float* S, const float* h, int n, int hd, int H, int dk, int dv) {
    for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x)
        S[idx] = h ? h[((size_t)n * H + hd) * dk * dv + idx] : 0.f;
    __syncthreads();
}

}  // namespace
}  // namespace dr
