// simt.cu -- fp32 CUDA-core path (no tensor cores) of the chunkwise delta rule:
// serves fp32 inputs, where the tolerance asks for fp32 arithmetic throughout.
//
// One CTA per (sequence, head) walks its chunks in order.  Each chunk of L <= C
// tokens, starting from the state S (d_k x d_v, S = W^T), is evaluated in the
// chunkwise form of the recurrence (decay before the residual, residual
// r = v - (decayed W) k, write beta r k^T, read W q; page "Linear Attention
// Architectures: Mechanisms, Trade-offs, and Cross-Layer Routing", section
// "Metodologia y Marco de Trabajo", item 1):
//   Gamma = within-chunk cumulative sum of the log-decay (per key channel)
//   Kb = k e^{Gamma}, Kr = k e^{-Gamma}, Qb = q e^{Gamma}, KC = k e^{Gamma_L - Gamma}
// (in the two Gram-type products, Kb Kr^T and Qb Kr^T, the factors are taken relative to
// Gamma_r, the cumulative log-decay at the chunk's middle token, so that neither overflows
// while each half of the chunk decays by less than e^-87; Wy and Qt use e^{Gamma} <= 1)
//   T  = (I + diag(beta) strict_lower(Kb Kr^T))^{-1}
//   Wy = T diag(beta) Kb,  Ut = T diag(beta) v,  Aqk = tril(Qb Kr^T)
//   Qt = scale (Qb - Aqk Wy),  Ot = scale Aqk Ut
//   U  = Ut - Wy S,  O = Qt S + Ot,  S <- diag(e^{Gamma_L}) S + KC^T U
// and the backward pass is the chain rule through exactly these steps.
// Small matrices live in a per-CTA scratch slice of the workspace (L1/L2
// resident); every helper is block-wide and ends with __syncthreads().
#include <mutex>

#include "common.cuh"
#include "simt_util.cuh"
#include "trace.cuh"

namespace dr {
namespace {

constexpr int kThreads = kSimtThreads;

enum {
    bS, bQ, bK, bV, bGam, bKb, bKr, bQb, bKC, bA, bT, bbK, bbV, bWy, bUt, bAqk, bQt, bOt, bU,
    bO, bVec, bTmp,
    // backward only
    bS0, bdS, bdSp, bdO, bdU, bdQt, bdWy, bdUt, bdKC, bdAqk, bdQb, bdKr, bdKb, bdT, bdA,
    bdbK, bdbV, bdGam, bdVec,
    kNumBufs
};

// Load one chunk's inputs into scratch and evaluate everything that does not
// depend on the state (steps Gamma .. Ot above).
__device__ void chunk_prep(const Params& p, const Scratch& s, int h, int row0, int L) {
    const int dk = p.dk, dv = p.dv, H = p.H, tid = threadIdx.x, nt = blockDim.x;
    float* q = s(bQ); float* k = s(bK); float* v = s(bV); float* gm = s(bGam);
    float* beta = s(bVec);  // [0, C): beta;  [C, C + dk): e^{Gamma_L};  [C + dk, C + 2 dk): Gamma_r
    for (int idx = tid; idx < L * dk; idx += nt) {
        const int i = idx / dk, c = idx % dk;
        const size_t e = ((size_t)(row0 + i) * H + h) * dk + c;
        q[idx] = ld_any(p.q, e, p.io_dtype);
        k[idx] = ld_any(p.k, e, p.io_dtype);
    }
    for (int idx = tid; idx < L * dv; idx += nt) {
        const int i = idx / dv, c = idx % dv;
        v[idx] = ld_any(p.v, ((size_t)(row0 + i) * H + h) * dv + c, p.io_dtype);
    }
    for (int i = tid; i < L; i += nt) beta[i] = p.beta[(size_t)(row0 + i) * H + h];
    // Gamma: within-chunk inclusive cumulative sum of the log-decay
    for (int c = tid; c < dk; c += nt) {
        float acc = 0.f;
        for (int i = 0; i < L; ++i) {
            float gi = 0.f;
            if (p.variant == DR_GDN) gi = p.g[(size_t)(row0 + i) * H + h];
            else if (p.variant == DR_KDA) gi = p.g[((size_t)(row0 + i) * H + h) * dk + c];
            acc += gi;
            gm[i * dk + c] = acc;
        }
        beta[p.C + c] = expf(acc);
    }
    __syncthreads();
    float* Kb = s(bKb); float* Kr = s(bKr); float* Qb = s(bQb); float* KC = s(bKC);
    float* bK = s(bbK); float* bV = s(bbV);
    float* Gr = beta + p.C + dk;
    for (int c = tid; c < dk; c += nt) Gr[c] = gm[((L - 1) / 2) * dk + c];
    __syncthreads();
    for (int idx = tid; idx < L * dk; idx += nt) {
        const int i = idx / dk, c = idx % dk;
        const float G = gm[idx], GL = gm[(L - 1) * dk + c], R = Gr[c];
        Kb[idx] = k[idx] * expf(G - R);   // Kb' (Gram)
        Kr[idx] = k[idx] * expf(R - G);   // Kr' (both Gram-type products)
        Qb[idx] = q[idx] * expf(G - R);   // Qb' (Aqk)
        KC[idx] = k[idx] * expf(GL - G);
        bK[idx] = beta[i] * k[idx] * expf(G);  // beta Kb with the absolute factor (Wy)
    }
    for (int idx = tid; idx < L * dv; idx += nt) bV[idx] = beta[idx / dv] * v[idx];
    __syncthreads();
    float* A = s(bA); float* T = s(bT);
    mm4(A, L, Kb, dk, false, Kr, dk, true, L, L, dk, 1.f, false);  // Gram (kept for backward)
    // T = (I + diag(beta) strict_lower(Gram))^{-1}, forward substitution by rows
    for (int i = 0; i < L; ++i) {
        for (int n = tid; n < L; n += nt) {
            float x = (n == i) ? 1.f : 0.f;
            if (n < i)
                for (int j = n; j < i; ++j) x -= beta[i] * A[i * L + j] * T[j * L + n];
            T[i * L + n] = x;
        }
        __syncthreads();
    }
    float* Wy = s(bWy); float* Ut = s(bUt); float* Aqk = s(bAqk);
    mm4(Wy, dk, T, L, false, bK, dk, false, L, dk, L, 1.f, false);
    mm4(Ut, dv, T, L, false, bV, dv, false, L, dv, L, 1.f, false);
    mm4(Aqk, L, Qb, dk, false, Kr, dk, true, L, L, dk, 1.f, false);
    for (int idx = tid; idx < L * L; idx += nt)
        if (idx % L > idx / L) Aqk[idx] = 0.f;
    __syncthreads();
    float* Qt = s(bQt); float* Ot = s(bOt);
    mm4(Qt, dk, Aqk, L, false, Wy, dk, false, L, dk, L, -p.scale, false);
    for (int idx = tid; idx < L * dk; idx += nt) Qt[idx] += p.scale * q[idx] * expf(gm[idx]);
    mm4(Ot, dv, Aqk, L, false, Ut, dv, false, L, dv, L, p.scale, false);
}

// U = Ut - Wy S; O = Qt S + Ot; S <- diag(e^{Gamma_L}) S + KC^T U
__device__ void chunk_scan(const Params& p, const Scratch& s, int L, float* S) {
    const int dk = p.dk, dv = p.dv, tid = threadIdx.x, nt = blockDim.x;
    float* U = s(bU); float* O = s(bO);
    for (int idx = tid; idx < L * dv; idx += nt) { U[idx] = s(bUt)[idx]; O[idx] = s(bOt)[idx]; }
    __syncthreads();
    mm4(U, dv, s(bWy), dk, false, S, dv, false, L, dv, dk, -1.f, true);
    mm4(O, dv, s(bQt), dk, false, S, dv, false, L, dv, dk, 1.f, true);
    const float* gL = s(bVec) + p.C;
    for (int idx = tid; idx < dk * dv; idx += nt) S[idx] *= gL[idx / dv];
    __syncthreads();
    mm4(S, dv, s(bKC), dk, true, U, dv, false, dk, dv, L, 1.f, true);
}

// Forward of one (sequence, head) unit per CTA over the scratch slice s.
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(Params p, float* scratch,
                                                            size_t unit_floats, int buf) {
    const int u = blockIdx.x, n = u / p.H, h = u % p.H;
    const Scratch s{scratch + (size_t)u * unit_floats, buf};
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);
    float* S = s(bS);
    load_state(S, p.h0, n, h, p.H, p.dk, p.dv);
    for (int c = 0; c < nc; ++c) {
        const int row0 = srow + c * p.C, L = min(p.C, slen - c * p.C);
        chunk_prep(p, s, h, row0, L);
        chunk_scan(p, s, L, S);
        const float* O = s(bO);
        const float* U = s(bU);
        for (int idx = threadIdx.x; idx < L * p.dv; idx += blockDim.x) {
            const int i = idx / p.dv, j = idx % p.dv;
            const size_t e = ((size_t)(row0 + i) * p.H + h) * p.dv + j;
            st_any(p.o, e, p.out_dtype, O[idx]);
            if (p.u) st_any(p.u, e, p.out_dtype, U[idx]);  // the write beta r
        }
        __syncthreads();
    }
    if (p.hT)
        for (int idx = threadIdx.x; idx < p.dk * p.dv; idx += blockDim.x)
            p.hT[((size_t)n * p.H + h) * p.dk * p.dv + idx] = S[idx];
}

__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(Params p, float* scratch,
                                                            float* states, int buf) {
    const int u = blockIdx.x, n = u / p.H, h = u % p.H;
    const int dk = p.dk, dv = p.dv, C = p.C, tid = threadIdx.x, nt = blockDim.x;
    const Scratch s{scratch + (size_t)u * kNumBufs * buf, buf};
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);
    const size_t SS = (size_t)dk * dv;
    // pass 1: the state at the start of every chunk
    float* S = s(bS);
    load_state(S, p.h0, n, h, p.H, dk, dv);
    for (int c = 0; c < nc; ++c) {
        const int row0 = srow + c * C, L = min(C, slen - c * C);
        float* dst = states + ((size_t)(c0 + c) * p.H + h) * SS;
        for (int idx = tid; idx < dk * dv; idx += nt) dst[idx] = S[idx];
        __syncthreads();
        chunk_prep(p, s, h, row0, L);
        chunk_scan(p, s, L, S);
    }
    // pass 2: reverse over chunks with dS = dL/dS_end
    float* dS = s(bdS);
    load_state(dS, p.dhT, n, h, p.H, dk, dv);
    for (int c = nc - 1; c >= 0; --c) {
        const int row0 = srow + c * C, L = min(C, slen - c * C);
        float* S0 = s(bS0);
        const float* src = states + ((size_t)(c0 + c) * p.H + h) * SS;
        for (int idx = tid; idx < dk * dv; idx += nt) { S0[idx] = src[idx]; S[idx] = src[idx]; }
        __syncthreads();
        chunk_prep(p, s, h, row0, L);
        chunk_scan(p, s, L, S);  // recomputes U (S is scratch here)
        float* dO = s(bdO);
        for (int idx = tid; idx < L * dv; idx += nt) {
            const int i = idx / dv, j = idx % dv;
            dO[idx] = ld_any(p.dO, ((size_t)(row0 + i) * p.H + h) * dv + j, p.io_dtype);
        }
        __syncthreads();
        const float* beta = s(bVec);
        const float* gL = s(bVec) + C;
        float* dU = s(bdU); float* dSp = s(bdSp);
        // dU = KC dS;  dS_prev = diag(gL) dS + Qt^T dO - Wy^T dU
        mm4(dU, dv, s(bKC), dk, false, dS, dv, false, L, dv, dk, 1.f, false);
        if (p.dU) {  // plus the gradient of the emitted write
            for (int idx = tid; idx < L * dv; idx += nt) {
                const int i = idx / dv, j = idx % dv;
                dU[idx] += ld_any(p.dU, ((size_t)(row0 + i) * p.H + h) * dv + j, p.io_dtype);
            }
            __syncthreads();
        }
        for (int idx = tid; idx < dk * dv; idx += nt) dSp[idx] = gL[idx / dv] * dS[idx];
        __syncthreads();
        mm4(dSp, dv, s(bQt), dk, true, dO, dv, false, dk, dv, L, 1.f, true);
        mm4(dSp, dv, s(bWy), dk, true, dU, dv, false, dk, dv, L, -1.f, true);
        // state-side gradients of the chunk
        float* dQt = s(bdQt); float* dWy = s(bdWy); float* dUt = s(bdUt); float* dKC = s(bdKC);
        mm4(dQt, dk, dO, dv, false, S0, dv, true, L, dk, dv, 1.f, false);
        mm4(dWy, dk, dU, dv, false, S0, dv, true, L, dk, dv, -1.f, false);
        mm4(dKC, dk, s(bU), dv, false, dS, dv, true, L, dk, dv, 1.f, false);
        float* dVec = s(bdVec);  // [0, dk): d e^{Gamma_L}; [128, 128 + C): dbeta
        for (int c2 = tid; c2 < dk; c2 += nt) {
            float acc = 0.f;
            for (int j = 0; j < dv; ++j) acc += dS[c2 * dv + j] * S0[c2 * dv + j];
            dVec[c2] = acc;
        }
        for (int idx = tid; idx < L * dv; idx += nt) dUt[idx] = dU[idx];
        __syncthreads();
        // Qt = scale (Qb - Aqk Wy), Ot = scale Aqk Ut
        const float sc = p.scale;
        float* dAqk = s(bdAqk); float* dQb = s(bdQb);
        mm4(dAqk, L, dQt, dk, false, s(bWy), dk, true, L, L, dk, -sc, false);
        mm4(dAqk, L, dO, dv, false, s(bUt), dv, true, L, L, dv, sc, true);
        for (int idx = tid; idx < L * L; idx += nt)
            if (idx % L > idx / L) dAqk[idx] = 0.f;
        __syncthreads();
        mm4(dWy, dk, s(bAqk), L, true, dQt, dk, false, L, dk, L, -sc, true);
        mm4(dUt, dv, s(bAqk), L, true, dO, dv, false, L, dv, L, sc, true);
        __syncthreads();
        // Aqk = tril(Qb Kr^T)
        float* dKr = s(bdKr); float* dKb = s(bdKb);
        mm4(dQb, dk, dAqk, L, false, s(bKr), dk, false, L, dk, L, 1.f, false);  // of Qb' 
        mm4(dKr, dk, dAqk, L, true, s(bQb), dk, false, L, dk, L, 1.f, false);
        // Wy = T bK, Ut = T bV
        float* dT = s(bdT); float* dbK = s(bdbK); float* dbV = s(bdbV); float* dA = s(bdA);
        float* tmp = s(bTmp);
        mm4(dT, L, dWy, dk, false, s(bbK), dk, true, L, L, dk, 1.f, false);
        mm4(dT, L, dUt, dv, false, s(bbV), dv, true, L, L, dv, 1.f, true);
        mm4(dbK, dk, s(bT), L, true, dWy, dk, false, L, dk, L, 1.f, false);
        mm4(dbV, dv, s(bT), L, true, dUt, dv, false, L, dv, L, 1.f, false);
        // T = (I + A)^{-1}: dA = -T^T dT T^T, strictly lower
        mm4(tmp, L, dT, L, false, s(bT), L, true, L, L, L, 1.f, false);
        mm4(dA, L, s(bT), L, true, tmp, L, false, L, L, L, -1.f, false);
        for (int idx = tid; idx < L * L; idx += nt)
            if (idx % L >= idx / L) dA[idx] = 0.f;
        __syncthreads();
        // A = diag(beta) strict_lower(Kb Kr^T) (Gram kept in bA)
        float* db = dVec + 128;  // per-token dbeta partials (after the d_k <= 128 values)
        const float* Gm = s(bA);
        for (int i = tid; i < L; i += nt) {
            float acc = 0.f;
            for (int j = 0; j < i; ++j) acc += dA[i * L + j] * Gm[i * L + j];
            for (int c2 = 0; c2 < dk; ++c2)  // beta Kb with the absolute factor
                acc += dbK[i * dk + c2] * s(bK)[i * dk + c2] * expf(s(bGam)[i * dk + c2]);
            for (int j = 0; j < dv; ++j) acc += dbV[i * dv + j] * s(bV)[i * dv + j];
            db[i] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < L * L; idx += nt) dA[idx] *= beta[idx / L];
        __syncthreads();
        mm4(dKb, dk, dA, L, false, s(bKr), dk, false, L, dk, L, 1.f, false);
        mm4(dKr, dk, dA, L, true, s(bKb), dk, false, L, dk, L, 1.f, true);
        // decay chain -> dq, dk, dv, dbeta, dGamma
        float* dGam = s(bdGam);
        const float* gm = s(bGam);
        for (int idx = tid; idx < L * dk; idx += nt) {
            const int i = idx / dk, c2 = idx % dk;
            // dKb, dKr, dQb hold the gradients of Kb', Kr', Qb'; sc dQt and beta dbK those of
            // the absolute Qb and Kb
            const float G = gm[idx], GL = gm[(L - 1) * dk + c2], R = s(bVec)[C + dk + c2];
            const float eG = expf(G), er = expf(G - R), eri = expf(R - G), eC = expf(GL - G);
            const float dQa = sc * s(bdQt)[idx], dKa = beta[i] * dbK[idx];
            const float qa = s(bQ)[idx] * eG, ka = s(bK)[idx] * eG;
            const size_t e = ((size_t)(row0 + i) * p.H + h) * dk + c2;
            st_any(p.dq, e, p.grad_dtype, dQa * eG + dQb[idx] * er);
            st_any(p.dk_, e, p.grad_dtype,
                   dKa * eG + dKb[idx] * er + dKr[idx] * eri + dKC[idx] * eC);
            dGam[idx] = dQa * qa + dQb[idx] * s(bQb)[idx] + dKa * ka + dKb[idx] * s(bKb)[idx] -
                        dKr[idx] * s(bKr)[idx] - dKC[idx] * s(bKC)[idx];
        }
        for (int idx = tid; idx < L * dv; idx += nt) {
            const int i = idx / dv, j = idx % dv;
            st_any(p.dv_, ((size_t)(row0 + i) * p.H + h) * dv + j, p.grad_dtype,
                   beta[i] * dbV[idx]);
        }
        for (int i = tid; i < L; i += nt) p.dbeta[(size_t)(row0 + i) * p.H + h] = db[i];
        __syncthreads();
        if (p.variant != DR_DELTANET) {
            // Gamma_L terms, then dg = reverse cumulative sum of dGamma
            for (int c2 = tid; c2 < dk; c2 += nt) {
                float acc = dVec[c2] * gL[c2];
                for (int i = 0; i < L; ++i) acc += dKC[i * dk + c2] * s(bKC)[i * dk + c2];
                dGam[(L - 1) * dk + c2] += acc;
                float run = 0.f;
                for (int i = L - 1; i >= 0; --i) {
                    run += dGam[i * dk + c2];
                    dGam[i * dk + c2] = run;
                }
            }
            __syncthreads();
            if (p.variant == DR_KDA) {
                for (int idx = tid; idx < L * dk; idx += nt) {
                    const int i = idx / dk, c2 = idx % dk;
                    p.dg[((size_t)(row0 + i) * p.H + h) * dk + c2] = dGam[idx];
                }
            } else {
                for (int i = tid; i < L; i += nt) {
                    float acc = 0.f;
                    for (int c2 = 0; c2 < dk; ++c2) acc += dGam[i * dk + c2];
                    p.dg[(size_t)(row0 + i) * p.H + h] = acc;
                }
            }
        }
        for (int idx = tid; idx < dk * dv; idx += nt) dS[idx] = dSp[idx];
        __syncthreads();
    }
    if (p.dh0)
        for (int idx = tid; idx < dk * dv; idx += nt)
            p.dh0[((size_t)n * p.H + h) * SS + idx] = dS[idx];
}

}  // namespace

// Floats per scratch matrix: every matrix of a chunk is at most max(C, d_k, d_v)
// squared (4096 for the sizes up to 64, 16384 at d = 128).
int simt_buf_floats(int C, int dk, int dv) {
    const int m = max(64, max(C, max(dk, dv)));
    return m * m;
}

size_t simt_workspace_bytes(int units, int num_chunks, int H, int dk, int dv, int C) {
    return (size_t)units * kNumBufs * simt_buf_floats(C, dk, dv) * sizeof(float) +
           (size_t)num_chunks * H * dk * dv * sizeof(float);
}

cudaError_t simt_fwd(const Params& p, cudaStream_t st) {
    const int units = p.N * p.H;
    if (units == 0) return cudaSuccess;
    float* scratch = reinterpret_cast<float*>(p.ws + 256);
    const int buf = simt_buf_floats(p.C, p.dk, p.dv);
    TraceScope ts("simt_fwd", st);
    simt_fwd_kernel<<<units, kThreads, 0, st>>>(p, scratch, (size_t)kNumBufs * buf, buf);
    return cudaGetLastError();
}

cudaError_t simt_bwd(const Params& p, cudaStream_t st) {
    const int units = p.N * p.H;
    if (units == 0) return cudaSuccess;
    const int buf = simt_buf_floats(p.C, p.dk, p.dv);
    float* scratch = reinterpret_cast<float*>(p.ws + 256);
    float* states = scratch + (size_t)units * kNumBufs * buf;
    TraceScope ts("simt_bwd", st);
    simt_bwd_kernel<<<units, kThreads, 0, st>>>(p, scratch, states, buf);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Forward without a caller-supplied workspace (dr_fwd_noalloc in dr.h).
//
// Some callers cannot allocate device memory at the point where they run this
// layer: code that is handed only its input and output buffers by a host
// framework, or that runs where a cudaMalloc would synchronise the device or
// is not allowed.  For them the scratch of the fp32 forward kernel lives in
// one file-scope device array owned by the library instead of the workspace.
// The array is a fixed kNoAllocScratchBytes on every GPU that loads the
// library and stays allocated until the process exits.  All calls share it:
// two calls whose kernels overlap on the GPU (different streams or devices
// sharing a context) race on it.  The kernel writes every scratch word before
// it reads it, so stale contents from an earlier call never leak into a result
// and nothing needs clearing.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;       // 16 MiB per GPU
constexpr int kNoAllocBufs = bTmp + 1;                          // forward-only buffers
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {
// Device address of g_noalloc_scratch, looked up once per device with that
// device current, and cached by device ordinal for the life of the process
// (the address belongs to the device's primary context; it is not valid after
// a cudaDeviceReset of that device, nor in another context made current on
// it).  The host-side name of the array is only a stand-in for the symbol;
// the kernel must receive this address.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

cudaError_t noalloc_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<float*>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}
}  // namespace

// Largest number of (sequence, head) units the static scratch holds for a problem
// of these sizes (the forward keeps kNoAllocBufs matrices per unit).
int simt_noalloc_max_units(int C, int dk, int dv) {
    return (int)(kNoAllocScratchBytes /
                 ((size_t)kNoAllocBufs * simt_buf_floats(C, dk, dv) * sizeof(float)));
}

// The forward kernel of this file over the static scratch, with the forward-only
// per-unit stride.
cudaError_t simt_fwd_noalloc(const Params& p, cudaStream_t st) {
    const int units = p.N * p.H;
    if (units == 0) return cudaSuccess;
    float* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    const int buf = simt_buf_floats(p.C, p.dk, p.dv);
    TraceScope ts("simt_fwd_noalloc", st);
    simt_fwd_kernel<<<units, kThreads, 0, st>>>(p, scratch, (size_t)kNoAllocBufs * buf, buf);
    return cudaGetLastError();
}

}  // namespace dr
