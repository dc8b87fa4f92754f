// simt_gdn2.cu -- Gated DeltaNet-2 (separate per-channel erase and write gates) on the
// fp32 CUDA-core chunkwise path.
//
// Recurrence ("Linear Attention Architectures: Mechanisms, Trade-offs, and Cross-Layer
// Routing", section "Metodologia y Marco de Trabajo", item 1, the Gated DeltaNet-2
// bullet, which gives it in words: erase gates choose which key channels are removed,
// write gates which value channels are stored; read with the scalar decay of the Gated
// DeltaNet bullet), on the state S = W^T (d_k x d_v), per token:
//   Sd = alpha S;  p = Sd^T k;  S = Sd - b p^T + k vw^T;  o = scale S^T q
// with b = erase . k and vw = write . v (Gated DeltaNet when erase = write = beta).
//
// Chunkwise form over L <= C tokens from the chunk-start state S0 (Gamma = within-chunk
// cumulative log-decay, one scalar per token; the rows of P are the predictions p):
//   Kb = e^G K, Kr = e^-G K, Br = e^-G B, Qb = e^G Q, KC = e^{G_L - G} K, BC = e^{G_L - G} B
//   T  = (I + strict_lower(Kb Br^T))^{-1},   Mk = strict_lower(Kb Kr^T)
//   Wy = T Kb,  X = Mk Vw,  Pt = T X              so that  P = Pt + Wy S0
//   Aqk = tril(Qb Kr^T), Aqb = tril(Qb Br^T)
//   Qt = scale (Qb - Aqb Wy),  Ot = scale (Aqk Vw - Aqb Pt)   so that  O = Ot + Qt S0
//   S_L = e^{G_L} S0 + KC^T Vw - BC^T P
// (the predictions satisfy (I + strict_lower(Kb Br^T)) P = Kb S0 + Mk Vw: each p_t sees
// the decayed start state and every earlier write and erase of the chunk).  The
// backward is the chain rule through exactly these steps.  One CTA per (sequence, head,
// slice of bv value columns) walks its chunks; matrices live in a per-CTA scratch slice
// of the workspace.  The value columns of the state evolve independently (the key-side
// matrices T, Wy, Aqk, Aqb, Qt do not depend on v), so a slice recomputes the key side
// and carries only its columns of S, P and O.  In the backward, the key-side gradients
// (dq, dk, derase, dg) are sums over the slices of the same formulas: each slice writes
// its partial sums and a reduction kernel adds them in slice order.
#include "common.cuh"
#include "simt_util.cuh"
#include "trace.cuh"

namespace dr {
namespace {

constexpr int kThreads2 = 512;  // one CTA per (sequence, head): few CTAs, so wide ones

// Scratch matrices.  The first group is one chunk's: the forward writes it into a
// record per (chunk, head, slice), where a backward with DR_FLAG_REUSE_FWD finds the
// chunk's key-side matrices and predictions instead of recomputing them.  The second
// group (the carried state and the backward's work matrices) is per CTA.
enum {
    gQ, gK, gV, gE, gWg, gVw, gB, gGam, gKb, gKr, gBr, gQb, gKC, gBC, gA, gMk, gT, gWy, gX,
    gPt, gAqk, gAqb, gQt, gOt, gP, gO, gTmp,
    kChunkBufs,
    gS = kChunkBufs,
    // backward only
    gS0, gdS, gdSp, gdO, gdP, gdQt, gdWy, gdPt, gdX, gdMk, gdKC, gdBC, gdVw, gdAqk, gdAqb, gdQb,
    gdKb, gdKr, gdBr, gdT, gdA, gdGam, gdVec,
    kNumBufs2
};
constexpr int kCtaBufs = kNumBufs2 - kChunkBufs;

struct Scratch2 {
    float* chunk;  // this chunk's record
    float* cta;    // this CTA's matrices
    __device__ float* operator()(int i) const {
        return i < kChunkBufs ? chunk + (size_t)i * kBuf : cta + (size_t)(i - kChunkBufs) * kBuf;
    }
};

// record of chunk c (global index) of head h, value slice y (of nsl)
__device__ __forceinline__ float* chunk_record(float* area, const Params& p, int c, int h, int y,
                                               int nsl) {
    return area + (((size_t)c * p.H + h) * nsl + y) * kChunkBufs * kBuf;
}

__device__ void mask(float* M, int L, bool keep_diag) {
    for (int idx = threadIdx.x; idx < L * L; idx += blockDim.x) {
        const int i = idx / L, j = idx % L;
        if (keep_diag ? j > i : j >= i) M[idx] = 0.f;
    }
    __syncthreads();
}

// Load one chunk and evaluate everything that does not depend on the state.
// gGam holds Gamma_i at [i] and e^{Gamma_L} at [C].
__device__ void chunk_prep2(const Params& p, const Scratch2& s, int h, int row0, int L, int j0,
                            int dv) {
    const int dk = p.dk, H = p.H, tid = threadIdx.x, nt = blockDim.x;
    const float sc = p.scale;
    float* q = s(gQ); float* k = s(gK); float* v = s(gV); float* e = s(gE); float* w = s(gWg);
    float* gm = s(gGam);
    for (int idx = tid; idx < L * dk; idx += nt) {
        const size_t a = ((size_t)(row0 + idx / dk) * H + h) * dk + idx % dk;
        q[idx] = ld_any(p.q, a, p.io_dtype);
        k[idx] = ld_any(p.k, a, p.io_dtype);
        e[idx] = p.erase[a];
    }
    for (int idx = tid; idx < L * dv; idx += nt) {
        const size_t a = ((size_t)(row0 + idx / dv) * H + h) * p.dv + j0 + idx % dv;
        v[idx] = ld_any(p.v, a, p.io_dtype);
        w[idx] = p.write[a];
    }
    if (tid < 32) {
        // Gamma: inclusive scan of the chunk's log-decays (L <= 64: two per lane)
        const int lane = tid;
        float g0 = lane < L ? p.g[(size_t)(row0 + lane) * H + h] : 0.f;
        float g1 = lane + 32 < L ? p.g[(size_t)(row0 + lane + 32) * H + h] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t0 = __shfl_up_sync(0xffffffffu, g0, o);
            const float t1 = __shfl_up_sync(0xffffffffu, g1, o);
            if (lane >= o) {
                g0 += t0;
                g1 += t1;
            }
        }
        g1 += __shfl_sync(0xffffffffu, g0, 31);
        if (lane < L) gm[lane] = g0;
        if (lane + 32 < L) gm[lane + 32] = g1;
        const float last = L > 32 ? __shfl_sync(0xffffffffu, g1, (L - 33) & 31)
                                  : __shfl_sync(0xffffffffu, g0, (L - 1) & 31);
        if (lane == 0) gm[p.C] = expf(last);
    }
    __syncthreads();
    float* Bm = s(gB); float* Vw = s(gVw); float* Kb = s(gKb); float* Kr = s(gKr);
    float* Br = s(gBr); float* Qb = s(gQb); float* KC = s(gKC); float* BC = s(gBC);
    const float GL = gm[L - 1];
    for (int idx = tid; idx < L * dk; idx += nt) {
        const float G = gm[idx / dk];
        const float eG = expf(G), enG = expf(-G), eC = expf(GL - G);
        const float b = e[idx] * k[idx];
        Bm[idx] = b;
        Kb[idx] = k[idx] * eG;
        Kr[idx] = k[idx] * enG;
        Br[idx] = b * enG;
        Qb[idx] = q[idx] * eG;
        KC[idx] = k[idx] * eC;
        BC[idx] = b * eC;
    }
    for (int idx = tid; idx < L * dv; idx += nt) Vw[idx] = w[idx] * v[idx];
    __syncthreads();
    // A^T (column j of A = strict_lower(Kb Br^T) contiguous): AT[j][i] = Br_j . Kb_i, i > j
    float* AT = s(gA); float* T = s(gT); float* Mk = s(gMk);
    mm4(AT, L, Br, dk, false, Kb, dk, true, L, L, dk, 1.f, false);
    for (int idx = tid; idx < L * L; idx += nt)
        if (idx % L <= idx / L) AT[idx] = 0.f;
    mm4(Mk, L, Kb, dk, false, Kr, dk, true, L, L, dk, 1.f, false);
    mask(Mk, L, false);
    // T = (I + A)^{-1} by 2 x 2 blocks of 32: T11 = (I + A11)^{-1} and T22 = (I + A22)^{-1}
    // side by side (thread n of each half solves column n right-looking: once x_j is final
    // it is subtracted from every later row, so the dependent chain is one multiply-add
    // per row), T12 = 0, then T21 = -T22 (A21 T11) with two tiled products
    if (L == 64) {
        if (tid < 64) {
            const int o = tid & 32, n = tid & 31;
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = (i == n) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < 31; ++j) {
                const float xj = x[j];
                const float* col = AT + (o + j) * 64 + o;
#pragma unroll
                for (int i4 = (j + 1) & ~3; i4 < 32; i4 += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(col + i4);
                    if (i4 + 0 > j) x[i4 + 0] = fmaf(-a.x, xj, x[i4 + 0]);
                    if (i4 + 1 > j) x[i4 + 1] = fmaf(-a.y, xj, x[i4 + 1]);
                    if (i4 + 2 > j) x[i4 + 2] = fmaf(-a.z, xj, x[i4 + 2]);
                    if (i4 + 3 > j) x[i4 + 3] = fmaf(-a.w, xj, x[i4 + 3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                T[(o + i) * 64 + o + n] = x[i];
                if (o == 0) T[i * 64 + 32 + n] = 0.f;
            }
        }
        __syncthreads();
        float* Y = s(gTmp);  // [32][32]: A21 T11, with A21[i][k] = AT[k][32 + i]
        mm4(Y, 32, AT + 32, 64, true, T, 64, false, 32, 32, 32, 1.f, false);
        mm4(T + 32 * 64, 64, T + 32 * 64 + 32, 64, false, Y, 32, false, 32, 32, 32, -1.f, false);
    } else {
        // a chunk's ragged tail: forward substitution by rows
        for (int i = 0; i < L; ++i) {
            for (int n = tid; n < L; n += nt) {
                float x = (n == i) ? 1.f : 0.f;
                if (n < i)
                    for (int j = n; j < i; ++j) x -= AT[j * L + i] * T[j * L + n];
                T[i * L + n] = x;
            }
            __syncthreads();
        }
    }
    float* Wy = s(gWy); float* X = s(gX); float* Pt = s(gPt); float* Aqk = s(gAqk);
    float* Aqb = s(gAqb); float* Qt = s(gQt); float* Ot = s(gOt);
    mm4(Wy, dk, T, L, false, Kb, dk, false, L, dk, L, 1.f, false);
    mm4(X, dv, Mk, L, false, Vw, dv, false, L, dv, L, 1.f, false);
    mm4(Pt, dv, T, L, false, X, dv, false, L, dv, L, 1.f, false);
    mm4(Aqk, L, Qb, dk, false, Kr, dk, true, L, L, dk, 1.f, false);
    mask(Aqk, L, true);
    mm4(Aqb, L, Qb, dk, false, Br, dk, true, L, L, dk, 1.f, false);
    mask(Aqb, L, true);
    mm4(Qt, dk, Aqb, L, false, Wy, dk, false, L, dk, L, -sc, false);
    for (int idx = tid; idx < L * dk; idx += nt) Qt[idx] += sc * Qb[idx];
    mm4(Ot, dv, Aqk, L, false, Vw, dv, false, L, dv, L, sc, false);
    mm4(Ot, dv, Aqb, L, false, Pt, dv, false, L, dv, L, -sc, true);
}

// P = Pt + Wy S; O = Ot + Qt S; S <- e^{Gamma_L} S + KC^T Vw - BC^T P
__device__ void chunk_scan2(const Params& p, const Scratch2& s, int L, float* S, int dv) {
    const int dk = p.dk, tid = threadIdx.x, nt = blockDim.x;
    float* P = s(gP); float* O = s(gO);
    for (int idx = tid; idx < L * dv; idx += nt) { P[idx] = s(gPt)[idx]; O[idx] = s(gOt)[idx]; }
    __syncthreads();
    mm4(P, dv, s(gWy), dk, false, S, dv, false, L, dv, dk, 1.f, true);
    mm4(O, dv, s(gQt), dk, false, S, dv, false, L, dv, dk, 1.f, true);
    const float gL = s(gGam)[p.C];
    for (int idx = tid; idx < dk * dv; idx += nt) S[idx] *= gL;
    __syncthreads();
    mm4(S, dv, s(gKC), dk, true, s(gVw), dv, false, dk, dv, L, 1.f, true);
    mm4(S, dv, s(gBC), dk, true, P, dv, false, dk, dv, L, -1.f, true);
}

// S (d_k x bv, columns j0.. of the [d_k][d_v] state h) into scratch; zero when h is NULL
__device__ void load_state_cols(float* S, const float* h, int n, int hd, const Params& p, int j0,
                                int bv) {
    for (int idx = threadIdx.x; idx < p.dk * bv; idx += blockDim.x)
        S[idx] = h ? h[(((size_t)n * p.H + hd) * p.dk + idx / bv) * p.dv + j0 + idx % bv] : 0.f;
    __syncthreads();
}
__device__ void store_state_cols(float* h, const float* S, int n, int hd, const Params& p, int j0,
                                 int bv) {
    for (int idx = threadIdx.x; idx < p.dk * bv; idx += blockDim.x)
        h[(((size_t)n * p.H + hd) * p.dk + idx / bv) * p.dv + j0 + idx % bv] = S[idx];
}

// The forward also leaves the chunk-start states (this slice's columns) in `states`, where
// a backward with DR_FLAG_REUSE_FWD reads them instead of recomputing them.
__global__ void __launch_bounds__(kThreads2) gdn2_fwd_kernel(Params p, float* scratch, int bv,
                                                                float* records, float* states) {
    const int u = blockIdx.x, n = u / p.H, h = u % p.H, j0 = blockIdx.y * bv;
    Scratch2 s{nullptr, scratch + ((size_t)u * gridDim.y + blockIdx.y) * kCtaBufs * kBuf};
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);
    float* S = s(gS);
    load_state_cols(S, p.h0, n, h, p, j0, bv);
    const size_t SS = (size_t)p.dk * p.dv;
    for (int c = 0; c < nc; ++c) {
        const int row0 = srow + c * p.C, L = min(p.C, slen - c * p.C);
        float* dst = states + ((size_t)(c0 + c) * p.H + h) * SS;
        for (int idx = threadIdx.x; idx < p.dk * bv; idx += blockDim.x)
            dst[(idx / bv) * p.dv + j0 + idx % bv] = S[idx];
        s.chunk = chunk_record(records, p, c0 + c, h, blockIdx.y, gridDim.y);
        chunk_prep2(p, s, h, row0, L, j0, bv);
        chunk_scan2(p, s, L, S, bv);
        const float* O = s(gO);
        for (int idx = threadIdx.x; idx < L * bv; idx += blockDim.x) {
            const size_t a = ((size_t)(row0 + idx / bv) * p.H + h) * p.dv + j0 + idx % bv;
            st_any(p.o, a, p.out_dtype, O[idx]);
        }
        __syncthreads();
    }
    if (p.hT) store_state_cols(p.hT, S, n, h, p, j0, bv);
}

// Key-side gradient partials of one slice: [slice][token·head][d_k] for dq, dk, derase and
// [slice][token·head] for dg (null when there is one slice: the kernel writes the outputs).
struct Gdn2Partials {
    float *q, *k, *e, *g;
};

__global__ void __launch_bounds__(kThreads2) gdn2_bwd_kernel(Params p, float* scratch,
                                                                float* records, float* states,
                                                                int bv, Gdn2Partials part,
                                                                int reuse) {
    const int u = blockIdx.x, n = u / p.H, h = u % p.H, j0 = blockIdx.y * bv;
    const int dk = p.dk, dv = bv, C = p.C, tid = threadIdx.x, nt = blockDim.x;
    const float sc = p.scale;
    Scratch2 s{nullptr, scratch + ((size_t)u * gridDim.y + blockIdx.y) * kCtaBufs * kBuf};
    const size_t th = (size_t)p.B * p.T * p.H;
    const bool direct = part.q == nullptr;
    float* pq = direct ? nullptr : part.q + blockIdx.y * th * dk;
    float* pk = direct ? nullptr : part.k + blockIdx.y * th * dk;
    float* pe = direct ? nullptr : part.e + blockIdx.y * th * dk;
    float* pg = direct ? nullptr : part.g + blockIdx.y * th;
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);
    const size_t SS = (size_t)dk * p.dv;
    // pass 1: the state at the start of every chunk (this slice's columns), unless the
    // forward left them
    float* S = s(gS);
    if (!reuse) load_state_cols(S, p.h0, n, h, p, j0, bv);
    for (int c = 0; c < nc && !reuse; ++c) {
        const int row0 = srow + c * C, L = min(C, slen - c * C);
        float* dst = states + ((size_t)(c0 + c) * p.H + h) * SS;
        for (int idx = tid; idx < dk * dv; idx += nt) dst[(idx / dv) * p.dv + j0 + idx % dv] = S[idx];
        __syncthreads();
        s.chunk = chunk_record(records, p, c0 + c, h, blockIdx.y, gridDim.y);
        chunk_prep2(p, s, h, row0, L, j0, bv);
        chunk_scan2(p, s, L, S, bv);
    }
    // pass 2: reverse over chunks with dS = dL/dS_end
    float* dS = s(gdS);
    load_state_cols(dS, p.dhT, n, h, p, j0, bv);
    for (int c = nc - 1; c >= 0; --c) {
        const int row0 = srow + c * C, L = min(C, slen - c * C);
        float* S0 = s(gS0);
        const float* src = states + ((size_t)(c0 + c) * p.H + h) * SS;
        for (int idx = tid; idx < dk * dv; idx += nt) {
            const float x = src[(idx / dv) * p.dv + j0 + idx % dv];
            S0[idx] = x;
            S[idx] = x;
        }
        __syncthreads();
        s.chunk = chunk_record(records, p, c0 + c, h, blockIdx.y, gridDim.y);
        if (!reuse) {  // else the forward's record of this chunk holds all of it
            chunk_prep2(p, s, h, row0, L, j0, bv);
            chunk_scan2(p, s, L, S, bv);  // recomputes P (S is scratch here)
        }
        float* dO = s(gdO);
        for (int idx = tid; idx < L * dv; idx += nt)
            dO[idx] = ld_any(p.dO, ((size_t)(row0 + idx / dv) * p.H + h) * p.dv + j0 + idx % dv,
                             p.io_dtype);
        __syncthreads();
        const float gL = s(gGam)[C];
        float* dP = s(gdP); float* dSp = s(gdSp); float* dQt = s(gdQt); float* dWy = s(gdWy);
        float* dPt = s(gdPt); float* dKC = s(gdKC); float* dBC = s(gdBC); float* dVw = s(gdVw);
        float* dVec = s(gdVec);
        // state update S_L = gL S0 + KC^T Vw - BC^T P and the reads O = Ot + Qt S0
        mm4(dP, dv, s(gBC), dk, false, dS, dv, false, L, dv, dk, -1.f, false);
        for (int idx = tid; idx < dk * dv; idx += nt) dSp[idx] = gL * dS[idx];
        for (int c2 = tid; c2 < dk; c2 += nt) {
            float acc = 0.f;
            for (int j = 0; j < dv; ++j) acc += dS[c2 * dv + j] * S0[c2 * dv + j];
            dVec[c2] = acc;  // d e^{Gamma_L}, per key row
        }
        __syncthreads();
        mm4(dSp, dv, s(gQt), dk, true, dO, dv, false, dk, dv, L, 1.f, true);
        mm4(dSp, dv, s(gWy), dk, true, dP, dv, false, dk, dv, L, 1.f, true);
        mm4(dQt, dk, dO, dv, false, S0, dv, true, L, dk, dv, 1.f, false);
        mm4(dWy, dk, dP, dv, false, S0, dv, true, L, dk, dv, 1.f, false);
        mm4(dKC, dk, s(gVw), dv, false, dS, dv, true, L, dk, dv, 1.f, false);
        mm4(dBC, dk, s(gP), dv, false, dS, dv, true, L, dk, dv, -1.f, false);
        mm4(dVw, dv, s(gKC), dk, false, dS, dv, false, L, dv, dk, 1.f, false);
        for (int idx = tid; idx < L * dv; idx += nt) dPt[idx] = dP[idx];
        __syncthreads();
        // Qt = sc (Qb - Aqb Wy), Ot = sc (Aqk Vw - Aqb Pt)
        float* dAqk = s(gdAqk); float* dAqb = s(gdAqb); float* dQb = s(gdQb);
        mm4(dAqb, L, dQt, dk, false, s(gWy), dk, true, L, L, dk, -sc, false);
        mm4(dAqb, L, dO, dv, false, s(gPt), dv, true, L, L, dv, -sc, true);
        mask(dAqb, L, true);
        mm4(dAqk, L, dO, dv, false, s(gVw), dv, true, L, L, dv, sc, false);
        mask(dAqk, L, true);
        mm4(dWy, dk, s(gAqb), L, true, dQt, dk, false, L, dk, L, -sc, true);
        mm4(dVw, dv, s(gAqk), L, true, dO, dv, false, L, dv, L, sc, true);
        mm4(dPt, dv, s(gAqb), L, true, dO, dv, false, L, dv, L, -sc, true);
        for (int idx = tid; idx < L * dk; idx += nt) dQb[idx] = sc * dQt[idx];
        __syncthreads();
        // Wy = T Kb, Pt = T X, X = Mk Vw
        float* dT = s(gdT); float* dKb = s(gdKb); float* dX = s(gdX); float* dMk = s(gdMk);
        mm4(dT, L, dWy, dk, false, s(gKb), dk, true, L, L, dk, 1.f, false);
        mm4(dT, L, dPt, dv, false, s(gX), dv, true, L, L, dv, 1.f, true);
        mm4(dKb, dk, s(gT), L, true, dWy, dk, false, L, dk, L, 1.f, false);
        mm4(dX, dv, s(gT), L, true, dPt, dv, false, L, dv, L, 1.f, false);
        mm4(dMk, L, dX, dv, false, s(gVw), dv, true, L, L, dv, 1.f, false);
        mask(dMk, L, false);
        mm4(dVw, dv, s(gMk), L, true, dX, dv, false, L, dv, L, 1.f, true);
        // T = (I + A)^{-1}: dA = -T^T dT T^T (strictly lower); A = Kb Br^T, Mk = Kb Kr^T
        float* dA = s(gdA); float* tmp = s(gTmp); float* dKr = s(gdKr); float* dBr = s(gdBr);
        mm4(tmp, L, dT, L, false, s(gT), L, true, L, L, L, 1.f, false);
        mm4(dA, L, s(gT), L, true, tmp, L, false, L, L, L, -1.f, false);
        mask(dA, L, false);
        mm4(dKb, dk, dA, L, false, s(gBr), dk, false, L, dk, L, 1.f, true);
        mm4(dBr, dk, dA, L, true, s(gKb), dk, false, L, dk, L, 1.f, false);
        mm4(dKb, dk, dMk, L, false, s(gKr), dk, false, L, dk, L, 1.f, true);
        mm4(dKr, dk, dMk, L, true, s(gKb), dk, false, L, dk, L, 1.f, false);
        // Aqk = tril(Qb Kr^T), Aqb = tril(Qb Br^T)
        mm4(dQb, dk, dAqk, L, false, s(gKr), dk, false, L, dk, L, 1.f, true);
        mm4(dKr, dk, dAqk, L, true, s(gQb), dk, false, L, dk, L, 1.f, true);
        mm4(dQb, dk, dAqb, L, false, s(gBr), dk, false, L, dk, L, 1.f, true);
        mm4(dBr, dk, dAqb, L, true, s(gQb), dk, false, L, dk, L, 1.f, true);
        // decay and gate chain -> dq, dk, derase, dv, dwrite, dGamma
        const float* gm = s(gGam);
        float* dGam = s(gdGam);
        const float* k = s(gK); const float* e = s(gE);
        for (int idx = tid; idx < L * dk; idx += nt) {
            const int i = idx / dk;
            const float G = gm[i], GL = gm[L - 1];
            const float eG = expf(G), enG = expf(-G), eC = expf(GL - G);
            const float dB = dBr[idx] * enG + dBC[idx] * eC;
            const size_t a = ((size_t)(row0 + i) * p.H + h) * dk + idx % dk;
            const float gq = dQb[idx] * eG;
            const float gk = dKb[idx] * eG + dKr[idx] * enG + dKC[idx] * eC + e[idx] * dB;
            if (direct) {
                st_any(p.dq, a, p.grad_dtype, gq);
                st_any(p.dk_, a, p.grad_dtype, gk);
                p.derase[a] = k[idx] * dB;
            } else {
                pq[a] = gq;
                pk[a] = gk;
                pe[a] = k[idx] * dB;
            }
            tmp[idx] = dQb[idx] * s(gQb)[idx] + dKb[idx] * s(gKb)[idx] - dKr[idx] * s(gKr)[idx] -
                       dKC[idx] * s(gKC)[idx] - dBr[idx] * s(gBr)[idx] - dBC[idx] * s(gBC)[idx];
            dGam[idx] = dKC[idx] * s(gKC)[idx] + dBC[idx] * s(gBC)[idx];  // Gamma_L terms
        }
        for (int idx = tid; idx < L * dv; idx += nt) {
            const size_t a = ((size_t)(row0 + idx / dv) * p.H + h) * p.dv + j0 + idx % dv;
            st_any(p.dv_, a, p.grad_dtype, s(gWg)[idx] * dVw[idx]);
            p.dwrite[a] = s(gV)[idx] * dVw[idx];
        }
        __syncthreads();
        // dGamma_i = sum over channels (tmp); Gamma_L also collects the KC, BC terms (dGam)
        // and the e^{Gamma_L} one (dVec); dg = reverse cumulative sum.  Row sums by one
        // thread per token, then warp 0 adds the tail and scans.
        float* rs = dVec + 64;  // [0, L): per-token sums; [64, 128): per-token tail parts
        for (int i = tid; i < L; i += nt) {
            float a = 0.f, b = 0.f;
            for (int c2 = 0; c2 < dk; ++c2) {
                a += tmp[i * dk + c2];
                b += dGam[i * dk + c2];
            }
            rs[i] = a;
            rs[64 + i] = b;
        }
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            float tail = 0.f;
            for (int c2 = lane; c2 < dk; c2 += 32) tail += dVec[c2];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tail += __shfl_xor_sync(0xffffffffu, tail, o);
            tail *= gL;
            float tb = (lane < L ? rs[64 + lane] : 0.f) + (lane + 32 < L ? rs[96 + lane] : 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tb += __shfl_xor_sync(0xffffffffu, tb, o);
            tail += tb;
            // reverse inclusive scan over tokens L-1 .. 0 (two per lane, from the end)
            float d0 = lane < L ? rs[lane] : 0.f, d1 = lane + 32 < L ? rs[lane + 32] : 0.f;
            if (lane == ((L - 1) & 31)) {
                if (L > 32) d1 += tail;
                else d0 += tail;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t0 = __shfl_down_sync(0xffffffffu, d0, o);
                const float t1 = __shfl_down_sync(0xffffffffu, d1, o);
                if (lane + o < 32) {
                    d0 += t0;
                    d1 += t1;
                }
            }
            d0 += __shfl_sync(0xffffffffu, d1, 0);
            float* out = direct ? p.dg : pg;
            if (lane < L) out[(size_t)(row0 + lane) * p.H + h] = d0;
            if (lane + 32 < L) out[(size_t)(row0 + lane + 32) * p.H + h] = d1;
        }
        for (int idx = tid; idx < dk * dv; idx += nt) dS[idx] = dSp[idx];
        __syncthreads();
    }
    if (p.dh0) store_state_cols(p.dh0, dS, n, h, p, j0, bv);
}

// dq, dk, derase, dg = the slices' partial sums, added in slice order
__global__ void __launch_bounds__(256) gdn2_reduce_kernel(Params p, Gdn2Partials part, int nsl) {
    const size_t th = (size_t)p.B * p.T * p.H, n = th * p.dk;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) {
        float q = 0.f, k = 0.f, e = 0.f;
        for (int sl = 0; sl < nsl; ++sl) {
            q += part.q[sl * n + i];
            k += part.k[sl * n + i];
            e += part.e[sl * n + i];
        }
        st_any(p.dq, i, p.grad_dtype, q);
        st_any(p.dk_, i, p.grad_dtype, k);
        p.derase[i] = e;
        if (i < th) {
            float g = 0.f;
            for (int sl = 0; sl < nsl; ++sl) g += part.g[sl * th + i];
            p.dg[i] = g;
        }
    }
}


}  // namespace

// Value-column slices per (sequence, head): 16-column slices while there are fewer units
// than SMs (more CTAs for the same work), else one slice.
int gdn2_slices(int units, int dv) { return (units >= 152 || dv < 32) ? 1 : dv / 16; }

// Workspace after the header: the CTAs' matrices, the chunk records, the chunk-start
// states, then (with several slices) the partial key-side gradients.
size_t gdn2_workspace_bytes(int units, int num_chunks, int H, int dk, int dv, long long th) {
    const int nsl = gdn2_slices(units, dv);
    return (size_t)units * nsl * kCtaBufs * kBuf * sizeof(float) +
           (size_t)num_chunks * H * nsl * kChunkBufs * kBuf * sizeof(float) +
           (size_t)num_chunks * H * dk * dv * sizeof(float) +
           (nsl > 1 ? (size_t)nsl * (size_t)th * (3 * dk + 1) * sizeof(float) : 0);
}

cudaError_t gdn2_fwd(const Params& p, cudaStream_t st) {
    const int units = p.N * p.H;
    if (units == 0) return cudaSuccess;
    const int nsl = gdn2_slices(units, p.dv);
    float* scratch = reinterpret_cast<float*>(p.ws + 256);
    float* records = scratch + (size_t)units * nsl * kCtaBufs * kBuf;
    float* states = records + (size_t)p.num_chunks * p.H * nsl * kChunkBufs * kBuf;
    TraceScope ts("gdn2_fwd", st);
    gdn2_fwd_kernel<<<dim3(units, nsl), kThreads2, 0, st>>>(p, scratch, p.dv / nsl, records, states);
    return cudaGetLastError();
}

cudaError_t gdn2_bwd(const Params& p, cudaStream_t st, bool reuse) {
    const int units = p.N * p.H;
    if (units == 0) return cudaSuccess;
    const int nsl = gdn2_slices(units, p.dv);
    const size_t th = (size_t)p.B * p.T * p.H;
    float* scratch = reinterpret_cast<float*>(p.ws + 256);
    float* records = scratch + (size_t)units * nsl * kCtaBufs * kBuf;
    float* states = records + (size_t)p.num_chunks * p.H * nsl * kChunkBufs * kBuf;
    Gdn2Partials part{nullptr, nullptr, nullptr, nullptr};
    if (nsl > 1) {
        float* base = states + (size_t)p.num_chunks * p.H * p.dk * p.dv;
        const size_t n = (size_t)nsl * th * p.dk;
        part = Gdn2Partials{base, base + n, base + 2 * n, base + 3 * n};
    }
    {
        TraceScope ts("gdn2_bwd", st);
        gdn2_bwd_kernel<<<dim3(units, nsl), kThreads2, 0, st>>>(p, scratch, records, states,
                                                               p.dv / nsl, part, reuse ? 1 : 0);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nsl == 1) return e;
    const size_t n = th * p.dk;
    const int grid = (int)((n + 255) / 256 < 65536 ? (n + 255) / 256 : 65535);
    TraceScope ts("gdn2_reduce", st);
    gdn2_reduce_kernel<<<grid, 256, 0, st>>>(p, part, nsl);
    return cudaGetLastError();
}

}  // namespace dr
