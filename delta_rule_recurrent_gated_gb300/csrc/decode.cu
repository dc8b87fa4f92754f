// decode.cu -- the recurrent step of the delta rule, token by token, on a state
// that stays resident in fp32 (inference: one or a few new tokens per sequence).
//
// Per (sequence n, head h), for each token t of the call in order, on
// S = W^T in [d_k][d_v] (the layout of h0 / hT):
//   S~ = D_t S                         (decay rows: DeltaNet none, GDN e^{g_t},
//                                       KDA e^{g_t[c]} on key channel c)
//   r  = v_t - S~^T k_t                (the residual the write corrects)
//   S  = S~ + beta_t k_t r^T           (delta-rule write)
//   o_t = scale S^T q_t                (read after the write)
// which is "The Delta Rule and its gated forms" recurrence step read directly,
// without chunking.
//
// One CTA per (sequence, head, 32 value columns): warp w owns key rows
// [w*R, (w+1)*R) of those columns, lane j column v0 + j, so every state row is
// read and written as 32 consecutive floats.  The two sums over key channels
// per token (S~^T k and S^T q) are per-thread partials over R rows, combined
// across the eight warps through shared memory in a fixed order.
//
// Gated DeltaNet-2 (GDN2): the same step with the erase gate e (per key channel) and
// the write gate w (per value channel) in place of beta: with p = S~^T k,
//   S = S~ - (e . k) p^T + k (w . v)^T      (Gated DeltaNet when e = w = beta),
// the decay the scalar one of Gated DeltaNet.
//
// With input preparation (PREP) the token's q and k are L2-normalised in shared
// memory (q * rsqrt(sum q^2 + 1e-6)), beta = sigmoid(b) and the gate
// log alpha = -softplus(x) are formed as they are read: the same maps as the
// chunked path's preparation kernels, applied here without a pass over HBM.
#include "common.cuh"
#include "trace.cuh"

namespace dr {
namespace {

constexpr int kDecodeThreads = 256;  // eight warps

__device__ __forceinline__ float neg_softplus(float x) {
    return -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
}

template <int DK, bool PREP, bool GDN2>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_kernel(const Params p, float* __restrict__ state) {
    constexpr int R = DK / 8;  // key rows per warp
    const int nh = blockIdx.x, n = nh / p.H, h = nh % p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncol = min(32, p.dv);
    const int v = blockIdx.y * ncol + lane;
    const bool col = lane < ncol;
    __shared__ float qs[DK], ks[DK], as[DK], es[GDN2 ? DK : 1], vs[32], ws[32];
    __shared__ float red[8][33];
    __shared__ float bsh, nrm_q, nrm_k;

    float* Sg = state + ((size_t)n * p.H + h) * DK * p.dv;
    float S[R];
#pragma unroll
    for (int i = 0; i < R; ++i) S[i] = col ? Sg[(size_t)(warp * R + i) * p.dv + v] : 0.f;

    for (int t = 0; t < p.T; ++t) {
        const size_t tok = (size_t)n * p.T + t;
        const size_t rk = (tok * p.H + h) * DK, rv = (tok * p.H + h) * p.dv;
        for (int c = threadIdx.x; c < DK; c += kDecodeThreads) {
            qs[c] = ld_any(p.q, rk + c, p.io_dtype);
            ks[c] = ld_any(p.k, rk + c, p.io_dtype);
            float a = 1.f;
            if (p.variant == DR_GDN || GDN2) {
                const float lg = p.g[tok * p.H + h];
                a = expf(PREP ? neg_softplus(lg) : lg);
            } else if (p.variant == DR_KDA) {
                const float lg = p.g[rk + c];
                a = expf(PREP ? neg_softplus(lg) : lg);
            }
            as[c] = a;
            if constexpr (GDN2) es[c] = p.erase[rk + c];
        }
        if (warp == 0) {
            vs[lane] = col ? ld_any(p.v, rv + v, p.io_dtype) : 0.f;
            if constexpr (GDN2) {
                ws[lane] = col ? p.write[rv + v] : 0.f;
            } else if (lane == 0) {
                const float b = p.beta[tok * p.H + h];
                bsh = PREP ? 1.f / (1.f + expf(-b)) : b;
            }
        }
        __syncthreads();
        if (PREP) {
            // warp 0 sums q^2, warp 1 k^2; every warp then reads both scales
            if (warp < 2) {
                const float* x = warp == 0 ? qs : ks;
                float ss = 0.f;
                for (int c = lane; c < DK; c += 32) ss = fmaf(x[c], x[c], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane == 0) (warp == 0 ? nrm_q : nrm_k) = rsqrtf(ss + 1e-6f);
            }
            __syncthreads();
        }
        // the norms enter as scales: S~^T k_hat = nrm_k (S~^T k), S^T q_hat = nrm_q (S^T q)
        const float scq = PREP ? nrm_q : 1.f, sck = PREP ? nrm_k : 1.f;
        // decay, then this thread's part of (S~^T k)[v]
        float pk = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int c = warp * R + i;
            S[i] *= as[c];
            pk = fmaf(S[i], ks[c], pk);
        }
        red[warp][lane] = pk;
        __syncthreads();
        float sk = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sk += red[w][lane];
        float pq = 0.f;
        if constexpr (GDN2) {
            // S = S~ - (e . k) p^T + k (w . v)^T on column v: p[v] = sk
            const float wv = ws[lane] * vs[lane];
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int c = warp * R + i;
                S[i] = fmaf(ks[c], wv, fmaf(-es[c] * ks[c], sk, S[i]));
                pq = fmaf(S[i], qs[c], pq);
            }
        } else {
            const float br = bsh * (vs[lane] - sck * sk);  // beta * r[v]
            const float brk = br * sck;                    // k_hat[c] = sck * ks[c]
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int c = warp * R + i;
                S[i] = fmaf(ks[c], brk, S[i]);
                pq = fmaf(S[i], qs[c], pq);
            }
        }
        __syncthreads();  // every warp has read red[] and the token's inputs
        red[warp][lane] = pq;
        __syncthreads();
        if (warp == 0 && col) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) o += red[w][lane];
            st_any(p.o, rv + v, p.out_dtype, p.scale * scq * o);
        }
        __syncthreads();  // red[] and the inputs are rewritten by the next token
    }
    if (col) {
#pragma unroll
        for (int i = 0; i < R; ++i) Sg[(size_t)(warp * R + i) * p.dv + v] = S[i];
    }
}

template <int DK>
cudaError_t launch(const Params& p, float* state, cudaStream_t st, bool prepare) {
    const int ncol = p.dv < 32 ? p.dv : 32;
    const dim3 grid(p.B * p.H, p.dv / ncol);
    TraceScope ts("decode", st);
    if (p.variant == DR_GDN2) decode_kernel<DK, false, true><<<grid, kDecodeThreads, 0, st>>>(p, state);
    else if (prepare) decode_kernel<DK, true, false><<<grid, kDecodeThreads, 0, st>>>(p, state);
    else decode_kernel<DK, false, false><<<grid, kDecodeThreads, 0, st>>>(p, state);
    return cudaGetLastError();
}

}  // namespace

// d_k in {16, 32, 64, 128}; d_v in {16, 32, 64, 128}; checked by the caller.  Gated
// DeltaNet-2 (p.variant == DR_GDN2) reads p.erase / p.write instead of p.beta.
cudaError_t decode(const Params& p, float* state, cudaStream_t st, bool prepare) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    switch (p.dk) {
        case 16: return launch<16>(p, state, st, prepare);
        case 32: return launch<32>(p, state, st, prepare);
        case 64: return launch<64>(p, state, st, prepare);
        default: return launch<128>(p, state, st, prepare);
    }
}

}  // namespace dr
