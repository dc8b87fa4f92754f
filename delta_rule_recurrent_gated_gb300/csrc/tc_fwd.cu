// tc_fwd.cu -- bf16 tensor-core forward of the chunkwise delta rule (sm_103a).
//
// The recurrence (page "Linear Attention Architectures: Mechanisms, Trade-offs,
// and Cross-Layer Routing", section "Metodologia y Marco de Trabajo", item 1:
// decay the memory before the residual, residual r = v - (decayed W) k, write
// beta r k^T, read W q) is evaluated per 64-token chunk in its UT/WY form.  With
// Gamma the within-chunk cumulative log-decay per key channel:
//   Kb = k e^{Gamma}, Kr = k e^{-Gamma}, Qb = q e^{Gamma}, KC = k e^{Gamma_last - Gamma}
//   T  = (I + diag(beta) strict_lower(Kb Kr^T))^{-1}          (the UT inverse)
//   Wy = T diag(beta) Kb,  Ut = T diag(beta) v,  Aqk = tril(Qb Kr^T)
//   Qt = scale (Qb - Aqk Wy),  Ot = scale Aqk Ut
// The two Gram-type products (Kb Kr^T, Qb Kr^T) only need the decay between two
// tokens, e^{Gamma_i - Gamma_j}, so their operands take the exponents relative to
// Gamma_r, the cumulative log-decay at the chunk's 32nd token: Kb' = k e^{Gamma -
// Gamma_r}, Kr' = k e^{Gamma_r - Gamma}, Qb' = q e^{Gamma - Gamma_r}.  Each factor
// then spans only the decay of one half-chunk (its exponent stays within the fp32
// range while each 32-token half decays by less than e^{-87}); Wy and Qt use the
// absolute e^{Gamma} <= 1.
// and, from the state S at the chunk start (W = S^T),
//   U = Ut - Wy S  (the writes beta r),  O = Qt S + Ot,
//   S_next = diag(e^{Gamma_last}) S + KC^T U.
//
// Kernel 1, tc_prep: one CTA per (chunk, head), fully parallel.  TMA loads the
// q/k/v tiles, CUDA cores apply the decay, tcgen05 computes the two Gram
// products, CUDA cores invert the unit-lower-triangular 64x64 matrix (2x2 blocks
// of 32 rows), tcgen05 forms Wy, Ut, Aqk Wy, Aqk Ut.  Writes Wy, Qt, KC (tile
// images), Ut, Ot (token rows), T and e^{Gamma_last}.
// Kernel 2, tc_scan_fwd: one CTA per (sequence, head, value tile of BV rows),
// sequential over the sequence's chunks.  The state slice W[v0:v0+BV, :] stays
// in fp32 registers (half a row per thread); per chunk one tcgen05 product
// ([Wy; Qt] W^T) gives U and O, and one more (U^T KC) the state increment.
// Also stores the chunk-start state S and U for the backward pass; o leaves by
// tensor stores from shared memory.
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "tc.cuh"
#include "tc_layout.cuh"
#include "trace.cuh"

namespace dr {
using namespace tc;

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

template <int VAR>
__device__ __forceinline__ float gate_at(const Params& p, int row, int h, int c) {
    if (VAR == DR_GDN) return p.g[(size_t)row * p.H + h];
    return p.g[((size_t)row * p.H + h) * p.dk + c];
}

__device__ __forceinline__ void record_timeout(const Params& p) {
    if (threadIdx.x == 0) atomicExch(p.err, kErrTimeout);
}

// ============================================================== tc_prep
template <int D>
struct PrepSmem {
    static constexpr int kTile = 64 * D * 2;
    static constexpr int kQ = 0, kK = kTile, kV = 2 * kTile, kX = 3 * kTile, kY = 4 * kTile;
    static constexpr int kAq = 5 * kTile, kT = kAq + 8192;
    static constexpr int kAf = (D == 128) ? kX : kT + 8192;  // fp32 [64][64] (16 KB)
    // fp32 blocks of the inverse (12 KB): the consumed Kr tile when it is large enough
    static constexpr int kInv = (D == 128) ? kK : kT + 8192 + 16384;
    static constexpr int kBeta = (D == 128) ? kT + 8192 : kT + 8192 + 16384 + 12288;
    static constexpr int kGL = kBeta + 256;              // [D] fp32 e^{Gamma_last - Gamma_r}
    static constexpr int kRf = kGL + D * 4;              // [D] fp32 e^{Gamma_r}; then Gamma_r (KDA)
    static constexpr int kRn = kRf + 2 * D * 4;          // [2][64] inverse norms of q, k rows
    static constexpr int kBytes = kRn + 2 * 64 * 4 + 1024;  // + alignment slack
};

// Inverse L2 norms of the 64 q and k rows of [64][D] SW128 tiles (DR_FLAG_PREPARE_INPUTS):
// a row's D / 8 threads are consecutive lanes and sum its squares by shuffles; all rows of
// a thread are loaded before any reduction so that the shuffle chains overlap.
template <int D, int NT>
__device__ __forceinline__ void row_inv_norms(const uint8_t* Qs, const uint8_t* Ks, float* rq, float* rk) {
    constexpr int kIt = 64 * (D / 8) / NT;
    static_assert(kIt * NT == 64 * (D / 8), "whole warps per pass");
    float sq[kIt], sk[kIt];
#pragma unroll
    for (int n = 0; n < kIt; ++n) {
        const int w = threadIdx.x + n * NT, i = w / (D / 8), c8 = (w % (D / 8)) * 8;
        const uint32_t off = sw128_offset(i, c8, 64);
        float q8[8], k8[8];
        unpack8(*reinterpret_cast<const uint4*>(Qs + off), q8);
        unpack8(*reinterpret_cast<const uint4*>(Ks + off), k8);
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            a = fmaf(q8[j], q8[j], a);
            b = fmaf(k8[j], k8[j], b);
        }
        sq[n] = a;
        sk[n] = b;
    }
#pragma unroll
    for (int n = 0; n < kIt; ++n) {
        sq[n] = lane_group_sum<D / 8>(sq[n]);
        sk[n] = lane_group_sum<D / 8>(sk[n]);
    }
#pragma unroll
    for (int n = 0; n < kIt; ++n) {
        const int w = threadIdx.x + n * NT;
        if (w % (D / 8) == 0) {
            rq[w / (D / 8)] = rsqrtf(sq[n] + kPrepEps);
            rk[w / (D / 8)] = rsqrtf(sk[n] + kPrepEps);
        }
    }
}

template <int D, int VAR, bool PREP>
__global__ void __launch_bounds__(128, 1)
    tc_prep_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                   const Params p, const TcLayout L) {
    using S = PrepSmem<D>;
    constexpr int kTile = S::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Qs = sm + S::kQ;   // q -> Qb
    uint8_t* Ks = sm + S::kK;   // k -> Kr -> Ut
    uint8_t* Vs = sm + S::kV;   // v -> beta v
    uint8_t* Xs = sm + S::kX;   // Kb -> (A fp32 when D == 128) -> Wy
    uint8_t* Ys = sm + S::kY;   // beta Kb
    uint8_t* Aqs = sm + S::kAq; // tril(Qb Kr^T) [64][64]
    uint8_t* Ts = sm + S::kT;   // T [64][64]
    float* Af = reinterpret_cast<float*>(sm + S::kAf);
    float* beta_s = reinterpret_cast<float*>(sm + S::kBeta);
    float* GLs = reinterpret_cast<float*>(sm + S::kGL);
    float* Rf = reinterpret_cast<float*>(sm + S::kRf);   // e^{Gamma_r} per key channel
    float* Gr = Rf + D;                                  // KDA: Gamma_r per key channel
    float* RQ = reinterpret_cast<float*>(sm + S::kRn);   // input preparation: 1 / |q row|
    float* RK = RQ + 64;                                 // and 1 / |k row|
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_base;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int chunk = blockIdx.x, h = blockIdx.y;
    int seq, row0, len;
    chunk_info(p, chunk, seq, row0, len);
    const size_t rec = (size_t)chunk * p.H + h;

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
        prefetch_tmap(&mq);
        prefetch_tmap(&mk);
        prefetch_tmap(&mv);
        if (VAR == DR_KDA) prefetch_tmap(&mg);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = warp_lane_base(tm);
    const int r2 = m64_row_x2(), h2 = m64_half_x2();  // M = 64 row and column half (tmem_ld16_x2)
    bool ok = true;
    bool ld_phase2 = false;  // KDA: the second gate copy was issued

    do {
        if (tid == 0) {
            // KDA: the gates of the first 32 tokens come with q, k, v (the second 32 later,
            // into the same staging buffer)
            mbar_arrive_expect_tx(&bar_ld, 3 * kTile + (VAR == DR_KDA ? 32 * D * 4 : 0));
            for (int kb = 0; kb < D / 64; ++kb) {
                tma_load_3d(Qs + kb * 8192, &mq, &bar_ld, kb * 64, h, row0);
                tma_load_3d(Ks + kb * 8192, &mk, &bar_ld, kb * 64, h, row0);
                tma_load_3d(Vs + kb * 8192, &mv, &bar_ld, kb * 64, h, row0);
            }
            if (VAR == DR_KDA) {
                tma_load_3d(Aqs, &mg, &bar_ld, 0, h, row0);
                tma_prefetch_3d(&mg, 0, h, row0 + 32);  // the second half's gates, into L2
            }
        }
        // GDN's log-decays (two per lane of warp 0) are read while the tiles land
        float ga0 = 0.f, ga1 = 0.f;
        if (VAR == DR_GDN && warp == 0) {
            const int ln2 = 2 * (tid & 31);
            ga0 = ln2 < len ? p.g[(size_t)(row0 + ln2) * p.H + h] : 0.f;
            ga1 = ln2 + 1 < len ? p.g[(size_t)(row0 + ln2 + 1) * p.H + h] : 0.f;
        }
        if (tid < 64) {
            const float b = tid < len ? p.beta[(size_t)(row0 + tid) * p.H + h] : 0.f;
            beta_s[tid] = tid < len ? (PREP ? prep_sigmoid(b) : b) : 0.f;
        }
        ok = mbar_wait(&bar_ld, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;

        // rows past the end of the sequence hold another sequence's tokens: zero them
        {
            const int pad = 64 - len;
            const int per_tile = (D / 64) * pad * 8;
            for (int w = tid; w < 3 * per_tile; w += 128) {
                const int t = w / per_tile, rem = w % per_tile;
                const int kb = rem / (pad * 8), rr = len + (rem % (pad * 8)) / 8, ch = rem % 8;
                uint8_t* base = (t == 0 ? Qs : t == 1 ? Ks : Vs) + kb * 8192;
                *reinterpret_cast<uint4*>(base + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        __syncthreads();
        if (PREP) {  // raw q, k rows: their inverse norms, applied in the decay pass
            row_inv_norms<D, 128>(Qs, Ks, RQ, RK);
            __syncthreads();
            if (tid == 0) {  // the norms for the backward chunk kernel (RQ, RK contiguous)
                bulk_s2g(L.RN + rec * 128, RQ, 512);
                bulk_commit();
            }
        }

        // decay, per token (DeltaNet, GDN): warp 0 scans the 64 log-decays, two per lane, and
        // keeps e^{Gamma - Gamma_r}, e^{Gamma_r - Gamma}, e^{Gamma_last - Gamma} and e^{Gamma}
        // per token in the still-unused Aqk tile; then an elementwise pass eight channels wide
        if (VAR != DR_KDA) {
            float* Er = reinterpret_cast<float*>(Aqs);  // [4][64]
            if (warp == 0) {
                const int lane = tid & 31;
                float a0 = 0.f, a1 = 0.f;
                if (VAR == DR_GDN) {
                    a0 = ga0;
                    a1 = ga1;
                    if (PREP) {
                        a0 = 2 * lane < len ? prep_neg_softplus(a0) : 0.f;
                        a1 = 2 * lane + 1 < len ? prep_neg_softplus(a1) : 0.f;
                    }
                }
                float x = a0 + a1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                const float GL = __shfl_sync(0xffffffffu, x, 31);
                const float G_r = __shfl_sync(0xffffffffu, x, 15);  // Gamma at token 31
                const bool dec = VAR != DR_DELTANET;
                const float x0 = x - a1;
                Er[2 * lane] = dec ? __expf(x0 - G_r) : 1.f;
                Er[2 * lane + 1] = dec ? __expf(x - G_r) : 1.f;
                Er[64 + 2 * lane] = dec ? __expf(G_r - x0) : 1.f;
                Er[64 + 2 * lane + 1] = dec ? __expf(G_r - x) : 1.f;
                Er[128 + 2 * lane] = dec ? __expf(GL - x0) : 1.f;
                Er[128 + 2 * lane + 1] = dec ? __expf(GL - x) : 1.f;
                Er[192 + 2 * lane] = dec ? __expf(x0) : 1.f;
                Er[192 + 2 * lane + 1] = dec ? __expf(x) : 1.f;
                const float eGL = dec ? expf(GL) : 1.f, eGr = dec ? expf(G_r) : 1.f;
                for (int c = lane; c < D; c += 32) {
                    L.gC[rec * D + c] = eGL;  // e^{Gamma_last}
                    Rf[c] = eGr;
                }
            }
            __syncthreads();
            uint8_t* kc_img = L.KC + rec * kTile;
            for (int w = tid; w < 64 * (D / 8); w += 128) {
                const int i = w / (D / 8), c8 = (w % (D / 8)) * 8;
                const uint32_t off = sw128_offset(i, c8, 64);
                float q8[8], k8[8], v8[8];
                unpack8(*reinterpret_cast<const uint4*>(Qs + off), q8);
                unpack8(*reinterpret_cast<const uint4*>(Ks + off), k8);
                unpack8(*reinterpret_cast<const uint4*>(Vs + off), v8);
                if (PREP) {
                    const float rq = RQ[i], rk = RK[i];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        q8[j] *= rq;
                        k8[j] *= rk;
                    }
                }
                const float b = beta_s[i], e = Er[i], ei = Er[64 + i], ec = Er[128 + i],
                            ea = Er[192 + i];
                uint32_t wq[4], wr[4], wb[4], wy[4], wv[4], wc[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float k0 = k8[2 * j], k1 = k8[2 * j + 1];
                    wq[j] = pack_bf16(q8[2 * j] * e, q8[2 * j + 1] * e);
                    wr[j] = pack_bf16(k0 * ei, k1 * ei);
                    wb[j] = pack_bf16(k0 * e, k1 * e);
                    wy[j] = pack_bf16(b * k0 * ea, b * k1 * ea);
                    wv[j] = pack_bf16(b * v8[2 * j], b * v8[2 * j + 1]);
                    wc[j] = pack_bf16(k0 * ec, k1 * ec);
                }
                *reinterpret_cast<uint4*>(Qs + off) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                *reinterpret_cast<uint4*>(Ks + off) = make_uint4(wr[0], wr[1], wr[2], wr[3]);
                *reinterpret_cast<uint4*>(Xs + off) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                *reinterpret_cast<uint4*>(Ys + off) = make_uint4(wy[0], wy[1], wy[2], wy[3]);
                *reinterpret_cast<uint4*>(Vs + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                *reinterpret_cast<uint4*>(kc_img + off) = make_uint4(wc[0], wc[1], wc[2], wc[3]);
            }
        } else
        // decay, per key channel (KDA): the gates arrive 32 tokens at a time in the
        // still-unused Aqk / T tiles; thread c carries its channel's cumulative log-decay
        // through both halves in place (Gamma_r is its value after the first half), then an
        // elementwise pass eight channels wide.  KC = Kr' e^{Gamma_last - Gamma_r} is written
        // once the last token's Gamma is known.
        {
            float* Gb = reinterpret_cast<float*>(Aqs);  // [32][D] fp32
            float G = 0.f;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                if (half == 1) {
                    if (tid == 0) {
                        mbar_arrive_expect_tx(&bar_ld, 32 * D * 4);
                        tma_load_3d(Aqs, &mg, &bar_ld, 0, h, row0 + 32);
                    }
                    ok = mbar_wait(&bar_ld, 1, kWaitLimitNs);
                    ld_phase2 = true;
                    if (__syncthreads_or(!ok)) break;
                }
                if (tid < D) {
                    // 16 rows at a time: the loads are issued together, then the dependent sums
#pragma unroll
                    for (int i0 = 0; i0 < 32; i0 += 16) {
                        float x[16];
#pragma unroll
                        for (int ii = 0; ii < 16; ++ii) x[ii] = Gb[(i0 + ii) * D + tid];
#pragma unroll
                        for (int ii = 0; ii < 16; ++ii) {
                            if (32 * half + i0 + ii < len) G += PREP ? prep_neg_softplus(x[ii]) : x[ii];
                            x[ii] = G;
                        }
#pragma unroll
                        for (int ii = 0; ii < 16; ++ii) Gb[(i0 + ii) * D + tid] = x[ii];
                    }
                    if (half == 0) {
                        Gr[tid] = G;
                        Rf[tid] = expf(G);
                    }
                }
                __syncthreads();
                // all passes' q, k, v pieces are loaded before the first store; a thread's
                // channels c8 .. c8+7 are the same in every pass (128 is a multiple of D / 8)
                constexpr int kIt = 32 * (D / 8) / 128;
                uint4 qb_[kIt], kb_[kIt], vb_[kIt];
                float R8[8], E8[8];  // Gamma_r and e^{Gamma_r} of those channels
                {
                    const int c8 = (tid % (D / 8)) * 8;
                    const float4* rp = reinterpret_cast<const float4*>(&Gr[c8]);
                    const float4 r0 = rp[0], r1 = rp[1];
                    R8[0] = r0.x; R8[1] = r0.y; R8[2] = r0.z; R8[3] = r0.w;
                    R8[4] = r1.x; R8[5] = r1.y; R8[6] = r1.z; R8[7] = r1.w;
                    const float4* ep = reinterpret_cast<const float4*>(&Rf[c8]);
                    const float4 f0 = ep[0], f1 = ep[1];
                    E8[0] = f0.x; E8[1] = f0.y; E8[2] = f0.z; E8[3] = f0.w;
                    E8[4] = f1.x; E8[5] = f1.y; E8[6] = f1.z; E8[7] = f1.w;
                }
#pragma unroll
                for (int u = 0; u < kIt; ++u) {
                    const int w = tid + 128 * u;
                    const uint32_t off = sw128_offset(32 * half + w / (D / 8), (w % (D / 8)) * 8, 64);
                    qb_[u] = *reinterpret_cast<const uint4*>(Qs + off);
                    kb_[u] = *reinterpret_cast<const uint4*>(Ks + off);
                    vb_[u] = *reinterpret_cast<const uint4*>(Vs + off);
                }
#pragma unroll
                for (int u = 0; u < kIt; ++u) {
                    const int w = tid + 128 * u;
                    const int ii = w / (D / 8), c8 = (w % (D / 8)) * 8, i = 32 * half + ii;
                    const uint32_t off = sw128_offset(i, c8, 64);
                    float q8[8], k8[8], v8[8], G8[8];
                    unpack8(qb_[u], q8);
                    unpack8(kb_[u], k8);
                    unpack8(vb_[u], v8);
                    if (PREP) {
                        const float rq = RQ[i], rk = RK[i];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            q8[j] *= rq;
                            k8[j] *= rk;
                        }
                    }
                    const float b = beta_s[i];
                    const float4* gp = reinterpret_cast<const float4*>(&Gb[ii * D + c8]);
                    const float4 g0 = gp[0], g1 = gp[1];
                    G8[0] = g0.x; G8[1] = g0.y; G8[2] = g0.z; G8[3] = g0.w;
                    G8[4] = g1.x; G8[5] = g1.y; G8[6] = g1.z; G8[7] = g1.w;
                    uint32_t wq[4], wr[4], wb[4], wy[4], wv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float e[2], ei[2], ea[2];
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            e[t] = __expf(G8[2 * j + t] - R8[2 * j + t]);  // e^{Gamma - Gamma_r}
                            ei[t] = fast_rcp(e[t]);
                            ea[t] = e[t] * E8[2 * j + t];                   // e^{Gamma}
                        }
                        const float k0 = k8[2 * j], k1 = k8[2 * j + 1];
                        wq[j] = pack_bf16(q8[2 * j] * e[0], q8[2 * j + 1] * e[1]);
                        wr[j] = pack_bf16(k0 * ei[0], k1 * ei[1]);
                        wb[j] = pack_bf16(k0 * e[0], k1 * e[1]);
                        wy[j] = pack_bf16(b * k0 * ea[0], b * k1 * ea[1]);
                        wv[j] = pack_bf16(b * v8[2 * j], b * v8[2 * j + 1]);
                    }
                    *reinterpret_cast<uint4*>(Qs + off) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                    *reinterpret_cast<uint4*>(Ks + off) = make_uint4(wr[0], wr[1], wr[2], wr[3]);
                    *reinterpret_cast<uint4*>(Xs + off) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                    *reinterpret_cast<uint4*>(Ys + off) = make_uint4(wy[0], wy[1], wy[2], wy[3]);
                    *reinterpret_cast<uint4*>(Vs + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_async_smem();  // the staging buffer is refilled by the next copy
                __syncthreads();
            }
            if (!ok) break;
            if (tid < D) {
                L.gC[rec * D + tid] = expf(G);   // e^{Gamma_last} per channel
                GLs[tid] = expf(G - Gr[tid]);    // e^{Gamma_last - Gamma_r}
            }
            __syncthreads();
            uint8_t* kc_img = L.KC + rec * kTile;
            const int c8k = (tid % (D / 8)) * 8;  // the same channels in every pass
            const float4* lp = reinterpret_cast<const float4*>(&GLs[c8k]);
            const float4 l0 = lp[0], l1 = lp[1];
            const float L8[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
            for (int w = tid; w < 64 * (D / 8); w += 128) {
                const int i = w / (D / 8), c8 = (w % (D / 8)) * 8;
                const uint32_t off = sw128_offset(i, c8, 64);
                float kr8[8];
                unpack8(*reinterpret_cast<const uint4*>(Ks + off), kr8);
                uint32_t wc[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    wc[j] = pack_bf16(kr8[2 * j] * L8[2 * j], kr8[2 * j + 1] * L8[2 * j + 1]);
                *reinterpret_cast<uint4*>(kc_img + off) = make_uint4(wc[0], wc[1], wc[2], wc[3]);
            }
        }
        fence_async_smem();
        __syncthreads();

        // Gram = Kb Kr^T -> cols [0,64);  Qb Kr^T -> cols [64,128)
        if (tid == 0) {
            tc_fence_after();
            const Tile tX{smem_u32(Xs), 64}, tK{smem_u32(Ks), 64}, tQ{smem_u32(Qs), 64};
            mma_tiles(tm + 0, tX, false, tK, false, 64, 64, D, false);
            mma_tiles(tm + 64, tQ, false, tK, false, 64, 64, D, false);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();

        // A = diag(beta) strict_lower(Gram) (fp32) and the masked Aqk tile; each row's 64
        // columns are split over two threads (columns 32 h2 + 16 cb + j)
        {
            const float br = beta_s[r2];
            for (int cb = 0; cb < 2; ++cb) {
                float g16[16], a16[16];
                tmem_ld16_x2<32>(tl + cb * 16, g16);
                tmem_ld16_x2<32>(tl + 64 + cb * 16, a16);
                tmem_ld_wait();
                const int c0 = h2 * 32 + cb * 16;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = c0 + j;
                    Af[col * 64 + r2] = col < r2 ? br * g16[j] : 0.f;  // column-major A
                    a16[j] = col <= r2 ? a16[j] : 0.f;
                }
                tile_store16(Aqs, r2, c0, 64, a16);
            }
        }
        tc_fence_before();
        __syncthreads();

        // T = (I + A)^{-1} by 2 x 2 blocks of 32: T11 = (I + A11)^{-1} and T22 = (I + A22)^{-1}
        // side by side (thread n of each half solves column n, right-looking, so the
        // dependent chain is one FMA per row), then T21 = -T22 (A21 T11) on all threads.
        // fp32 throughout.
        {
            float* T11 = reinterpret_cast<float*>(sm + S::kInv);  // [32][32] row-major
            float* T22 = T11 + 1024;                     // [32][32] row-major
            float* Y = T22 + 1024;                       // [32][32] row-major, A21 T11
            // T goes to the operand tile only; its workspace image is one bulk copy of it
            auto put_t = [&](int i, int n, float x) {
                *reinterpret_cast<__nv_bfloat16*>(Ts + sw128_offset(i, n, 64)) =
                    __float2bfloat16_rn(x);
            };
            if (tid < 64) {
                const int o = tid & 32, n = tid & 31;
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = (i == n) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < 31; ++j) {
                    const float xj = x[j];
                    const float* col = Af + (o + j) * 64 + o;
#pragma unroll
                    for (int i4 = (j + 1) & ~3; i4 < 32; i4 += 4) {
                        const float4 a = *reinterpret_cast<const float4*>(col + i4);
                        if (i4 + 0 > j) x[i4 + 0] = fmaf(-a.x, xj, x[i4 + 0]);
                        if (i4 + 1 > j) x[i4 + 1] = fmaf(-a.y, xj, x[i4 + 1]);
                        if (i4 + 2 > j) x[i4 + 2] = fmaf(-a.z, xj, x[i4 + 2]);
                        if (i4 + 3 > j) x[i4 + 3] = fmaf(-a.w, xj, x[i4 + 3]);
                    }
                }
                float* Tb = o ? T22 : T11;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    Tb[i * 32 + n] = x[i];
                    put_t(o + i, o + n, x[i]);
                    put_t(i, 32 + n, 0.f);  // T12 = 0 (written twice, the same value)
                }
            }
            __syncthreads();
            // Y = A21 T11: thread (rows i0..i0+7, column n); A21[i][k] = Af[k * 64 + 32 + i]
            const int n = tid & 31, i0 = (tid >> 5) * 8;
            {
                float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int k = 0; k < 32; ++k) {
                    const float t = T11[k * 32 + n];
                    const float4 a0 = *reinterpret_cast<const float4*>(Af + k * 64 + 32 + i0);
                    const float4 a1 = *reinterpret_cast<const float4*>(Af + k * 64 + 36 + i0);
                    y[0] = fmaf(a0.x, t, y[0]);
                    y[1] = fmaf(a0.y, t, y[1]);
                    y[2] = fmaf(a0.z, t, y[2]);
                    y[3] = fmaf(a0.w, t, y[3]);
                    y[4] = fmaf(a1.x, t, y[4]);
                    y[5] = fmaf(a1.y, t, y[5]);
                    y[6] = fmaf(a1.z, t, y[6]);
                    y[7] = fmaf(a1.w, t, y[7]);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) Y[(i0 + q) * 32 + n] = y[q];
            }
            __syncthreads();
            // T21 = -T22 Y
            {
                float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int k = 0; k < 32; ++k) {
                    const float yk = Y[k * 32 + n];
#pragma unroll
                    for (int q = 0; q < 8; ++q) z[q] = fmaf(T22[(i0 + q) * 32 + k], yk, z[q]);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) put_t(32 + i0 + q, n, -z[q]);
            }
        }
        fence_async_smem();
        __syncthreads();

        // Wy = T (beta Kb) -> cols [0,D);  Ut = T (beta v) -> cols [128,128+D)
        if (tid == 0) {
            bulk_s2g(L.T + rec * 8192, Ts, 8192);
            bulk_commit();
            tc_fence_after();
            const Tile tT{smem_u32(Ts), 64}, tY{smem_u32(Ys), 64}, tV{smem_u32(Vs), 64};
            mma_tiles(tm + 0, tT, false, tY, true, 64, D, 64, false);
            mma_tiles(tm + 128, tT, false, tV, true, 64, D, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, 1, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();

        // Wy and Ut into their operand tiles (Ut where Kr was, which is consumed); the
        // workspace images ([64][D] SW128 tile images) are bulk copies of those tiles
        for (int cb = 0; cb < D / 32; ++cb) {
            float w16[16], u16[16];
            tmem_ld16_x2<D / 2>(tl + cb * 16, w16);
            tmem_ld16_x2<D / 2>(tl + 128 + cb * 16, u16);
            tmem_ld_wait();
            const int c0 = h2 * (D / 2) + cb * 16;
            tile_store16(Xs, r2, c0, 64, w16);
            tile_store16(Ks, r2, c0, 64, u16);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // Aqk Wy -> cols [0,D);  Ot / scale = Aqk Ut -> cols [128,128+D)
        if (tid == 0) {
            bulk_s2g(L.Wy + rec * kTile, Xs, kTile);
            bulk_s2g(L.Ut + rec * kTile, Ks, kTile);
            bulk_commit();
            tc_fence_after();
            const Tile tA{smem_u32(Aqs), 64}, tW{smem_u32(Xs), 64}, tU{smem_u32(Ks), 64};
            mma_tiles(tm + 0, tA, false, tW, true, 64, D, 64, false);
            mma_tiles(tm + 128, tA, false, tU, true, 64, D, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();

        // Qt in place over Qb' (each thread rewrites the elements it read), Ot in the
        // consumed v tile; their [64][D] SW128 workspace images are bulk copies of the tiles
        {
            const float sc = p.scale;
            for (int cb = 0; cb < D / 32; ++cb) {
                float w16[16], o16[16], qb[16];
                tmem_ld16_x2<D / 2>(tl + cb * 16, w16);
                tmem_ld16_x2<D / 2>(tl + 128 + cb * 16, o16);
                tmem_ld_wait();
                const int c0 = h2 * (D / 2) + cb * 16;
                tile_load16(Qs, r2, c0, 64, qb);  // Qb' = q e^{Gamma - Gamma_r}
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    qb[j] = sc * (qb[j] * Rf[c0 + j] - w16[j]);
                    o16[j] *= sc;
                }
                tile_store16(Qs, r2, c0, 64, qb);
                tile_store16(Vs, r2, c0, 64, o16);
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g(L.Qt + rec * kTile, Qs, kTile);
            bulk_s2g(L.Ot + rec * kTile, Vs, kTile);
            bulk_commit();
        }
    } while (0);

    if (!ok) {
        record_timeout(p);
        mbar_wait(&bar_ld, 0, kWaitLimitNs);  // let an outstanding copy land before exit
        if (ld_phase2) mbar_wait(&bar_ld, 1, kWaitLimitNs);
    }
    if (tid == 0) bulk_wait_all();  // the image copies are complete
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================== tc_scan_fwd
// Shared memory: the state operand, the U operand, and two stages of the per-chunk
// inputs so the next chunk's tiles load while this chunk computes.
template <int D, int BV>
struct ScanSmem {
    static constexpr int kTile = 64 * D * 2;
    // [BV][D] state W (bf16 operand); with 64-row value tiles two of them, the chunk's
    // and the next one's, so the state update need not wait for the state image copy
    static constexpr int kWBufs = BV == 64 ? 2 : 1, kWBytes = BV * D * 2;
    static constexpr int kW = 0;
    static constexpr int kUs = kWBufs * kWBytes;       // [64][BV] U operand
    static constexpr int kStage0 = kUs + BV * 128;
    // stage layout: [Wy; Qt] as one [128][D] tile (column block b holds the 64 Wy rows,
    // then the 64 Qt rows), KC [64][D]; Ut, Ot [64][BV] (columns v0 .. v0+BV-1 of their
    // [64][D] images); gC [D] fp32
    static constexpr int kWQ = 0, kKC = 2 * kTile, kUt = 3 * kTile, kOt = kUt + BV * 128,
                         kG = kOt + BV * 128;
    static constexpr int kStageBytes = (kG + D * 4 + 1023) / 1024 * 1024;
    static constexpr int kBytes = kStage0 + 2 * kStageBytes + 1024;
    static_assert(kBytes <= 232448 - 1024, "shared memory of one CTA");
    static constexpr uint32_t kStageTx = 3 * kTile + 2 * BV * 128 + D * 4;
};

// 256 threads, warp w on TMEM lane quarter w % 4 and half w / 4 of the columns.  Per
// chunk one product [Wy; Qt] W^T (M = 128) gives, in lanes 0..63, Wy S for the writes
// U = Ut - Wy S and, in lanes 64..127, Qt S for the outputs O = Ot + Qt S (token t of
// either in lane t, resp. 64 + t), so the threads of quarters 0-1 form U and those of
// quarters 2-3 form o at the same time, each 16 bytes at a time along a token row.
// Then U^T KC (M = BV value rows) gives the state increment; each thread updates half a
// state row (BV = 128: row 32 (w % 4) + lane; BV = 64: the M = 64 row layout).  A ninth
// warp issues the bulk copies (its lane 0: the state image, the next chunk's tiles, the
// o boxes), so no epilogue warp waits on their issue.
constexpr int kScanFwdThreads = 288;
constexpr int kScanMathThreads = 256;

template <int D, int BV>
__global__ void __launch_bounds__(kScanFwdThreads, 1)
    tc_scan_fwd_kernel(const __grid_constant__ CUtensorMap mo, const Params p, const TcLayout L,
                       int write_o, int stage_o) {
    using S = ScanSmem<D, BV>;
    constexpr int kTile = S::kTile;
    constexpr int DH = D / 2;   // key columns of a state thread
    constexpr int HC = BV / 2;  // value columns of an epilogue thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Ws = sm + S::kW;
    uint8_t* Us = sm + S::kUs;
    __shared__ uint64_t bar_ld[2], bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = tid < kScanMathThreads;   // the eight epilogue / state warps
    const int hf = (warp >> 2) & 1;             // which half of the columns
    const int erow = (warp & 3) * 32 + lane;    // row of the stacked product (M = 128)
    const int etok = erow & 63;                 // its token
    const bool u_row = erow < 64;               // lanes 0..63: Wy S; 64..127: Qt S
    const int unit = blockIdx.x, n = unit / p.H, h = unit % p.H;
    const int v0 = blockIdx.y * BV;
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);

    if (tid == 0) {
        mbar_init(&bar_ld[0], 1);
        mbar_init(&bar_ld[1], 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
        s_fail = 0;
        if (stage_o) prefetch_tmap(&mo);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = warp_lane_base(tm);
    // state row of U^T KC (or -1) and this thread's key columns: BV = 128 gives a thread
    // half a row; BV = 64 (an M = 64 accumulator, read with the two-half-warp shape) a
    // quarter of a row
    const int r = !math ? -1 : (BV == 128) ? (tid & 127) : m64_row_x2();
    constexpr int WC = BV == 128 ? DH : DH / 2;
    const int cbase = hf * DH + (BV == 128 ? 0 : m64_half_x2() * (DH / 2));

    const int v = v0 + (r < 0 ? 0 : r);
    const size_t state_off = ((size_t)n * p.H + h) * D * D;
    // Thread kIss (lane 0 of the copy warp) issues the copies: the chunk-start state image,
    // the next chunk's tiles and the o boxes.  Thread 0 issues the products and the U image.
    constexpr int kIss = kScanMathThreads;
    int issued[2] = {0, 0};  // bulk-load phases per stage (thread kIss)

    auto load_chunk = [&](int ci) {  // thread kIss: fetch chunk ci into stage ci & 1
        const int s = ci & 1;
        uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        mbar_arrive_expect_tx(&bar_ld[s], S::kStageTx);
        for (int kb = 0; kb < D / 64; ++kb) {
            bulk_g2s(st + S::kWQ + kb * 16384, L.Wy + rec * kTile + kb * 8192, 8192, &bar_ld[s]);
            bulk_g2s(st + S::kWQ + kb * 16384 + 8192, L.Qt + rec * kTile + kb * 8192, 8192, &bar_ld[s]);
        }
        bulk_g2s(st + S::kKC, L.KC + rec * kTile, kTile, &bar_ld[s]);
        bulk_g2s(st + S::kUt, L.Ut + rec * kTile + (size_t)v0 * 128, BV * 128, &bar_ld[s]);
        bulk_g2s(st + S::kOt, L.Ot + rec * kTile + (size_t)v0 * 128, BV * 128, &bar_ld[s]);
        bulk_g2s(st + S::kG, L.gC + rec * D, D * 4, &bar_ld[s]);
        ++issued[s];
        if (ci + 1 < nc) {  // the chunk after it into L2, one step ahead of its copy
            const size_t rn = rec + p.H;
            bulk_prefetch_l2(L.Wy + rn * kTile, kTile);
            bulk_prefetch_l2(L.Qt + rn * kTile, kTile);
            bulk_prefetch_l2(L.KC + rn * kTile, kTile);
            bulk_prefetch_l2(L.Ut + rn * kTile + (size_t)v0 * 128, BV * 128);
            bulk_prefetch_l2(L.Ot + rn * kTile + (size_t)v0 * 128, BV * 128);
        }
    };
    if (tid == kIss && nc > 0) load_chunk(0);

    float W[WC];  // W[v, cbase + c] = S[cbase + c, v], fp32
#pragma unroll
    for (int c = 0; c < WC; ++c) W[c] = (p.h0 && r >= 0) ? p.h0[state_off + (size_t)(cbase + c) * D + v] : 0.f;
    if (r >= 0) {
#pragma unroll
        for (int cb = 0; cb < WC / 16; ++cb) {
            float t[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) t[j] = W[cb * 16 + j];
            tile_store16(Ws, r, cbase + cb * 16, BV, t);
        }
    }
    fence_async_smem();
    __syncthreads();

    bool ok = true;
    for (int ci = 0; ci < nc && ok; ++ci) {
        const int s = ci & 1;
        uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        const int row0 = srow + ci * 64, len = min(64, slen - ci * 64);
        // o of a whole chunk is written in place over its Ot tile and leaves by tensor
        // stores; a ragged last chunk, and fp32 o, by 16-byte stores of token rows
        const bool tile_o = write_o && stage_o && len == 64;
        // this chunk's state operand, and the one its state update writes
        uint8_t* Wc = Ws + (S::kWBufs == 2 ? (ci & 1) * S::kWBytes : 0);
        uint8_t* Wn = Ws + (S::kWBufs == 2 ? ((ci + 1) & 1) * S::kWBytes : 0);
        if (tid == 0) bulk_wait_read();  // the previous chunk's U image has left Us
        ok = mbar_wait(&bar_ld[s], (ci >> 1) & 1, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;

        // [Wy; Qt] W^T -> cols [0, BV)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm, Tile{smem_u32(st + S::kWQ), 128}, false, Tile{smem_u32(Wc), BV}, false, 128, BV, D,
                      false);
            mma_commit(&bar_mma);
        }
        if (tid == kIss) {
            // the chunk-start state rows [v0, v0+BV) of the W-layout state image; then,
            // once the previous chunk's o tiles have left stage s^1 (and, with two state
            // tiles, the previous state image the other tile), the next chunk's tiles
            uint8_t* s_img = L.S + rec * (size_t)D * D * 2;
            for (int kb = 0; kb < D / 64; ++kb)
                bulk_s2g(s_img + (size_t)kb * D * 128 + (size_t)v0 * 128, Wc + kb * BV * 128, BV * 128);
            bulk_commit();
            bulk_wait_read_but_newest();
            if (ci + 1 < nc) load_chunk(ci + 1);
        }
        if (math && !mbar_wait(&bar_mma, 0, kWaitLimitNs)) s_fail = 1;
        tc_fence_after();
        // U = Ut - Wy S into the U operand (quarters 0-1); o = Ot + Qt S (quarters 2-3)
        if (math && (u_row || write_o)) {
            const uint8_t* src = st + (u_row ? S::kUt : S::kOt);
#pragma unroll 1
            for (int cb = 0; cb < HC / 16; cb += 2) {
                const int col = hf * HC + cb * 16;  // first of this pass's 32 value columns
                float a[16], b[16], x[16], y[16];
                tmem_ld16(tl + col, a);
                tmem_ld16(tl + col + 16, b);
                tmem_ld_wait();
                tile_load16(src, etok, col, 64, x);
                tile_load16(src, etok, col + 16, 64, y);
                if (u_row) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        x[j] -= a[j];
                        y[j] -= b[j];
                    }
                    tile_store16(Us, etok, col, 64, x);
                    tile_store16(Us, etok, col + 16, 64, y);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        x[j] += a[j];
                        y[j] += b[j];
                    }
                    if (tile_o) {  // in place: the Ot tile becomes the o box(es)
                        tile_store16(st + S::kOt, etok, col, 64, x);
                        tile_store16(st + S::kOt, etok, col + 16, 64, y);
                    } else if (etok < len) {
                        const size_t e0 = ((size_t)(row0 + etok) * p.H + h) * D + v0 + col;
                        if (p.out_dtype == DR_F32) {
                            float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.o) + e0);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                d[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                                d[4 + q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
                            }
                        } else {
                            uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + e0);
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                d[q] = make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                                                  pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
                                d[2 + q] = make_uint4(pack_bf16(y[8 * q], y[8 * q + 1]), pack_bf16(y[8 * q + 2], y[8 * q + 3]),
                                                      pack_bf16(y[8 * q + 4], y[8 * q + 5]), pack_bf16(y[8 * q + 6], y[8 * q + 7]));
                            }
                        }
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // U^T KC -> cols [128, 128+D); the U rows of the U image; the o boxes
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + 128, Tile{smem_u32(Us), 64}, true, Tile{smem_u32(st + S::kKC), 64}, true, BV, D, 64,
                      false);
            mma_commit(&bar_mma);
            bulk_s2g(L.U + rec * kTile + (size_t)v0 * 128, Us, BV * 128);
            bulk_commit();
        }
        if (tid == kIss) {
            if (tile_o) {
                for (int b = 0; b < BV / 64; ++b) tma_store_3d(&mo, st + S::kOt + b * 8192, v0 + 64 * b, h, row0);
                bulk_commit();
            }
            // one state tile: the state image has left it before the update rewrites it
            if (S::kWBufs == 1) {
                if (tile_o)
                    bulk_wait_read_but_newest();
                else
                    bulk_wait_read();
            }
        }
        if (math && !mbar_wait(&bar_mma, 1, kWaitLimitNs)) s_fail = 1;
        if (S::kWBufs == 1) __syncthreads();  // the state image has left Ws, rewritten below
        tc_fence_after();
        const float* gCs = reinterpret_cast<const float*>(st + S::kG) + cbase;
        if (math) {
#pragma unroll
            for (int cb = 0; cb < WC / 16; cb += 2) {  // two loads in flight per wait
                constexpr bool kPair = WC / 16 >= 2;
                float acc[16], acc2[16];
                if constexpr (BV == 128) {
                    tmem_ld16(tl + 128 + hf * DH + cb * 16, acc);
                    tmem_ld16(tl + 128 + hf * DH + (cb + 1) * 16, acc2);
                } else {  // the second half-warp reads DH / 2 columns further
                    tmem_ld16_x2<DH / 2>(tl + 128 + hf * DH + cb * 16, acc);
                    if (kPair) tmem_ld16_x2<DH / 2>(tl + 128 + hf * DH + (cb + 1) * 16, acc2);
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = cb * 16 + j;
                    W[c] = fmaf(W[c], gCs[c], acc[j]);
                    acc[j] = W[c];
                    if (kPair) {
                        W[c + 16] = fmaf(W[c + 16], gCs[c + 16], acc2[j]);
                        acc2[j] = W[c + 16];
                    }
                }
                if (r >= 0) {
                    tile_store16(Wn, r, cbase + cb * 16, BV, acc);
                    if (kPair) tile_store16(Wn, r, cbase + (cb + 1) * 16, BV, acc2);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(s_fail != 0)) {
            ok = false;
            break;
        }
    }

    if (ok) {
        if (p.hT && r >= 0) {
#pragma unroll
            for (int c = 0; c < WC; ++c) p.hT[state_off + (size_t)(cbase + c) * D + v] = W[c];
        }
    } else {
        record_timeout(p);
        if (tid == kIss)  // the latest copy issued into each stage has landed before exit
            for (int s = 0; s < 2; ++s)
                if (issued[s] > 0) mbar_wait(&bar_ld[s], (issued[s] - 1) & 1, kWaitLimitNs);
    }
    if (tid == 0 || tid == kIss) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}


}  // namespace

// [rows, H, D] bf16 tensor, box = 64 channels x 1 head x 64 rows, 128B swizzle
// The write u = U (token-major, out_dtype) from the U tile images the forward scan
// leaves in the workspace ([64 tokens][D] SW128 images): thread (token i, channels
// 8c .. 8c+7) moves one 16-byte piece of row i.
template <int D>
__global__ void __launch_bounds__(256) unpack_u_kernel(const Params p, const TcLayout L) {
    const int chunk = blockIdx.x, h = blockIdx.y;
    int seq, row0, len;
    chunk_info(p, chunk, seq, row0, len);
    const uint8_t* img = L.U + ((size_t)chunk * p.H + h) * (64 * D * 2);
    for (int w = threadIdx.x; w < 64 * (D / 8); w += blockDim.x) {
        const int i = w / (D / 8), c8 = (w % (D / 8)) * 8;
        if (i >= len) continue;
        const uint4 piece = *reinterpret_cast<const uint4*>(img + sw128_offset(i, c8, 64));
        const size_t e = ((size_t)(row0 + i) * p.H + h) * D + c8;
        if (p.out_dtype == DR_F32) {
            float x[8];
            unpack8(piece, x);
            float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.u) + e);
            d[0] = make_float4(x[0], x[1], x[2], x[3]);
            d[1] = make_float4(x[4], x[5], x[6], x[7]);
        } else {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.u) + e) = piece;
        }
    }
}

bool make_token_map(CUtensorMap* m, const void* ptr, int D, int H, long long rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output rows [rows][H][D] (bf16 or fp32) written by tensor stores: one box is the D values
// of 32 consecutive tokens of one head, dense (no swizzle) in shared memory
bool make_out_map(CUtensorMap* m, void* ptr, int D, int H, long long rows, bool f32) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int esz = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, 32};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr,
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 per-key-channel gates [rows][H][D]: one box is the D gates of box_rows tokens of
// one head, dense (no swizzle) in shared memory
bool make_gate_map(CUtensorMap* m, const void* ptr, int D, int H, long long rows, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_records(const Params& p) { return (size_t)p.num_chunks * p.H; }

TcLayout tc_layout(const Params& p) {
    return tc_layout_at(p.ws + 256, tc_records(p), p.dk, p.prepare != 0);
}

size_t tc_workspace_bytes(const Params& p) { return tc_layout_bytes(tc_records(p), p.dk, p.prepare != 0); }

template <int D, int VAR, bool PREP>
cudaError_t launch_prep(const Params& p, const TcLayout& L, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mg;
    const long long rows = (long long)p.B * p.T;
    if (!make_token_map(&mq, p.q, D, p.H, rows) || !make_token_map(&mk, p.k, D, p.H, rows) ||
        !make_token_map(&mv, p.v, D, p.H, rows))
        return cudaErrorInvalidValue;
    if (VAR == DR_KDA ? !make_gate_map(&mg, p.g, D, p.H, rows, 32) : !make_token_map(&mg, p.q, D, p.H, rows))
        return cudaErrorInvalidValue;
    constexpr int smem = PrepSmem<D>::kBytes;
    static std::atomic<unsigned long long> attr{0};
    {
        const cudaError_t e = set_smem_once(tc_prep_kernel<D, VAR, PREP>, smem, attr);
        if (e != cudaSuccess) return e;
    }
    if (p.num_chunks == 0) return cudaSuccess;
    TraceScope ts("tc_prep", st);
    tc_prep_kernel<D, VAR, PREP><<<dim3(p.num_chunks, p.H), 128, smem, st>>>(mq, mk, mv, mg, p, L);
    return cudaGetLastError();
}

template <int D, int BV>
cudaError_t launch_scan_fwd(const Params& p, const TcLayout& L, cudaStream_t st, bool write_o) {
    constexpr int smem = ScanSmem<D, BV>::kBytes;
    static std::atomic<unsigned long long> attr{0};
    {
        const cudaError_t e = set_smem_once(tc_scan_fwd_kernel<D, BV>, smem, attr);
        if (e != cudaSuccess) return e;
    }
    if (p.N * p.H == 0) return cudaSuccess;
    // bf16 o leaves whole chunks by tensor stores (a map over [rows, H, D], as the inputs)
    CUtensorMap mo;
    std::memset(&mo, 0, sizeof(mo));
    const bool stage_o = write_o && p.o && p.out_dtype == DR_BF16 &&
                         make_token_map(&mo, p.o, D, p.H, (long long)p.B * p.T);
    TraceScope ts("tc_scan_fwd", st);
    tc_scan_fwd_kernel<D, BV><<<dim3(p.N * p.H, D / BV), kScanFwdThreads, smem, st>>>(
        mo, p, L, write_o ? 1 : 0, stage_o ? 1 : 0);
    return cudaGetLastError();
}

template <int D>
cudaError_t tc_fwd_d(const Params& p, cudaStream_t st, bool write_o) {
    const TcLayout L = tc_layout(p);
    cudaError_t e;
    switch (p.variant * 2 + (p.prepare ? 1 : 0)) {
        case 2 * DR_DELTANET: e = launch_prep<D, DR_DELTANET, false>(p, L, st); break;
        case 2 * DR_DELTANET + 1: e = launch_prep<D, DR_DELTANET, true>(p, L, st); break;
        case 2 * DR_GDN: e = launch_prep<D, DR_GDN, false>(p, L, st); break;
        case 2 * DR_GDN + 1: e = launch_prep<D, DR_GDN, true>(p, L, st); break;
        case 2 * DR_KDA: e = launch_prep<D, DR_KDA, false>(p, L, st); break;
        default: e = launch_prep<D, DR_KDA, true>(p, L, st); break;
    }
    if (e != cudaSuccess) return e;
    // one 128-row value tile per (sequence, head) when that already fills the SMs; two
    // 64-row tiles otherwise (more CTAs for few, long sequences)
    if constexpr (D == 128) {
        if (p.N * p.H >= 120) e = launch_scan_fwd<D, 128>(p, L, st, write_o);
        else e = launch_scan_fwd<D, 64>(p, L, st, write_o);
    } else {
        e = launch_scan_fwd<D, 64>(p, L, st, write_o);
    }
    if (e != cudaSuccess || !p.u || p.num_chunks == 0) return e;
    TraceScope ts("unpack_u", st);
    unpack_u_kernel<D><<<dim3(p.num_chunks, p.H), 256, 0, st>>>(p, L);
    return cudaGetLastError();
}

cudaError_t tc_fwd(const Params& p, cudaStream_t st, bool write_o) {
    return p.dk == 128 ? tc_fwd_d<128>(p, st, write_o) : tc_fwd_d<64>(p, st, write_o);
}

}  // namespace dr
