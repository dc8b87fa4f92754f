// tc_bwd.cu -- bf16 tensor-core backward of the chunkwise delta rule (sm_103a).
//
// Chain rule through the chunk steps of tc_fwd.cu, per chunk with state S at
// its start and dS = dL/d(state at its end):
//   dU   = KC dS                         dS_prev = diag(e^{Gamma_last}) dS + Qt^T dO - Wy^T dU
//   dQt  = dO S^T,  dWyA = dU S^T,  dKC = U dS^T,  dgC = rowsum(dS * S)
//   dAqk = scale tril(dO Ut^T - dQt Wy^T) = scale tril(P T^T),
//          P = (dO v^T - dQt Kb^T) diag(beta)
//   dWy  = -dWyA - scale Aqk^T dQt,       dUt = dU + scale Aqk^T dO
//   dT   = (dWy Kb^T + dUt v^T) diag(beta)
//   d(beta Kb) = T^T dWy,  d(beta v) = T^T dUt
//   dA   = -T^T (dT T^T)  (strictly lower),  dG = diag(beta) dA
//   dKb  = dG Kr + beta d(beta Kb),  dKr = dG^T Kb + dAqk^T Qb,  dQb = scale dQt + dAqk Kr
// then the decay: dq = dQb e^{Gamma}, dk = dKb e^{Gamma} + dKr e^{-Gamma} + dKC e^{Gamma_last-Gamma},
// dGamma = dQb Qb + dKb Kb - dKr Kr - dKC KC (+ sum_i dKC KC + dgC e^{Gamma_last} at the
// last token), dg = reverse cumulative sum of dGamma within the chunk.
//
// Kernels: tc_scan_bwd (reverse over chunks, one CTA per (sequence, head, value
// tile), dS kept in fp32 registers) and tc_bwd_chunk (chunk-parallel: first the
// state-side products dO S^T, dU S^T, U dS^T and rowsum(dS * S), then the rest).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"
#include "tc_layout.cuh"
#include "trace.cuh"

namespace dr {
using namespace tc;

bool make_token_map(CUtensorMap* m, const void* ptr, int D, int H, long long rows);
TcLayout tc_layout(const Params& p);
cudaError_t tc_fwd(const Params& p, cudaStream_t st, bool write_o);

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}
__device__ __forceinline__ void record_timeout(const Params& p) {
    if (threadIdx.x == 0) atomicExch(p.err, kErrTimeout);
}
template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}
__device__ __forceinline__ void zero_pad_rows(uint8_t* tile, int D, int len) {
    const int pad = 64 - len;
    const int n = (D / 64) * pad * 8;
    for (int w = threadIdx.x; w < n; w += blockDim.x) {
        const int kb = w / (pad * 8), rr = len + (w % (pad * 8)) / 8, ch = w % 8;
        *reinterpret_cast<uint4*>(tile + kb * 8192 + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
    }
}

// ============================================================== tc_scan_bwd
template <int D, int BV>
struct BScanSmem {
    static constexpr int kTile = 64 * D * 2;
    static constexpr int kW = 0;                 // [BV][D]  dS^T slice (bf16 operand)
    static constexpr int kdU = BV * D * 2;       // [BV][64] -dU^T operand
    static constexpr int kStage0 = kdU + BV * 128;
    // stage layout: KC, Qt, Wy [64][D] tiles; dO [64 tokens][BV] tile; gC [D] fp32
    static constexpr int kKC = 0, kQt = kTile, kWy = 2 * kTile, kdO = 3 * kTile,
                         kG = kdO + BV * 128;
    static constexpr int kStageBytes = (kG + D * 4 + 1023) / 1024 * 1024;
    static constexpr int kBytes = kStage0 + 2 * kStageBytes + 1024;
    static constexpr uint32_t kStageTx = 3 * kTile + BV * 128 + D * 4;
};

template <int D, int BV>
__global__ void __launch_bounds__(128, 1)
    tc_scan_bwd_kernel(const __grid_constant__ CUtensorMap mdo, const Params p, const TcLayout L) {
    using S = BScanSmem<D, BV>;
    constexpr int kTile = S::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Ws = sm + S::kW;
    uint8_t* dUs = sm + S::kdU;
    __shared__ uint64_t bar_ld[2], bar_mma;
    __shared__ uint32_t tmem_base;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, n = unit / p.H, h = unit % p.H;
    const int v0 = blockIdx.y * BV;
    int c0, nc, srow, slen;
    seq_chunks(p, n, c0, nc, srow, slen);

    if (tid == 0) {
        mbar_init(&bar_ld[0], 1);
        mbar_init(&bar_ld[1], 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
        prefetch_tmap(&mdo);
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
    const int r = (BV == 128) ? tid : m64_row();
    const int v = v0 + (r < 0 ? 0 : r);
    const size_t state_off = ((size_t)n * p.H + h) * D * D;
    int issued[2] = {0, 0}, waited[2] = {0, 0};

    // iteration it handles chunk nc-1-it, in stage it & 1
    auto load_iter = [&](int it) {
        const int s = it & 1, ci = nc - 1 - it;
        uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        const int row0 = srow + ci * 64;
        mbar_arrive_expect_tx(&bar_ld[s], S::kStageTx);
        bulk_g2s(st + S::kKC, L.KC + rec * kTile, kTile, &bar_ld[s]);
        bulk_g2s(st + S::kQt, L.Qt + rec * kTile, kTile, &bar_ld[s]);
        bulk_g2s(st + S::kWy, L.Wy + rec * kTile, kTile, &bar_ld[s]);
        for (int kb = 0; kb < BV / 64; ++kb)
            tma_load_3d(st + S::kdO + kb * 8192, &mdo, &bar_ld[s], v0 + kb * 64, h, row0);
        bulk_g2s(st + S::kG, L.gC + rec * D, D * 4, &bar_ld[s]);
        ++issued[s];
    };
    if (tid == 0 && nc > 0) load_iter(0);

    float W[D];  // dS[:, v] (the gradient of the state at the current chunk end)
#pragma unroll
    for (int c = 0; c < D; ++c) W[c] = (p.dhT && r >= 0) ? p.dhT[state_off + (size_t)c * D + v] : 0.f;
    if (r >= 0) {
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb) {
            float t[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) t[j] = W[cb * 16 + j];
            tile_store16(Ws, r, cb * 16, BV, t);
        }
    }
    fence_async_smem();
    __syncthreads();

    bool ok = true;
    for (int it = 0; it < nc && ok; ++it) {
        const int s = it & 1, ci = nc - 1 - it;
        const uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        if (tid == 0) {
            if (it + 1 < nc) load_iter(it + 1);
            // rows [v0, v0+BV) of the W-layout image of dS at this chunk's end
            uint8_t* ds_img = L.dS + rec * (size_t)D * D * 2;
            for (int kb = 0; kb < D / 64; ++kb)
                bulk_s2g(ds_img + (size_t)kb * D * 128 + (size_t)v0 * 128, Ws + kb * BV * 128, BV * 128);
            bulk_commit();
        }
        ok = mbar_wait(&bar_ld[s], (it >> 1) & 1, kWaitLimitNs);
        if (tid == 0) ++waited[s];
        if (__syncthreads_or(!ok)) break;

        // dU^T = dS^T KC^T -> cols [0,64)
        if (tid == 0) {
            tc_fence_after();
            const Tile tW{smem_u32(Ws), BV}, tK{smem_u32(st + S::kKC), 64};
            mma_tiles(tm + 0, tW, false, tK, false, BV, 64, D, false);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        for (int g = 0; g < 4; ++g) {
            float acc[16];
            tmem_ld16(tl + g * 16, acc);
            tmem_ld_wait();
            if (r >= 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = -acc[j];
                tile_store16(dUs, r, g * 16, BV, acc);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // dO^T Qt - dU^T Wy -> cols [64, 64+D); -dU^T rows [v0, v0+BV) of its image
        if (tid == 0) {
            tc_fence_after();
            const Tile tO{smem_u32(st + S::kdO), 64}, tU{smem_u32(dUs), BV},
                tQ{smem_u32(st + S::kQt), 64}, tWy{smem_u32(st + S::kWy), 64};
            mma_tiles(tm + 64, tO, true, tQ, true, BV, D, 64, false);
            mma_tiles(tm + 64, tU, false, tWy, true, BV, D, 64, true);
            mma_commit(&bar_mma);
            bulk_s2g(L.dU + rec * kTile + (size_t)v0 * 128, dUs, BV * 128);
            bulk_commit();
        }
        ok = mbar_wait(&bar_mma, 1, kWaitLimitNs);
        if (tid == 0) bulk_wait_read();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        const float* gCs = reinterpret_cast<const float*>(st + S::kG);
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb) {
            float acc[16];
            tmem_ld16(tl + 64 + cb * 16, acc);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = cb * 16 + j;
                W[c] = fmaf(W[c], gCs[c], acc[j]);
                acc[j] = W[c];
            }
            if (r >= 0) tile_store16(Ws, r, cb * 16, BV, acc);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    if (ok) {
        if (p.dh0 && r >= 0) {
#pragma unroll
            for (int c = 0; c < D; ++c) p.dh0[state_off + (size_t)c * D + v] = W[c];
        }
    } else {
        record_timeout(p);
        if (tid == 0)
            for (int s = 0; s < 2; ++s)
                if (issued[s] > waited[s]) mbar_wait(&bar_ld[s], waited[s] & 1, kWaitLimitNs);
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================== tc_bwd_chunk
// 256 threads: warps w and w+4 read the same TMEM lane quarter (the same
// accumulator rows of an M = 64 product) and split its columns between them.
constexpr int kChunkThreads = 256;

template <int D, int VAR>
struct BChunkSmem {
    static constexpr int kTile = 64 * D * 2, kCC = 8192;
    static constexpr int kQ = 0, kK = kTile, kV = 2 * kTile, kdO = 3 * kTile, kdQ = 4 * kTile,
                         kKb = 5 * kTile, kdWy = 6 * kTile, kdUt = 7 * kTile;
    static constexpr int kT = 8 * kTile, kAq = kT + kCC, kB8a = kAq + kCC, kB8b = kB8a + kCC,
                         kdAq = kB8b + kCC;
    static constexpr int kGam = kdAq + kCC;                         // KDA: fp32 [64][D]
    static constexpr int kGS = D + 4;  // row stride of the per-channel fp32 arrays
    static constexpr int kSmall = kGam + (VAR == DR_KDA ? 64 * kGS * 4 : 0);
    // small arrays: beta[64], e^{Gamma_last}[D], dgC[D], rowsum[64], Gamma_row[64],
    // e^{Gamma_row}[64], e^{-Gamma_row}[64], per-row partials of the second warp half [3][64]
    static constexpr int kBytes = kSmall + (64 * 8 + D * 2) * 4 + 1024;
};

template <int D, int VAR>
__global__ void __launch_bounds__(kChunkThreads, 1)
    tc_bwd_chunk_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                        const Params p, const TcLayout L) {
    using S = BChunkSmem<D, VAR>;
    constexpr int kTile = S::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Qs = sm + S::kQ;     // q -> Qb
    uint8_t* Ks = sm + S::kK;     // k -> Kr
    uint8_t* Vs = sm + S::kV;     // v
    uint8_t* dOs = sm + S::kdO;   // dO, later dKC
    uint8_t* dQs = sm + S::kdQ;   // dQt = dO S^T
    uint8_t* Kbs = sm + S::kKb;   // Kb
    uint8_t* dWys = sm + S::kdWy; // dWyA -> dWy
    uint8_t* dUts = sm + S::kdUt; // -dU^T -> dUt^T  ([value][token])
    uint8_t* Ts = sm + S::kT;
    uint8_t* Aqs = sm + S::kAq;   // tril(Qb Kr^T)
    uint8_t* B8a = sm + S::kB8a;  // P, then X = dT T^T
    uint8_t* B8b = sm + S::kB8b;  // dT, then dG
    uint8_t* dAqs = sm + S::kdAq; // dAqk
    float* Gam = reinterpret_cast<float*>(sm + S::kGam);  // KDA: g, Gamma, e^Gamma, dGamma
    float* beta_s = reinterpret_cast<float*>(sm + S::kSmall);
    float* gC_s = beta_s + 64;
    float* dgC_s = gC_s + D;
    float* rowsum = dgC_s + D;
    float* Grow = rowsum + 64;    // GDN: Gamma per row, later sum of dKC*KC per row
    float* Erow = Grow + 64;      // GDN: e^{Gamma} per row
    float* Eirow = Erow + 64;     // GDN: e^{-Gamma} per row
    float* part = Eirow + 64;     // [3][64] partial row sums of warps 4..7
    __shared__ uint64_t bar_ld, bar_mma, bar_kc;
    __shared__ uint32_t tmem_base;

    constexpr uint32_t R_dbK = 128, R_dbV = 128 + D, R_dQ = 128 + 2 * D, R_dKr = 128 + D;
    const int tid = threadIdx.x, warp = tid >> 5, half = warp >> 2;
    const int chunk = blockIdx.x, h = blockIdx.y;
    int seq, row0, len;
    chunk_info(p, chunk, seq, row0, len);
    const size_t rec = (size_t)chunk * p.H + h;
    const float sc = p.scale;

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_kc, 1);
        fence_barrier_init();
        prefetch_tmap(&mq);
        prefetch_tmap(&mk);
        prefetch_tmap(&mv);
        prefetch_tmap(&mdo);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    const uint32_t tl = warp_lane_base(tm);
    const int r = m64_row();
    bool ok = true;
    uint32_t mph = 0;  // bar_mma phase
    auto mma_done = [&]() -> bool {
        const bool good = mbar_wait(&bar_mma, mph, kWaitLimitNs);
        mph ^= 1;
        return good;
    };

    do {
        // Phase A: what the state-side products need.  S sits in the Aqk / P / dG / dAqk
        // tiles, dS in the Kb / dWy tiles and U^T in the v tile, all idle until later.
        uint8_t* Sst = Aqs;   // [D][D] W-layout state at the chunk start
        uint8_t* dSst = Kbs;  // [D][D] W-layout state gradient at the chunk end
        uint8_t* Ust = Vs;    // [D][64] U^T
        constexpr uint32_t kDD = D * D * 2;
        if (tid == 0) {
            const uint32_t gbytes = VAR == DR_KDA ? (uint32_t)len * D * 4 : 0u;
            mbar_arrive_expect_tx(&bar_ld, 3 * kTile + 2 * kDD + 8192 + D * 4 + gbytes);
            bulk_g2s(dUts, L.dU + rec * kTile, kTile, &bar_ld);
            bulk_g2s(Ust, L.U + rec * kTile, kTile, &bar_ld);
            bulk_g2s(Sst, L.S + rec * kDD, kDD, &bar_ld);
            bulk_g2s(dSst, L.dS + rec * kDD, kDD, &bar_ld);
            for (int kb = 0; kb < D / 64; ++kb)
                tma_load_3d(dOs + kb * 8192, &mdo, &bar_ld, kb * 64, h, row0);
            bulk_g2s(Ts, L.T + rec * 8192, 8192, &bar_ld);
            bulk_g2s(gC_s, L.gC + rec * D, D * 4, &bar_ld);
        }
        __syncthreads();  // the expected byte count is registered before the gate rows go out
        if (VAR == DR_KDA && warp == 1) {
            for (int i = tid & 31; i < len; i += 32)
                bulk_g2s(Gam + i * S::kGS, p.g + ((size_t)(row0 + i) * p.H + h) * D, D * 4, &bar_ld);
        }
        if (tid < 64) beta_s[tid] = tid < len ? p.beta[(size_t)(row0 + tid) * p.H + h] : 0.f;
        ok = mbar_wait(&bar_ld, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        zero_pad_rows(dOs, D, len);
        fence_async_smem();
        __syncthreads();

        // M0: dO S^T -> [0,D) ; -dU S^T -> [D,2D) ; U dS^T -> [2D,3D)
        if (tid == 0) {
            tc_fence_after();
            const Tile tS{smem_u32(Sst), D}, tdS{smem_u32(dSst), D};
            mma_tiles(tm + 0, Tile{smem_u32(dOs), 64}, false, tS, true, 64, D, D, false);
            mma_tiles(tm + D, Tile{smem_u32(dUts), D}, true, tS, true, 64, D, D, false);
            mma_tiles(tm + 2 * D, Tile{smem_u32(Ust), D}, true, tdS, true, 64, D, D, false);
            mma_commit(&bar_mma);
        }
        // while M0 runs: dgC[c] = sum_v dS[c, v] S[c, v], and the cumulative log-decay
        // (KDA: per key channel, in place in Gam; GDN: per token, with its two
        // exponentials); rows past the end of the sequence add nothing
        for (int c = tid; c < D; c += kChunkThreads) {
            float acc = 0.f;
            for (int vv = 0; vv < D; ++vv)
                acc = fmaf(__bfloat162float(*tile_elem(Sst, vv, c, D)),
                           __bfloat162float(*tile_elem(dSst, vv, c, D)), acc);
            dgC_s[c] = acc;
        }
        if (VAR == DR_KDA) {
            // kChunkThreads / D threads per channel, each a contiguous block of rows, then
            // every block adds the totals of the blocks above it
            constexpr int P = kChunkThreads / D, R = 64 / P;
            const int c = tid % D, pt = tid / D;
            float* tot = reinterpret_cast<float*>(Qs);  // [P][D]; q arrives only after M0
            float G = 0.f;
#pragma unroll 8
            for (int i = pt * R; i < pt * R + R; ++i) {
                if (i < len) G += Gam[i * S::kGS + c];
                Gam[i * S::kGS + c] = G;
            }
            tot[pt * D + c] = G;
            __syncthreads();
            float off = 0.f;
            for (int q = 0; q < pt; ++q) off += tot[q * D + c];
            if (pt > 0)
                for (int i = pt * R; i < pt * R + R; ++i) Gam[i * S::kGS + c] += off;
        } else if (VAR == DR_GDN) {
            if (warp == 0) {
                const int lane = tid & 31;
                const float a0 = 2 * lane < len ? p.g[(size_t)(row0 + 2 * lane) * p.H + h] : 0.f;
                const float a1 = 2 * lane + 1 < len ? p.g[(size_t)(row0 + 2 * lane + 1) * p.H + h] : 0.f;
                float x = a0 + a1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                const float g0 = x - a1, g1 = x;
                Grow[2 * lane] = g0;
                Grow[2 * lane + 1] = g1;
                const float e0 = __expf(g0), e1 = __expf(g1);
                Erow[2 * lane] = e0;
                Erow[2 * lane + 1] = e1;
                Eirow[2 * lane] = fast_rcp(e0);
                Eirow[2 * lane + 1] = fast_rcp(e1);
            }
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        // Phase B: q, k, v (v replaces U^T, which M0 has consumed)
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_ld, 3 * kTile);
            for (int kb = 0; kb < D / 64; ++kb) {
                tma_load_3d(Qs + kb * 8192, &mq, &bar_ld, kb * 64, h, row0);
                tma_load_3d(Ks + kb * 8192, &mk, &bar_ld, kb * 64, h, row0);
                tma_load_3d(Vs + kb * 8192, &mv, &bar_ld, kb * 64, h, row0);
            }
        }
        // E0: dQt -> its tile, -dWyA -> the dWy tile (dS is consumed), dKC -> its
        // workspace image (reloaded for the last phase)
        for (int cb = half; cb < D / 16; cb += 2) {
            float a[16], b[16], c_[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld16(tl + D + cb * 16, b);
            tmem_ld16(tl + 2 * D + cb * 16, c_);
            tmem_ld_wait();
            if (r >= 0) {
                tile_store16(dQs, r, cb * 16, 64, a);
                tile_store16(dWys, r, cb * 16, 64, b);
                tile_store16(L.dKC + rec * kTile, r, cb * 16, 64, c_);
            }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // dKC image -> bulk reload
        ok = mbar_wait(&bar_ld, 1, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        zero_pad_rows(Qs, D, len);
        zero_pad_rows(Ks, D, len);
        zero_pad_rows(Vs, D, len);
        __syncthreads();
        // E1b: Qb = q e^G, Kr = k e^-G, Kb = k e^G, eight channels per step
        for (int w = tid; w < 64 * (D / 8); w += kChunkThreads) {
            const int i = w / (D / 8), c8 = (w % (D / 8)) * 8;
            const uint32_t off = sw128_offset(i, c8, 64);
            const uint4 qv = *reinterpret_cast<const uint4*>(Qs + off);
            const uint4 kv = *reinterpret_cast<const uint4*>(Ks + off);
            if (VAR == DR_DELTANET) {
                *reinterpret_cast<uint4*>(Kbs + off) = kv;
                continue;
            }
            float q8[8], k8[8], e8[8], i8[8];
            unpack8(qv, q8);
            unpack8(kv, k8);
            if (VAR == DR_KDA) {
                float4* gp = reinterpret_cast<float4*>(&Gam[i * S::kGS + c8]);
                const float4 g0 = gp[0], g1 = gp[1];
                const float G8[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    e8[j] = __expf(G8[j]);
                    i8[j] = fast_rcp(e8[j]);
                }
                gp[0] = make_float4(e8[0], e8[1], e8[2], e8[3]);  // e^Gamma from here on
                gp[1] = make_float4(e8[4], e8[5], e8[6], e8[7]);
            } else {
                const float e = Erow[i], ei = Eirow[i];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    e8[j] = e;
                    i8[j] = ei;
                }
            }
            uint32_t wq[4], wr[4], wb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wq[j] = pack_bf16(q8[2 * j] * e8[2 * j], q8[2 * j + 1] * e8[2 * j + 1]);
                wr[j] = pack_bf16(k8[2 * j] * i8[2 * j], k8[2 * j + 1] * i8[2 * j + 1]);
                wb[j] = pack_bf16(k8[2 * j] * e8[2 * j], k8[2 * j + 1] * e8[2 * j + 1]);
            }
            *reinterpret_cast<uint4*>(Qs + off) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
            *reinterpret_cast<uint4*>(Ks + off) = make_uint4(wr[0], wr[1], wr[2], wr[3]);
            *reinterpret_cast<uint4*>(Kbs + off) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        }
        fence_async_smem();
        __syncthreads();

        // M1: Qb Kr^T -> [0,64) ; dO v^T -> [64,128) ; dQt Kb^T -> [128,192)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + 0, Tile{smem_u32(Qs), 64}, false, Tile{smem_u32(Ks), 64}, false, 64, 64, D, false);
            mma_tiles(tm + 64, Tile{smem_u32(dOs), 64}, false, Tile{smem_u32(Vs), 64}, false, 64, 64, D, false);
            mma_tiles(tm + 128, Tile{smem_u32(dQs), 64}, false, Tile{smem_u32(Kbs), 64}, false, 64, 64, D, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        for (int cb = half; cb < 4; cb += 2) {
            float a[16], p1[16], p2[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld16(tl + 64 + cb * 16, p1);
            tmem_ld16(tl + 128 + cb * 16, p2);
            tmem_ld_wait();
            if (r >= 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = cb * 16 + j;
                    a[j] = col <= r ? a[j] : 0.f;
                    p1[j] = beta_s[col] * (p1[j] - p2[j]);
                }
                tile_store16(Aqs, r, cb * 16, 64, a);
                tile_store16(B8a, r, cb * 16, 64, p1);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M2: P T^T -> [0,64) ; Aqk^T dQt -> [64,64+D) ; dO^T Aqk -> [64+D, 128+D) (M = D)
        if (tid == 0) {
            tc_fence_after();
            const Tile tAq{smem_u32(Aqs), 64};
            mma_tiles(tm + 0, Tile{smem_u32(B8a), 64}, false, Tile{smem_u32(Ts), 64}, false, 64, 64, 64, false);
            mma_tiles(tm + 64, tAq, true, Tile{smem_u32(dQs), 64}, true, 64, D, 64, false);
            mma_tiles(tm + 64 + D, Tile{smem_u32(dOs), 64}, true, tAq, true, D, 64, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        if (tid == 0) {  // dO is consumed: bring dKC into its buffer for the last phase
            mbar_arrive_expect_tx(&bar_kc, kTile);
            bulk_g2s(dOs, L.dKC + rec * kTile, kTile, &bar_kc);
        }
        for (int cb = half; cb < 4; cb += 2) {
            float a[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld_wait();
            if (r >= 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) a[j] = (cb * 16 + j <= r) ? sc * a[j] : 0.f;
                tile_store16(dAqs, r, cb * 16, 64, a);
            }
        }
        for (int cb = half; cb < D / 16; cb += 2) {
            float a[16];
            tmem_ld16(tl + 64 + cb * 16, a);
            tmem_ld_wait();
            if (r >= 0) {
                float wa[16];
                tile_load16(dWys, r, cb * 16, 64, wa);
#pragma unroll
                for (int j = 0; j < 16; ++j) a[j] = wa[j] - sc * a[j];  // dWy (the tile held -dWyA)
                tile_store16(dWys, r, cb * 16, 64, a);
            }
        }
        {
            // dUts holds -dU^T ([value][token]); the accumulator rows are value channels
            const int rv = (D == 128) ? (tid & 127) : r;
            for (int g = half; g < 4; g += 2) {
                float b[16];
                tmem_ld16(tl + 64 + D + g * 16, b);
                tmem_ld_wait();
                if (rv >= 0) {
                    float nd[16];
                    tile_load16(dUts, rv, g * 16, D, nd);
#pragma unroll
                    for (int j = 0; j < 16; ++j) b[j] = sc * b[j] - nd[j];  // dUt^T
                    tile_store16(dUts, rv, g * 16, D, b);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M3: dWy Kb^T -> [0,64) ; dUt v^T -> [64,128) ; T^T dWy -> R_dbK ; T^T dUt -> R_dbV ;
        //     dAqk Kr -> R_dQ
        if (tid == 0) {
            tc_fence_after();
            const Tile tT{smem_u32(Ts), 64}, tdW{smem_u32(dWys), 64}, tdU{smem_u32(dUts), D};
            mma_tiles(tm + 0, tdW, false, Tile{smem_u32(Kbs), 64}, false, 64, 64, D, false);
            mma_tiles(tm + 64, tdU, true, Tile{smem_u32(Vs), 64}, false, 64, 64, D, false);
            mma_tiles(tm + R_dbK, tT, true, tdW, true, 64, D, 64, false);
            mma_tiles(tm + R_dbV, tT, true, tdU, false, 64, D, 64, false);
            mma_tiles(tm + R_dQ, Tile{smem_u32(dAqs), 64}, false, Tile{smem_u32(Ks), 64}, true, 64, D, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        float dbeta_acc = 0.f;
        for (int cb = half; cb < 4; cb += 2) {
            float a[16], b[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld16(tl + 64 + cb * 16, b);
            tmem_ld_wait();
            if (r >= 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) a[j] = beta_s[cb * 16 + j] * (a[j] + b[j]);  // dT
                tile_store16(B8b, r, cb * 16, 64, a);
            }
        }
        for (int cb = half; cb < D / 16; cb += 2) {
            float a[16];
            tmem_ld16(tl + R_dbV + cb * 16, a);
            tmem_ld_wait();
            if (r >= 0) {
                float vv[16];
                tile_load16(Vs, r, cb * 16, 64, vv);
                const float br = beta_s[r];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    dbeta_acc = fmaf(a[j], vv[j], dbeta_acc);
                    a[j] *= br;
                }
                if (r < len) store_row16(p.dv_, ((size_t)(row0 + r) * p.H + h) * D + cb * 16, p.grad_dtype, a);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M4: X = dT T^T -> [0,64)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + 0, Tile{smem_u32(B8b), 64}, false, Tile{smem_u32(Ts), 64}, false, 64, 64, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        for (int cb = half; cb < 4; cb += 2) {
            float a[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld_wait();
            if (r >= 0) tile_store16(B8a, r, cb * 16, 64, a);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M5: T^T X -> [0,64) (dA = -it) ; Gram Kb Kr^T -> [64,128)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + 0, Tile{smem_u32(Ts), 64}, true, Tile{smem_u32(B8a), 64}, true, 64, 64, 64, false);
            mma_tiles(tm + 64, Tile{smem_u32(Kbs), 64}, false, Tile{smem_u32(Ks), 64}, false, 64, 64, D, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        for (int cb = half; cb < 4; cb += 2) {
            float a[16], gm[16];
            tmem_ld16(tl + cb * 16, a);
            tmem_ld16(tl + 64 + cb * 16, gm);
            tmem_ld_wait();
            if (r >= 0) {
                const float br = beta_s[r];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float dA = (cb * 16 + j < r) ? -a[j] : 0.f;
                    dbeta_acc = fmaf(dA, gm[j], dbeta_acc);
                    a[j] = br * dA;  // dG
                }
                tile_store16(B8b, r, cb * 16, 64, a);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M6: dG Kr -> [0,D) ; dG^T Kb + dAqk^T Qb -> R_dKr
        if (tid == 0) {
            tc_fence_after();
            const Tile tG{smem_u32(B8b), 64};
            mma_tiles(tm + 0, tG, false, Tile{smem_u32(Ks), 64}, true, 64, D, 64, false);
            mma_tiles(tm + R_dKr, tG, true, Tile{smem_u32(Kbs), 64}, true, 64, D, 64, false);
            mma_tiles(tm + R_dKr, Tile{smem_u32(dAqs), 64}, true, Tile{smem_u32(Qs), 64}, true, 64, D, 64, true);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        ok = ok && mbar_wait(&bar_kc, 0, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();

        // E7: the decay chain, per row; each warp half takes every other 16-column block
        {
            // KDA: per-(row, channel) dKC * KC kept for a fixed-order sum over rows, in
            // the T / Aqk / P / dG / dAqk tiles (40 KB contiguous), all consumed by now;
            // rows padded to kGS floats so that lanes owning different rows hit different banks
            float* Fa = reinterpret_cast<float*>(Ts);
            float grow = 0.f, frow = 0.f;
            float er = 1.f, eir = 1.f;
            if (VAR == DR_GDN && r >= 0) {
                er = Erow[r];
                eir = Eirow[r];
            }
            const float br = r >= 0 ? beta_s[r] : 0.f;
            for (int cb = half; cb < D / 16; cb += 2) {
                float dq_[16], dbk[16], dkb[16], dkr[16];
                tmem_ld16(tl + R_dQ + cb * 16, dq_);
                tmem_ld16(tl + R_dbK + cb * 16, dbk);
                tmem_ld16(tl + 0 + cb * 16, dkb);
                tmem_ld16(tl + R_dKr + cb * 16, dkr);
                tmem_ld_wait();
                if (r >= 0) {
                    float qb[16], kb[16], kr[16], dqt[16], dkc[16];
                    tile_load16(Qs, r, cb * 16, 64, qb);
                    tile_load16(Kbs, r, cb * 16, 64, kb);
                    tile_load16(Ks, r, cb * 16, 64, kr);
                    tile_load16(dQs, r, cb * 16, 64, dqt);
                    tile_load16(dOs, r, cb * 16, 64, dkc);
                    float oq[16], ok_[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c = cb * 16 + j;
                        float e = er, ei = eir;
                        if (VAR == DR_KDA) {
                            e = Gam[r * S::kGS + c];  // e^Gamma, stored by the decay pass
                            ei = fast_rcp(e);
                        }
                        const float gc = gC_s[c];
                        const float dQb = sc * dqt[j] + dq_[j];
                        const float dKb = dkb[j] + br * dbk[j];
                        const float KC = kr[j] * gc;
                        dbeta_acc = fmaf(dbk[j], kb[j], dbeta_acc);
                        const float dG = dQb * qb[j] + dKb * kb[j] - dkr[j] * kr[j] - dkc[j] * KC;
                        if (VAR == DR_KDA) {
                            Gam[r * S::kGS + c] = dG;
                            Fa[r * S::kGS + c] = dkc[j] * KC;
                        } else if (VAR == DR_GDN) {
                            grow += dG;
                            frow = fmaf(dkc[j], KC, frow);
                        }
                        oq[j] = dQb * e;
                        ok_[j] = dKb * e + dkr[j] * ei + dkc[j] * gc * ei;
                    }
                    if (r < len) {
                        const size_t eidx = ((size_t)(row0 + r) * p.H + h) * D + cb * 16;
                        store_row16(p.dq, eidx, p.grad_dtype, oq);
                        store_row16(p.dk_, eidx, p.grad_dtype, ok_);
                    }
                }
            }
            // combine the two warp halves' row partials in a fixed order
            if (half == 1 && r >= 0) {
                part[r] = dbeta_acc;
                part[64 + r] = grow;
                part[128 + r] = frow;
            }
            __syncthreads();
            if (half == 0 && r >= 0) {
                dbeta_acc += part[r];
                if (VAR == DR_GDN) {
                    rowsum[r] = grow + part[64 + r];
                    Grow[r] = frow + part[128 + r];  // this row's Gamma is no longer needed
                }
                if (r < len) p.dbeta[(size_t)(row0 + r) * p.H + h] = dbeta_acc;
            }
        }
        __syncthreads();

        // E8: dg_i = (dgC e^{Gamma_last} + sum_rows dKC KC) + sum_{j >= i} dGamma_j
        if (VAR == DR_KDA) {
            // P threads per key channel, each owning 64 / P consecutive rows
            constexpr int P = kChunkThreads / D, R = 64 / P;
            const int c = tid % D, pt = tid / D, i0 = pt * R;
            const float* Fa = reinterpret_cast<const float*>(Ts);
            float* Sp = reinterpret_cast<float*>(Ts + 64 * S::kGS * 4);  // [P][D] row sums of dGamma
            float* Fp = Sp + P * D;                                 // [P][D] row sums of dKC KC
            float sg = 0.f, sf = 0.f;
            for (int i = i0; i < i0 + R; ++i) {
                sf += Fa[i * S::kGS + c];
                if (i < len) sg += Gam[i * S::kGS + c];
            }
            Sp[pt * D + c] = sg;
            Fp[pt * D + c] = sf;
            __syncthreads();
            float run = dgC_s[c] * gC_s[c];
            for (int q = 0; q < P; ++q) {
                run += Fp[q * D + c];
                if (q > pt) run += Sp[q * D + c];
            }
            for (int i = i0 + R - 1; i >= i0; --i) {
                if (i < len) {
                    run += Gam[i * S::kGS + c];
                    p.dg[((size_t)(row0 + i) * p.H + h) * D + c] = run;
                }
            }
        } else if (VAR == DR_GDN) {
            if (warp == 0) {
                const int lane = tid & 31;
                float e = Grow[lane] + Grow[lane + 32];  // per-row sums of dKC KC
                for (int c = lane; c < D; c += 32) e += dgC_s[c] * gC_s[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
                const float a0 = 2 * lane < len ? rowsum[2 * lane] : 0.f;
                const float a1 = 2 * lane + 1 < len ? rowsum[2 * lane + 1] : 0.f;
                float x = a0 + a1;  // suffix sum over lanes >= this one
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_down_sync(0xffffffffu, x, o);
                    if (lane + o < 32) x += y;
                }
                if (2 * lane < len) p.dg[(size_t)(row0 + 2 * lane) * p.H + h] = e + x;
                if (2 * lane + 1 < len) p.dg[(size_t)(row0 + 2 * lane + 1) * p.H + h] = e + x - a0;
            }
        }
    } while (0);
    if (!ok) {
        record_timeout(p);
        mbar_wait(&bar_ld, 0, kWaitLimitNs);
        mbar_wait(&bar_ld, 1, kWaitLimitNs);
        mbar_wait(&bar_kc, 0, kWaitLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int D>
cudaError_t tc_bwd_d(const Params& p, cudaStream_t st, bool reuse) {
    if (!reuse) {
        cudaError_t e = tc_fwd(p, st, false);
        if (e != cudaSuccess) return e;
    }
    const TcLayout L = tc_layout(p);
    const long long rows = (long long)p.B * p.T;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_token_map(&mq, p.q, D, p.H, rows) || !make_token_map(&mk, p.k, D, p.H, rows) ||
        !make_token_map(&mv, p.v, D, p.H, rows) || !make_token_map(&mdo, p.dO, D, p.H, rows))
        return cudaErrorInvalidValue;
    {
        auto launch_scan = [&](auto kernel, int bv, int smem, bool& attr) -> cudaError_t {
            if (!attr) {
                cudaError_t e = set_smem(kernel, smem);
                if (e != cudaSuccess) return e;
                attr = true;
            }
            TraceScope ts("tc_scan_bwd", st);
            kernel<<<dim3(p.N * p.H, D / bv), 128, smem, st>>>(mdo, p, L);
            return cudaGetLastError();
        };
        static bool s64 = false, s128 = false;
        cudaError_t e;
        if (D == 128 && p.N * p.H >= 120)
            e = launch_scan(tc_scan_bwd_kernel<D, (D == 128 ? 128 : 64)>, D == 128 ? 128 : 64,
                            BScanSmem<D, (D == 128 ? 128 : 64)>::kBytes, s128);
        else
            e = launch_scan(tc_scan_bwd_kernel<D, 64>, 64, BScanSmem<D, 64>::kBytes, s64);
        if (e != cudaSuccess) return e;
    }
    if (p.num_chunks == 0) return cudaSuccess;
    auto chunk_launch = [&](auto kernel, int smem, bool& attr) -> cudaError_t {
        if (!attr) {
            cudaError_t e = set_smem(kernel, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        {
            TraceScope ts("tc_bwd_chunk", st);
            kernel<<<dim3(p.num_chunks, p.H), kChunkThreads, smem, st>>>(mq, mk, mv, mdo, p, L);
        }
        return cudaGetLastError();
    };
    static bool a0 = false, a1 = false, a2 = false;
    switch (p.variant) {
        case DR_DELTANET:
            return chunk_launch(tc_bwd_chunk_kernel<D, DR_DELTANET>, BChunkSmem<D, DR_DELTANET>::kBytes, a0);
        case DR_GDN:
            return chunk_launch(tc_bwd_chunk_kernel<D, DR_GDN>, BChunkSmem<D, DR_GDN>::kBytes, a1);
        default:
            return chunk_launch(tc_bwd_chunk_kernel<D, DR_KDA>, BChunkSmem<D, DR_KDA>::kBytes, a2);
    }
}

}  // namespace

cudaError_t tc_bwd(const Params& p, cudaStream_t st, bool reuse) {
    return p.dk == 128 ? tc_bwd_d<128>(p, st, reuse) : tc_bwd_d<64>(p, st, reuse);
}

}  // namespace dr
