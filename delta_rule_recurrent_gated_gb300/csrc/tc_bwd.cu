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
// As in the forward, the Gram-type operands take their exponents relative to Gamma_r
// (the cumulative log-decay at the chunk's 32nd token): Qb' = q e^{Gamma - Gamma_r},
// Kb' = k e^{Gamma - Gamma_r}, Kr' = k e^{Gamma_r - Gamma}.  The products with the
// absolute Kb (dQt Kb^T, Kb dWy^T) use Kb' against dQt and dWy scaled by e^{Gamma_r} per
// key channel, so every formula above holds with e^{Gamma} replaced by e^{Gamma -
// Gamma_r}, e^{Gamma_last} by e^{Gamma_last - Gamma_r} (in dk and KC) and dQt, dWy, dbK by
// their scaled forms; L does not depend on Gamma_r, so dg needs no term for it.
//
// Kernels: tc_scan_bwd (reverse over chunks, one CTA per (sequence, head, value
// tile), dS kept in fp32 registers) and tc_bwd_chunk (chunk-parallel: first the
// state-side products dO S^T, dU S^T, U dS^T and rowsum(dS * S), then the rest).
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "tc.cuh"
#include "tc_layout.cuh"
#include "trace.cuh"

namespace dr {
using namespace tc;

bool make_token_map(CUtensorMap* m, const void* ptr, int D, int H, long long rows);
bool make_gate_map(CUtensorMap* m, const void* ptr, int D, int H, long long rows, int box_rows);
bool make_out_map(CUtensorMap* m, void* ptr, int D, int H, long long rows, bool f32);
TcLayout tc_layout(const Params& p);
cudaError_t tc_fwd(const Params& p, cudaStream_t st, bool write_o);

namespace {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}
__device__ __forceinline__ void record_timeout(const Params& p) {
    if (threadIdx.x == 0) atomicExch(p.err, kErrTimeout);
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
// 288 threads: warps 0-7 carry the chain (the thread of warp w holds state row r, lane
// quarter w % 4, and the half w / 4 of its key columns and of the -dU^T tokens); warp 8
// issues the loads and the dS image.
constexpr int kScanBwdThreads = 288;
constexpr int kScanBwdMathThreads = 256;

template <int D, int BV>
struct BScanSmem {
    static constexpr int kTile = 64 * D * 2;
    // [BV][D] dS^T slice (bf16 operand); with 64-row value tiles two of them, the chunk's
    // and the previous one's, so the update need not wait for the dS image copy
    static constexpr int kWBufs = BV == 64 ? 2 : 1, kWBytes = BV * D * 2;
    static constexpr int kW = 0;
    static constexpr int kdU = kWBufs * kWBytes;  // [BV][64] -dU^T operand
    static constexpr int kStage0 = kdU + BV * 128;
    // stage layout: KC, Qt, Wy [64][D] tiles; dO [64 tokens][BV] tile; gC [D] fp32;
    // rows [v0, v0+BV) of the -dU^T image of the emitted write's gradient (dr_bwd_u)
    static constexpr int kKC = 0, kQt = kTile, kWy = 2 * kTile, kdO = 3 * kTile,
                         kG = kdO + BV * 128, kdUx = kG + D * 4;
    static constexpr int kStageBytes = (kdUx + BV * 128 + 1023) / 1024 * 1024;
    static constexpr int kBytes = kStage0 + 2 * kStageBytes + 1024;
    static_assert(kBytes <= 232448 - 1024, "shared memory of one CTA");
    static constexpr uint32_t kStageTx = 3 * kTile + BV * 128 + D * 4;
};

template <int D, int BV>
__global__ void __launch_bounds__(kScanBwdThreads, 1)
    tc_scan_bwd_kernel(const __grid_constant__ CUtensorMap mdo, const Params p, const TcLayout L) {
    using S = BScanSmem<D, BV>;
    constexpr int kTile = S::kTile;
    constexpr int DH = D / 2;  // key columns of a state thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Ws = sm + S::kW;
    uint8_t* dUs = sm + S::kdU;
    __shared__ uint64_t bar_ld[2], bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5;
    const bool math = tid < kScanBwdMathThreads;  // the eight epilogue / state warps
    const int hf = (warp >> 2) & 1;               // which half of the columns
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
        s_fail = 0;
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
    // state row (or -1) and this thread's key columns: BV = 128 gives a thread half a row;
    // BV = 64 (M = 64 accumulators, read with the two-half-warp shape) a quarter of a row,
    // and 16 of the tokens of -dU^T
    const int r = !math ? -1 : (BV == 128) ? (tid & 127) : m64_row_x2();
    const int v = v0 + (r < 0 ? 0 : r);
    constexpr int WC = BV == 128 ? DH : DH / 2;
    const int h2 = m64_half_x2();
    const int cbase = hf * DH + (BV == 128 ? 0 : h2 * (DH / 2));
    const size_t state_off = ((size_t)n * p.H + h) * D * D;
    // Thread kIss (lane 0 of the copy warp) issues the loads and the dS image; thread 0
    // the products and the -dU^T image.
    constexpr int kIss = kScanBwdMathThreads;
    int issued[2] = {0, 0};  // bulk-load phases per stage (thread kIss)

    // iteration it handles chunk nc-1-it, in stage it & 1
    auto load_iter = [&](int it) {
        const int s = it & 1, ci = nc - 1 - it;
        uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        const int row0 = srow + ci * 64;
        mbar_arrive_expect_tx(&bar_ld[s], S::kStageTx + (p.dU ? BV * 128 : 0));
        if (p.dU) bulk_g2s(st + S::kdUx, L.dUx + rec * kTile + (size_t)v0 * 128, BV * 128, &bar_ld[s]);
        bulk_g2s(st + S::kKC, L.KC + rec * kTile, kTile, &bar_ld[s]);
        bulk_g2s(st + S::kQt, L.Qt + rec * kTile, kTile, &bar_ld[s]);
        bulk_g2s(st + S::kWy, L.Wy + rec * kTile, kTile, &bar_ld[s]);
        for (int kb = 0; kb < BV / 64; ++kb)
            tma_load_3d(st + S::kdO + kb * 8192, &mdo, &bar_ld[s], v0 + kb * 64, h, row0);
        bulk_g2s(st + S::kG, L.gC + rec * D, D * 4, &bar_ld[s]);
        ++issued[s];
    };
    if (tid == kIss && nc > 0) load_iter(0);

    float W[WC];  // dS[cbase + c, v] (the gradient of the state at the current chunk end)
#pragma unroll
    for (int c = 0; c < WC; ++c) W[c] = (p.dhT && r >= 0) ? p.dhT[state_off + (size_t)(cbase + c) * D + v] : 0.f;
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
    for (int it = 0; it < nc && ok; ++it) {
        const int s = it & 1, ci = nc - 1 - it;
        uint8_t* st = sm + S::kStage0 + s * S::kStageBytes;
        const size_t rec = (size_t)(c0 + ci) * p.H + h;
        // this chunk's dS operand, and the one its update writes
        uint8_t* Wc = Ws + (S::kWBufs == 2 ? (it & 1) * S::kWBytes : 0);
        uint8_t* Wn = Ws + (S::kWBufs == 2 ? ((it + 1) & 1) * S::kWBytes : 0);
        if (tid == kIss) {
            // the next chunk's tiles into stage s^1 (released at the end of the previous
            // iteration), then rows [v0, v0+BV) of the W-layout image of dS at this chunk's end
            if (it + 1 < nc) load_iter(it + 1);
            uint8_t* ds_img = L.dS + rec * (size_t)D * D * 2;
            for (int kb = 0; kb < D / 64; ++kb)
                bulk_s2g(ds_img + (size_t)kb * D * 128 + (size_t)v0 * 128, Wc + kb * BV * 128, BV * 128);
            bulk_commit();
            // two dS tiles: the previous dS image has left the one this chunk's update writes
            if (S::kWBufs == 2) bulk_wait_read_but_newest();
        }
        // no block barrier here: the previous iteration ended with one (its update is
        // complete), and the threads that read this chunk's stage wait for it themselves
        const uint32_t ldph = (it >> 1) & 1;
        // dU^T = dS^T KC^T -> cols [0,64); then dO^T Qt -> cols [64, 64+D), which does not
        // depend on the chain and runs during the -dU^T epilogue
        if (tid == 0) {
            if (mbar_wait(&bar_ld[s], ldph, kWaitLimitNs)) {
                tc_fence_after();
                mma_tiles(tm + 0, Tile{smem_u32(Wc), BV}, false, Tile{smem_u32(st + S::kKC), 64}, false, BV, 64,
                          D, false);
                mma_commit(&bar_mma);
                mma_tiles(tm + 64, Tile{smem_u32(st + S::kdO), 64}, true, Tile{smem_u32(st + S::kQt), 64}, true,
                          BV, D, 64, false);
            } else {
                s_fail = 1;
            }
        }
        if (math && (!mbar_wait(&bar_mma, 0, kWaitLimitNs) || !mbar_wait(&bar_ld[s], ldph, kWaitLimitNs)))
            s_fail = 1;
        tc_fence_after();
        if (math && BV == 64) {  // -dU^T for this thread's 16 tokens [32 hf + 16 h2, + 16)
            float acc[16];
            tmem_ld16_x2<16>(tl + hf * 32, acc);
            tmem_ld_wait();
            const int tb = hf * 32 + h2 * 16;
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = -acc[j];
            if (p.dU) {  // plus the packed -dU^T of the emitted write: row r, swizzled chunks
                const uint8_t* xrow = st + S::kdUx + r * 128;
                float x[16];
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    unpack8(*reinterpret_cast<const uint4*>(xrow + (((tb / 8 + q) ^ (r & 7)) << 4)), x + 8 * q);
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] += x[j];
            }
            tile_store16(dUs, r, tb, BV, acc);
        } else if (math) {  // -dU^T for this thread's 32 tokens [32 hf, 32 hf + 32)
            float acc[16], acc2[16];
            tmem_ld16(tl + hf * 32, acc);
            tmem_ld16(tl + hf * 32 + 16, acc2);
            tmem_ld_wait();
            if (r >= 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    acc[j] = -acc[j];
                    acc2[j] = -acc2[j];
                }
                if (p.dU) {  // plus the packed -dU^T of the emitted write: row r, swizzled chunks
                    const uint8_t* xrow = st + S::kdUx + r * 128;
                    float x[16];
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        unpack8(*reinterpret_cast<const uint4*>(xrow + (((4 * hf + q) ^ (r & 7)) << 4)), x + 8 * q);
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] += x[j];
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        unpack8(*reinterpret_cast<const uint4*>(xrow + (((4 * hf + 2 + q) ^ (r & 7)) << 4)), x + 8 * q);
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc2[j] += x[j];
                }
                tile_store16(dUs, r, hf * 32, BV, acc);
                tile_store16(dUs, r, hf * 32 + 16, BV, acc2);
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(s_fail != 0)) {
            ok = false;
            break;
        }

        // + (-dU^T) Wy -> cols [64, 64+D); -dU^T rows [v0, v0+BV) of its image
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + 64, Tile{smem_u32(dUs), BV}, false, Tile{smem_u32(st + S::kWy), 64}, true, BV, D, 64,
                      true);
            mma_commit(&bar_mma);
            bulk_s2g(L.dU + rec * kTile + (size_t)v0 * 128, dUs, BV * 128);
            bulk_commit();
        }
        if (S::kWBufs == 1 && tid == kIss) bulk_wait_read();  // the dS image has left Ws
        if (math && !mbar_wait(&bar_mma, 1, kWaitLimitNs)) s_fail = 1;
        if (S::kWBufs == 1) __syncthreads();
        tc_fence_after();
        const float* gCs = reinterpret_cast<const float*>(st + S::kG) + cbase;
        if (math) {
#pragma unroll
            for (int cb = 0; cb < WC / 16; cb += 2) {  // two loads in flight per wait
                constexpr bool kPair = WC / 16 >= 2;
                float acc[16], acc2[16];
                if constexpr (BV == 128) {
                    tmem_ld16(tl + 64 + hf * DH + cb * 16, acc);
                    tmem_ld16(tl + 64 + hf * DH + (cb + 1) * 16, acc2);
                } else {  // the second half-warp reads DH / 2 columns further
                    tmem_ld16_x2<DH / 2>(tl + 64 + hf * DH + cb * 16, acc);
                    if (kPair) tmem_ld16_x2<DH / 2>(tl + 64 + hf * DH + (cb + 1) * 16, acc2);
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
        if (tid == 0) bulk_wait_read();  // the -dU^T image has left dUs before the next epilogue
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(s_fail != 0)) {
            ok = false;
            break;
        }
    }

    if (ok) {
        if (p.dh0 && r >= 0) {
#pragma unroll
            for (int c = 0; c < WC; ++c) p.dh0[state_off + (size_t)(cbase + c) * D + v] = W[c];
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

// ============================================================== tc_bwd_chunk
// kChunkThreads threads = kChunkThreads / 128 warp groups of four warps (one warp per
// TMEM lane quarter).  Two accumulator shapes alternate:
//  * token-by-token products (M = 64): row i of the accumulator sits in lane
//    16*(i/16) + i%16 of warp quarter i/16; the warp groups split its columns;
//  * channel-by-token products (M = D, the transposes of every d-wide result):
//    channel c sits in lane c (D = 128) or in the M = 64 lane of row c (D = 64);
//    the warp groups split the 64 tokens.  Everything per element of
//    the d-wide results (dv, dq, dk, KDA's dGamma and its reverse cumulative sum)
//    then runs on full warps, with 32 consecutive channels of one token per
//    warp store, and the sums over channels are warp transpose-reductions.
constexpr int kChunkThreads = 512;

template <int D, int VAR>
struct BChunkSmem {
    static constexpr int kTile = 64 * D * 2, kCC = 8192;
    // Eight tile buffers P0..P7 of kTile bytes.  P1 holds k -> Kr, P2 v, P3 dO; the roles
    // of P0 and P4..P7 alternate between consecutive work items of a CTA (ChunkRoles), so
    // that the next item's inputs can be copied in while this item finishes.
    // [64][D] token-row tiles: q -> Qb, k -> Kr, v, dO, Kb
    // U [64][D] (token rows); [D][64] channel-row tiles: dQt^T, -dWyA^T -> dWy^T, -dU^T -> dUt^T
    static constexpr int kK = kTile, kV = 2 * kTile, kdO = 3 * kTile;
    // five 8 KB tiles: T, then Aqk / P-X / dT-dG / dAqk, which hold S before those
    static constexpr int kT = 8 * kTile, kAq = kT + kCC, kB8a = kAq + kCC, kB8b = kB8a + kCC,
                         kdAq = kB8b + kCC;
    static constexpr int kGam = kdAq + kCC;                         // KDA: fp32 [64][kGS]
    static constexpr int kGS = D;  // row stride of the per-channel fp32 array (a dense TMA box)
    static constexpr int kX = kGam + (VAR == DR_KDA ? 64 * kGS * 4 : 0);  // fp32 scratch, 8 KB
    static constexpr int kSmall = kX + 8192;
    // small arrays: beta[64], e^{Gamma_last}[2][D] (this item's and the next one's),
    // dgC[D], dGamma per row[64], e^{Gamma - Gamma_r} per row[64], e^{Gamma_r - Gamma} per
    // row[64], dbeta partials of the other warp groups [3][64], e^{Gamma_r}[D],
    // e^{Gamma_last - Gamma_r}[D], and with input preparation the inverse norms of the q and
    // k rows [2][64], GDN's sigmoid of the raw gate arguments [64]
    static constexpr int kBytes = kSmall + (64 * 10 + D * 5) * 4 + 1024;
};

// Sum over the 32 lanes of v[lane][k] for every k < N (N = 16 or 32): on return lane
// L holds the sum for k = L % N.  31 shuffles, fixed order.
template <int N>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= N; s >>= 1) {  // fold lanes that share k % N
#pragma unroll
        for (int k = 0; k < N; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], s);
    }
#pragma unroll
    for (int s = N / 2; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int k = 0; k < s; ++k) {
            const float send = up ? v[k] : v[k + s];
            const float keep = up ? v[k + s] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// A [64][D] output block staged in shared memory in the output's own element type,
// tokens [0,32) in one buffer and [32,64) in another (a token's D values contiguous);
// `sb` points at this thread's channel in the row of its first token.
template <int D, bool F32>
__device__ __forceinline__ void stage_put(uint8_t* sb, int k, float x) {
    if (F32)
        reinterpret_cast<float*>(sb)[k * D] = x;
    else
        reinterpret_cast<__nv_bfloat16*>(sb)[k * D] = __float2bfloat16_rn(x);
}
// The whole block, after the staging writes and a block barrier: 16-byte loads from
// the staging rows, 16-byte stores to the token rows (rows past `len` are not written).
template <int D, bool F32>
__device__ __forceinline__ void stage_copy_out(void* out, const uint8_t* lo, const uint8_t* hi,
                                               const Params& p, int row0, int len, int h) {
    constexpr int kRow = D * (F32 ? 4 : 2), kChunks = kRow / 16;
    for (int w = threadIdx.x; w < len * kChunks; w += kChunkThreads) {
        const int i = w / kChunks, c = w % kChunks;
        const uint8_t* src = (i < 32 ? lo + i * kRow : hi + (i - 32) * kRow) + c * 16;
        *reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + ((size_t)(row0 + i) * p.H + h) * kRow +
                                  c * 16) = *reinterpret_cast<const uint4*>(src);
    }
}

// The same copy-out for the gradient of a normalised input (DR_FLAG_PREPARE_INPUTS): the
// staged rows hold dL/dx_hat of x_hat = x r, r = rsqrt(sum x^2 + eps) = rinv[row]; each row
// is chained to dL/dx = r (dx_hat - x_hat (x_hat . dx_hat)).  x_hat comes from
//   SRC 0: the raw bf16 rows x in global memory (read once, before the first store);
//   SRC 1: the decayed operand tile (x_hat e^{+-(Gamma - Gamma_r)}, bf16) times a per-row
//          factor rowf[row] that undoes the decay (GDN; DeltaNet with rowf = null);
//   SRC 2: the decayed tile divided by the per-element factor gam[row][channel] (KDA).
// The kChunks threads of a row are consecutive lanes of one warp and sum the dot product
// by shuffles, so every thread runs every pass (rows past `len` are not written).
template <int D, bool F32, int SRC>
__device__ __forceinline__ void stage_copy_out_prep(void* out, const uint8_t* lo, const uint8_t* hi,
                                                    const Params& p, int row0, int len, int h,
                                                    const __nv_bfloat16* __restrict__ raw,
                                                    const float* rinv, const uint8_t* tile,
                                                    const float* rowf, const float* gam) {
    constexpr int kRow = D * (F32 ? 4 : 2), kChunks = kRow / 16, E = F32 ? 4 : 8;
    constexpr int kPass = 64 * kChunks / kChunkThreads;
    static_assert(kPass * kChunkThreads == 64 * kChunks && kChunks <= 32, "whole warps per pass");
    // every row piece is loaded before the first store (they may not be reordered past it)
    float x[kPass][E];
#pragma unroll
    for (int ps = 0; ps < kPass; ++ps) {
        const int w = threadIdx.x + ps * kChunkThreads, i = w / kChunks, c = w % kChunks;
        if (SRC == 0) {
            const size_t e0 = ((size_t)(row0 + i) * p.H + h) * D + c * E;
            if (i >= len) {
#pragma unroll
                for (int j = 0; j < E; ++j) x[ps][j] = 0.f;
            } else if constexpr (F32) {
                const uint2 u = *reinterpret_cast<const uint2*>(raw + e0);
                const uint32_t wv[2] = {u.x, u.y};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
                    x[ps][2 * j] = __low2float(b);
                    x[ps][2 * j + 1] = __high2float(b);
                }
            } else {
                unpack8(*reinterpret_cast<const uint4*>(raw + e0), x[ps]);
            }
        } else {
            const int cb = c * E;  // first channel of the piece
            const uint8_t* src = tile + sw128_offset(i, cb & ~7, 64) + (cb & 7) * 2;
            if constexpr (F32) {
                const uint2 u = *reinterpret_cast<const uint2*>(src);
                const uint32_t wv[2] = {u.x, u.y};
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&wv[j]);
                    x[ps][2 * j] = __low2float(b);
                    x[ps][2 * j + 1] = __high2float(b);
                }
            } else {
                unpack8(*reinterpret_cast<const uint4*>(src), x[ps]);
            }
            if (SRC == 1 && rowf) {
                const float f = rowf[i];
#pragma unroll
                for (int j = 0; j < E; ++j) x[ps][j] *= f;
            } else if (SRC == 2) {
#pragma unroll
                for (int j = 0; j < E; ++j) x[ps][j] *= fast_rcp(gam[i * D + cb + j]);
            }
        }
    }
    float d[kPass][E], xd[kPass];
#pragma unroll
    for (int ps = 0; ps < kPass; ++ps) {
        const int w = threadIdx.x + ps * kChunkThreads, i = w / kChunks, c = w % kChunks;
        const uint8_t* src = (i < 32 ? lo + i * kRow : hi + (i - 32) * kRow) + c * 16;
        if constexpr (F32) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            d[ps][0] = v.x; d[ps][1] = v.y; d[ps][2] = v.z; d[ps][3] = v.w;
        } else {
            unpack8(*reinterpret_cast<const uint4*>(src), d[ps]);
        }
        xd[ps] = 0.f;
#pragma unroll
        for (int j = 0; j < E; ++j) xd[ps] = fmaf(x[ps][j], d[ps][j], xd[ps]);
    }
#pragma unroll
    for (int ps = 0; ps < kPass; ++ps) xd[ps] = lane_group_sum<kChunks>(xd[ps]);
#pragma unroll
    for (int ps = 0; ps < kPass; ++ps) {
        const int w = threadIdx.x + ps * kChunkThreads, i = w / kChunks, c = w % kChunks;
        const size_t e0 = ((size_t)(row0 + i) * p.H + h) * D + c * E;
        const float r = rinv[i];
        // x_hat . dx_hat, and the factor of x in the chain (x_hat itself for SRC > 0)
        const float f = SRC == 0 ? r * r * xd[ps] : xd[ps];
#pragma unroll
        for (int j = 0; j < E; ++j) d[ps][j] = r * (d[ps][j] - x[ps][j] * f);
        if (i < len) {
            uint8_t* dst = static_cast<uint8_t*>(out) + e0 * (F32 ? 4 : 2);
            if constexpr (F32) {
                *reinterpret_cast<float4*>(dst) = make_float4(d[ps][0], d[ps][1], d[ps][2], d[ps][3]);
            } else {
                *reinterpret_cast<uint4*>(dst) =
                    make_uint4(pack_bf16(d[ps][0], d[ps][1]), pack_bf16(d[ps][2], d[ps][3]),
                               pack_bf16(d[ps][4], d[ps][5]), pack_bf16(d[ps][6], d[ps][7]));
            }
        }
    }
}

// Buffer roles of one work item.  Even items: q in P0, U in P4 (then dQt^T), dS in
// P5..P6 (then Kb in P5, dWy^T in P6), -dU^T in P7.  Odd items: q in P5, U in P0 (then
// Kb), dS in P6..P7 (then dQt^T in P6, dWy^T in P7), -dU^T in P4.  What an even item
// still reads after its last product (Kb, Kr) and where it stages dk (P2, P3) is
// disjoint from where the next odd item's state goes, and the reverse.
struct ChunkRoles {
    uint8_t *Q, *U, *dQ, *dS, *Kb, *dWy, *dUt;
};
__device__ __forceinline__ ChunkRoles chunk_roles(uint8_t* sm, int kTile, bool odd) {
    auto P = [&](int i) { return sm + i * kTile; };
    if (odd) return ChunkRoles{P(5), P(0), P(6), P(6), P(0), P(7), P(4)};
    return ChunkRoles{P(0), P(4), P(4), P(5), P(5), P(6), P(7)};
}

template <int D, int VAR, bool PREP, bool F32OUT>
__global__ void __launch_bounds__(kChunkThreads, 1)
    tc_bwd_chunk_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                        const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mgq,
                        const __grid_constant__ CUtensorMap mgk, const __grid_constant__ CUtensorMap mgv,
                        const Params p, const TcLayout L) {
    using S = BChunkSmem<D, VAR>;
    constexpr int kTile = S::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* Ks = sm + S::kK;     // k -> Kr
    uint8_t* Vs = sm + S::kV;     // v, then dv and dk staging
    uint8_t* dOs = sm + S::kdO;   // dO, then dv and dk staging
    uint8_t* Ts = sm + S::kT;
    uint8_t* Aqs = sm + S::kAq;   // tril(Qb Kr^T)
    uint8_t* B8a = sm + S::kB8a;  // P, then X = dT T^T
    uint8_t* B8b = sm + S::kB8b;  // dT^T, then dG
    uint8_t* dAqs = sm + S::kdAq; // dAqk
    float* Gam = reinterpret_cast<float*>(sm + S::kGam);  // KDA: g -> Gamma -> e^Gamma
    float* Xs = reinterpret_cast<float*>(sm + S::kX);
    float* beta_s = reinterpret_cast<float*>(sm + S::kSmall);
    float* gC_b = beta_s + 64;    // [2][D]
    float* dgC_s = gC_b + 2 * D;
    float* rowsum = dgC_s + D;    // GDN: dGamma per row
    float* Erow = rowsum + 64;    // GDN: e^{Gamma - Gamma_r} per row
    float* Eirow = Erow + 64;     // GDN: e^{Gamma_r - Gamma} per row
    float* part = Eirow + 64;     // [3][64] dbeta partials of warp groups 1..
    float* eref = part + 3 * 64;  // [D] e^{Gamma_r} per key channel
    float* gcr = eref + D;        // [D] e^{Gamma_last - Gamma_r} per key channel
    float* rq_s = gcr + D;        // [64] rsqrt(sum q^2 + eps) per token (input preparation)
    float* rk_s = rq_s + 64;      // [64] the same for k
    float* sgx = rk_s + 64;       // GDN, input preparation: sigmoid(x) per token
    __shared__ uint64_t bar_st, bar_tok, bar_mma;
    __shared__ uint32_t tmem_base;

    // TMEM columns, 64 each.  C0 / C1 / C2 are reused phase by phase; the others hold
    // one result from its product to its last reader.
    constexpr uint32_t C0 = 0, C1 = 64, C2 = 128, C3 = 192, C4 = 256, C_dQ = 320, C6 = 384,
                       C_dKC = 448;
    constexpr int kG = kChunkThreads / 128, kTok = 64 / kG;  // warp groups, tokens per group
    constexpr int kIssuer = kChunkThreads - 32;  // lane 0 of the last warp: the next item's copies
    const int tid = threadIdx.x, warp = tid >> 5, grp = warp >> 2, lane = tid & 31;
    const int nitems = p.num_chunks * p.H;  // work item = (chunk, head), item = chunk * H + h
    const float sc = p.scale;
    constexpr bool f32out = F32OUT;  // fp32 gradients (else bf16): one compact loop per type

    if (tid == 0) {
        mbar_init(&bar_st, 1);
        mbar_init(&bar_tok, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
        prefetch_tmap(&mq);
        prefetch_tmap(&mk);
        prefetch_tmap(&mv);
        prefetch_tmap(&mdo);
        if (VAR == DR_KDA) prefetch_tmap(&mg);
        prefetch_tmap(&mgv);
        if (!PREP) {
            prefetch_tmap(&mgq);
            prefetch_tmap(&mgk);
        }
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
    // row of an M = 64 accumulator read with tmem_ld8_x2, and which 8 of a 16-column block
    const int r2 = m64_row_x2(), h2 = m64_half_x2();
    const int cl = D == 128 ? (tid & 127) : m64_row();  // channel of an M = D accumulator, or -1
    const int t0 = kTok * grp;                          // first token of this thread's group
    // Element (t0 + k, cl) of a [64][D] SW128 token tile sits at xo[k % 8] + 128 k: the
    // swizzle depends on the row only through k % 8 because t0 is a multiple of 16.
    uint32_t xo[8];
    {
        const int c = cl < 0 ? 0 : cl;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            xo[k] = (uint32_t)((c >> 6) * 8192 + t0 * 128 + ((((c >> 3) & 7) ^ k) << 4) + (c & 7) * 2);
    }
    auto tok = [&](const uint8_t* tile, int k) -> float {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + xo[k & 7] + k * 128));
    };
    bool ok = true;
    uint32_t mph = 0;  // bar_mma phase
    auto mma_done = [&]() -> bool {
        const bool good = mbar_wait(&bar_mma, mph, kWaitLimitNs);
        mph ^= 1;
        return good;
    };
    // e^{Gamma} and e^{-Gamma} of token t0 + k for this thread's channel
    const float* gam_t = Gam + t0 * S::kGS + (cl < 0 ? 0 : cl);
    // 16 (8) consecutive per-token values starting at token t0 + k0 (k0 multiple of 4)
    auto load16 = [&](const float* src, int k0, float (&v)[16]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 x = *reinterpret_cast<const float4*>(src + t0 + k0 + 4 * q);
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
        }
    };
    auto load8 = [&](const float* src, int k0, float (&v)[8]) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 x = *reinterpret_cast<const float4*>(src + t0 + k0 + 4 * q);
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
        }
    };
    // e^{Gamma} and e^{-Gamma} of tokens t0 + 8 b .. + 7 for this thread's channel
    auto decay8 = [&](int b, float (&e)[8], float (&ei)[8], bool from_tmem) {
        if (VAR == DR_KDA) {
            if (from_tmem) {
                tmem_ld8(tl + C3 + t0 + 8 * b, e);  // copied there by the dq stage
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = gam_t[(8 * b + j) * S::kGS];  // from the decay pass
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) ei[j] = fast_rcp(e[j]);
        } else if (VAR == DR_GDN) {
            load8(Erow, 8 * b, e);
            load8(Eirow, 8 * b, ei);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = ei[j] = 1.f;
        }
    };
    // staging address of (token t0, this thread's channel): tokens [0,32) in lo, [32,64) in hi
    auto stage_base = [&](uint8_t* lo, uint8_t* hi, bool f32) -> uint8_t* {
        const int esz = f32 ? 4 : 2;
        return (t0 >= 32 ? hi : lo) + (t0 & 31) * D * esz + (cl < 0 ? 0 : cl) * esz;
    };
    // a whole chunk's staged rows leave as two tensor stores of 32 tokens (thread kIssuer,
    // after the staging barrier); the copy warp waits for them to read the staging tiles
    // before anything refills those
    auto tensor_out = [&](const CUtensorMap* map, const uint8_t* lo, const uint8_t* hi, int hh, int r0) {
        tma_store_3d(map, lo, 0, hh, r0);
        tma_store_3d(map, hi, 0, hh, r0 + 32);
        bulk_commit();
    };
    // dGamma of this thread's channel and tokens (KDA), or its share of each token's
    // dGamma (GDN), is accumulated in TMEM columns C1 + t0 .. + kTok - 1 from E4 on
    float fsum = 0.f;  // sum over this thread's tokens of dKC * KC

    constexpr uint32_t kDD = D * D * 2;
    uint8_t* Sst = Aqs;  // [D][D] W-layout state at the chunk start, in the four 8 KB tiles
    // State-side copies of an item: S, dS, U, -dU^T, T, e^{Gamma_last} (and KDA's
    // gates, one [64][D] fp32 box) on bar_st; token side q, k, v, dO on bar_tok.
    auto issue_state = [&](int itm, bool odd) {
        const int c = itm / p.H, hh = itm % p.H;
        int sq, r0, ln;
        chunk_info(p, c, sq, r0, ln);
        const size_t rc = (size_t)c * p.H + hh;
        const ChunkRoles R = chunk_roles(sm, kTile, odd);
        mbar_arrive_expect_tx(&bar_st, 2 * kTile + 2 * kDD + 8192 + D * 4 + (VAR == DR_KDA ? 64 * D * 4 : 0));
        bulk_g2s(Sst, L.S + rc * kDD, kDD, &bar_st);
        bulk_g2s(R.dS, L.dS + rc * kDD, kDD, &bar_st);
        bulk_g2s(R.U, L.U + rc * kTile, kTile, &bar_st);
        bulk_g2s(R.dUt, L.dU + rc * kTile, kTile, &bar_st);
        bulk_g2s(Ts, L.T + rc * 8192, 8192, &bar_st);
        bulk_g2s(gC_b + (odd ? D : 0), L.gC + rc * D, D * 4, &bar_st);
        if (VAR == DR_KDA) tma_load_3d(Gam, &mg, &bar_st, 0, hh, r0);
    };
    auto issue_tok = [&](int itm, bool odd) {
        const int c = itm / p.H, hh = itm % p.H;
        int sq, r0, ln;
        chunk_info(p, c, sq, r0, ln);
        const ChunkRoles R = chunk_roles(sm, kTile, odd);
        mbar_arrive_expect_tx(&bar_tok, 4 * kTile + (PREP ? 512 : 0));
        if (PREP) bulk_g2s(rq_s, L.RN + ((size_t)c * p.H + hh) * 128, 512, &bar_tok);  // row norms
        for (int kb = 0; kb < D / 64; ++kb) {
            tma_load_3d(R.Q + kb * 8192, &mq, &bar_tok, kb * 64, hh, r0);
            tma_load_3d(Ks + kb * 8192, &mk, &bar_tok, kb * 64, hh, r0);
            tma_load_3d(Vs + kb * 8192, &mv, &bar_tok, kb * 64, hh, r0);
            tma_load_3d(dOs + kb * 8192, &mdo, &bar_tok, kb * 64, hh, r0);
        }
    };
    // per-token scalars of an item, read into registers ahead of time: beta (threads
    // 64..127) and GDN's log-decays (two per lane of warp 1).  With input preparation the
    // loads are raw and map_scalars applies the maps (beta = sigmoid(b), g = -softplus(x),
    // and sigmoid(x) for the chain of dg) at the end of the previous item, where these
    // warps wait for warp 0's dg scan, so neither the loads nor the maps delay an item.
    float beta_ld = 0.f, gl0 = 0.f, gl1 = 0.f, sg0 = 0.f, sg1 = 0.f;
    int scal_len = 0;  // the length of the item whose scalars are held
    auto load_scalars = [&](int itm) {
        const int c = itm / p.H, hh = itm % p.H;
        int sq, r0, ln;
        chunk_info(p, c, sq, r0, ln);
        scal_len = ln;
        beta_ld = (tid >= 64 && tid < 128 && tid - 64 < ln) ? p.beta[(size_t)(r0 + tid - 64) * p.H + hh] : 0.f;
        if (VAR == DR_GDN && warp == 1) {
            gl0 = 2 * lane < ln ? p.g[(size_t)(r0 + 2 * lane) * p.H + hh] : 0.f;
            gl1 = 2 * lane + 1 < ln ? p.g[(size_t)(r0 + 2 * lane + 1) * p.H + hh] : 0.f;
        }
    };
    auto map_scalars = [&]() {
        if (!PREP) return;
        const int ln = scal_len;
        if (tid >= 64 && tid < 128) beta_ld = tid - 64 < ln ? prep_sigmoid(beta_ld) : 0.f;
        if (VAR == DR_GDN && warp == 1) {
            sg0 = prep_sigmoid(gl0);
            sg1 = prep_sigmoid(gl1);
            gl0 = 2 * lane < ln ? prep_neg_softplus(gl0) : 0.f;
            gl1 = 2 * lane + 1 < ln ? prep_neg_softplus(gl1) : 0.f;
        }
    };
    uint32_t n_st = 0, n_tok = 0;  // copy groups issued on bar_st / bar_tok
    if (VAR == DR_DELTANET)  // no decay: the reference factors are 1 for every item
        for (int c = tid; c < D; c += kChunkThreads) eref[c] = gcr[c] = 1.f;
    if ((int)blockIdx.x < nitems) {
        load_scalars(blockIdx.x);
        map_scalars();
        if (tid == 0) {
            issue_tok(blockIdx.x, false);
            issue_state(blockIdx.x, false);
        }
        n_st = n_tok = 1;
    }

    int it = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++it) {
        const bool odd = it & 1;
        const uint32_t ph = (uint32_t)(it & 1);
        const int chunk = item / p.H, h = item % p.H;
        int seq, row0, len;
        chunk_info(p, chunk, seq, row0, len);
        const int next = item + gridDim.x;
        const ChunkRoles R = chunk_roles(sm, kTile, odd);
        // dq, dk, dv by tensor stores for whole chunks; per thread for a ragged chunk, and dq,
        // dk with input preparation (whose write-out chains every row through its norm)
        const bool tstore = !PREP && len == 64, tstore_v = len == 64;
        uint8_t* Qs = R.Q;      // q -> Qb
        uint8_t* Ust = R.U;     // [64][D] U
        uint8_t* dQs = R.dQ;    // dQt^T = S dO^T
        uint8_t* dSst = R.dS;   // [D][D] W-layout state gradient at the chunk end
        uint8_t* Kbs = R.Kb;    // Kb
        uint8_t* dWys = R.dWy;  // -dWyA^T -> dWy^T
        uint8_t* dUts = R.dUt;  // -dU^T -> dUt^T
        float* gC_s = gC_b + (odd ? D : 0);
        fsum = 0.f;
        if (tid >= 64 && tid < 128) beta_s[tid - 64] = beta_ld;  // mapped already (preparation)
        if (tid == kIssuer && next < nitems) {
            // the next item's q, k, v, dO boxes into L2 now; their loads into shared memory
            // can only be issued once this item's last stage has read those buffers
            const int nc = next / p.H, nh = next % p.H;
            int nsq, nr0, nln;
            chunk_info(p, nc, nsq, nr0, nln);
            for (int kb = 0; kb < D / 64; ++kb) {
                tma_prefetch_3d(&mq, kb * 64, nh, nr0);
                tma_prefetch_3d(&mk, kb * 64, nh, nr0);
                tma_prefetch_3d(&mv, kb * 64, nh, nr0);
                tma_prefetch_3d(&mdo, kb * 64, nh, nr0);
            }
            if (VAR == DR_KDA) tma_prefetch_3d(&mg, 0, nh, nr0);  // its gates (one box)
        }
        // two products of M0 read the state side only: thread 0 issues them while the token
        // tiles land (the state side was issued during the previous item's last stages)
        bool st_ok = true;
        if (tid == 0) {
            st_ok = mbar_wait(&bar_st, ph, kWaitLimitNs);
            if (st_ok) {
                tc_fence_after();
                mma_tiles(tm + C1, Tile{smem_u32(Sst), D}, true, Tile{smem_u32(dUts), D}, true, D, 64, D, false);
                mma_tiles(tm + C_dKC, Tile{smem_u32(dSst), D}, true, Tile{smem_u32(Ust), 64}, false, D, 64, D,
                          false);
            }
        }
        ok = mbar_wait(&bar_tok, ph, kWaitLimitNs) && st_ok;
        if (VAR == DR_KDA) ok = ok && mbar_wait(&bar_st, ph, kWaitLimitNs);  // the gates
        if (__syncthreads_or(!ok)) break;
        zero_pad_rows(Qs, D, len);
        zero_pad_rows(Ks, D, len);
        zero_pad_rows(Vs, D, len);
        zero_pad_rows(dOs, D, len);
        // cumulative log-decay: KDA per key channel, in place in Gam (rows past the end of
        // the sequence repeat the total); GDN per token, with its two exponentials
        float* tot = Xs + 1024;  // KDA: [P][D] block totals
        constexpr int kP = kChunkThreads / D, kR = 64 / kP;  // KDA: threads per channel, rows each
        if (VAR == DR_KDA) {
            // kP threads per channel, each the cumulative sum of a contiguous block of kR
            // rows; the decay pass adds the totals of the blocks above
            const int c = tid % D, pt = tid / D;
            float v[kR];
#pragma unroll
            for (int t = 0; t < kR; ++t) {
                v[t] = Gam[(pt * kR + t) * S::kGS + c];
                if (PREP) v[t] = prep_neg_softplus(v[t]);  // rows past the end are not added
            }
            float G = 0.f;
#pragma unroll
            for (int t = 0; t < kR; ++t) {
                if (pt * kR + t < len) G += v[t];
                v[t] = G;
            }
#pragma unroll
            for (int t = 0; t < kR; ++t) Gam[(pt * kR + t) * S::kGS + c] = v[t];
            tot[pt * D + c] = G;
        } else if (VAR == DR_GDN) {
            if (warp == 1) {
                if (PREP) {  // g = -softplus(x) (mapped already); sigmoid(x) for the chain of dg
                    sgx[2 * lane] = sg0;
                    sgx[2 * lane + 1] = sg1;
                }
                float x = gl0 + gl1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                const float G_r = __shfl_sync(0xffffffffu, x, 15);  // Gamma at token 31
                const float GL = __shfl_sync(0xffffffffu, x, 31);
                const float x0 = x - gl1;
                Erow[2 * lane] = __expf(x0 - G_r);
                Erow[2 * lane + 1] = __expf(x - G_r);
                Eirow[2 * lane] = __expf(G_r - x0);
                Eirow[2 * lane + 1] = __expf(G_r - x);
                const float er = expf(G_r), lr = expf(GL - G_r);
                for (int c = lane; c < D; c += 32) {
                    eref[c] = er;
                    gcr[c] = lr;
                }
            }
        }
        __syncthreads();
        // decay pass: Qb = q e^G and Kr = k e^-G in place; Kb = k e^G is held in registers
        // until the state-side products have read dS out of the Kb tile
        constexpr int kPer = 64 * (D / 8) / kChunkThreads;
        uint4 kbr[kPer];
        // the rows of every pass are loaded first (the stores below may not pass them), and
        // with input preparation their norms reduced together
        uint4 qv_[kPer], kv_[kPer];
        float rq_[kPer], rk_[kPer];
#pragma unroll
        for (int n = 0; n < kPer; ++n) {
            const int w = tid + n * kChunkThreads;
            const uint32_t off = sw128_offset(w / (D / 8), (w % (D / 8)) * 8, 64);
            kv_[n] = *reinterpret_cast<const uint4*>(Ks + off);
            qv_[n] = *reinterpret_cast<const uint4*>(Qs + off);
        }
        if (PREP) {  // the inverse norms of the raw rows, as tc_prep formed them (with the tiles)
#pragma unroll
            for (int n = 0; n < kPer; ++n) {
                const int i = (tid + n * kChunkThreads) / (D / 8);
                rq_[n] = rq_s[i];
                rk_[n] = rk_s[i];
            }
        }
#pragma unroll
        for (int n = 0; n < kPer; ++n) {
            const int w = tid + n * kChunkThreads;
            const int i = w / (D / 8), c8 = (w % (D / 8)) * 8;
            const uint32_t off = sw128_offset(i, c8, 64);
            const uint4 kv = kv_[n];
            if (VAR == DR_DELTANET && !PREP) {
                kbr[n] = kv;
                continue;
            }
            const uint4 qv = qv_[n];
            float q8[8], k8[8], e8[8], i8[8];
            unpack8(qv, q8);
            unpack8(kv, k8);
            if (PREP) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    q8[j] *= rq_[n];
                    k8[j] *= rk_[n];
                }
            }
            if (VAR == DR_DELTANET) {
#pragma unroll
                for (int j = 0; j < 8; ++j) e8[j] = i8[j] = 1.f;
            } else if (VAR == DR_KDA) {
                float4* gp = reinterpret_cast<float4*>(&Gam[i * S::kGS + c8]);
                const float4 g0 = gp[0], g1 = gp[1];
                float G8[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                float R8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // Gamma_r
                float L8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // Gamma_last
                for (int q = 0; q < kP; ++q) {  // totals of the row blocks
                    const float4* tp = reinterpret_cast<const float4*>(tot + q * D + c8);
                    const float4 t0v = tp[0], t1v = tp[1];
                    const float T8[8] = {t0v.x, t0v.y, t0v.z, t0v.w, t1v.x, t1v.y, t1v.z, t1v.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (q < i / kR) G8[j] += T8[j];   // the blocks above this row
                        if (q < 32 / kR) R8[j] += T8[j];  // the first 32 rows
                        L8[j] += T8[j];
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    e8[j] = __expf(G8[j] - R8[j]);
                    i8[j] = fast_rcp(e8[j]);
                }
                if (i == 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        eref[c8 + j] = expf(R8[j]);
                        gcr[c8 + j] = expf(L8[j] - R8[j]);
                    }
                }
                gp[0] = make_float4(e8[0], e8[1], e8[2], e8[3]);  // e^{Gamma - Gamma_r} from here on
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
            kbr[n] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        }
        fence_async_smem();
        __syncthreads();
        // MA: Qb Kr^T -> C3 ; dO v^T -> C4
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + C3, Tile{smem_u32(Qs), 64}, false, Tile{smem_u32(Ks), 64}, false, 64, 64, D, false);
            mma_tiles(tm + C4, Tile{smem_u32(dOs), 64}, false, Tile{smem_u32(Vs), 64}, false, 64, 64, D, false);
        }
        ok = mbar_wait(&bar_st, ph, kWaitLimitNs);
        if (__syncthreads_or(!ok)) break;

        // M0 (M = D): dQt^T = S dO^T -> C0 ; -dWyA^T = S (-dU)^T -> C1 and dKC^T = dS U^T -> C_dKC
        // were issued at the start of the item; the commit covers them
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + C0, Tile{smem_u32(Sst), D}, true, Tile{smem_u32(dOs), 64}, false, D, 64, D, false);
            mma_commit(&bar_mma);
        }
        // while M0 runs: dgC[c] = sum_v dS[c, v] S[c, v] (eight channels by a block of
        // value rows per thread, partials added in a fixed order after the wait)
        if (tid < 256) {  // the first eight warps
            constexpr int kOct = D / 8, kGroups = 256 / kOct, kRows = D / kGroups;
            const int c8 = (tid % kOct) * 8, g = tid / kOct;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int t = 0; t < kRows; ++t) {
                const uint32_t off = sw128_offset(g * kRows + t, c8, D);
                float s8[8], d8[8];
                unpack8(*reinterpret_cast<const uint4*>(Sst + off), s8);
                unpack8(*reinterpret_cast<const uint4*>(dSst + off), d8);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(s8[j], d8[j], acc[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
            if ((lane & 16) == 0) {
                const int pg = warp * (16 / kOct) + lane / kOct;  // 128 / kOct partial rows
#pragma unroll
                for (int j = 0; j < 8; ++j) Xs[pg * D + c8 + j] = acc[j];
            }
        }
        ok = mma_done();  // MA and M0
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        for (int c = tid; c < D; c += kChunkThreads) {
            float a = 0.f;
            for (int q = 0; q < 128 / (D / 8); ++q) a += Xs[q * D + c];
            dgC_s[c] = a;
        }
        // E0: Kb' into its tile; dQt^T -> its tile (U is consumed), -dWyA^T -> the dWy
        // tile (dS is consumed), both scaled by e^{Gamma_r} of their key channel
#pragma unroll
        for (int n = 0; n < kPer; ++n) {
            const int w = tid + n * kChunkThreads;
            *reinterpret_cast<uint4*>(Kbs + sw128_offset(w / (D / 8), (w % (D / 8)) * 8, 64)) = kbr[n];
        }
#pragma unroll 1
        for (int b = 0; b < kTok / 16; ++b) {
            float a[16], c_[16];
            tmem_ld16(tl + C0 + t0 + 16 * b, a);
            tmem_ld16(tl + C1 + t0 + 16 * b, c_);
            tmem_ld_wait();
            if (cl >= 0) {
                if (VAR != DR_DELTANET) {
                    const float er = eref[cl];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        a[j] *= er;
                        c_[j] *= er;
                    }
                }
                tile_store16(dQs, cl, t0 + 16 * b, D, a);
                tile_store16(dWys, cl, t0 + 16 * b, D, c_);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M1: dQt Kb^T -> C2 ; Gram Kb Kr^T -> C6 (read in E6)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + C2, Tile{smem_u32(dQs), D}, true, Tile{smem_u32(Kbs), 64}, false, 64, 64, D, false);
            mma_tiles(tm + C6, Tile{smem_u32(Kbs), 64}, false, Tile{smem_u32(Ks), 64}, false, 64, 64, D, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        // E2: Aqk = tril(Qb Kr^T) ; P = (dO v^T - dQt Kb^T) diag(beta)
#pragma unroll 1
        for (int cb = grp; cb < 4; cb += kG) {
            float a[8], p1[8], p2[8];
            tmem_ld8_x2<8>(tl + C3 + cb * 16, a);
            tmem_ld8_x2<8>(tl + C4 + cb * 16, p1);
            tmem_ld8_x2<8>(tl + C2 + cb * 16, p2);
            tmem_ld_wait();
            const int c0 = cb * 16 + h2 * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = c0 + j;
                a[j] = col <= r2 ? a[j] : 0.f;
                p1[j] = beta_s[col] * (p1[j] - p2[j]);
            }
            tile_store8(Aqs, r2, c0, 64, a);
            tile_store8(B8a, r2, c0, 64, p1);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M2: P T^T -> C0 ; dQt^T Aqk -> C1 (M = D) ; dO^T Aqk -> C2 (M = D)
        if (tid == 0) {
            tc_fence_after();
            const Tile tAq{smem_u32(Aqs), 64};
            mma_tiles(tm + C0, Tile{smem_u32(B8a), 64}, false, Tile{smem_u32(Ts), 64}, false, 64, 64, 64, false);
            mma_tiles(tm + C1, Tile{smem_u32(dQs), D}, false, tAq, true, D, 64, 64, false);
            mma_tiles(tm + C2, Tile{smem_u32(dOs), 64}, true, tAq, true, D, 64, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
#pragma unroll 1
        for (int cb = grp; cb < 4; cb += kG) {
            float a[8];
            tmem_ld8_x2<8>(tl + C0 + cb * 16, a);
            tmem_ld_wait();
            const int c0 = cb * 16 + h2 * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = (c0 + j <= r2) ? sc * a[j] : 0.f;
            tile_store8(dAqs, r2, c0, 64, a);
        }
#pragma unroll 1
        for (int b = 0; b < kTok / 16; ++b) {
            float a[16], u[16];
            tmem_ld16(tl + C1 + t0 + 16 * b, a);
            tmem_ld16(tl + C2 + t0 + 16 * b, u);
            tmem_ld_wait();
            if (cl >= 0) {
                float wa[16], nd[16];
                tile_load16(dWys, cl, t0 + 16 * b, D, wa);
                tile_load16(dUts, cl, t0 + 16 * b, D, nd);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    a[j] = wa[j] - sc * a[j];  // dWy^T (the tile held -dWyA^T)
                    u[j] = sc * u[j] - nd[j];  // dUt^T (the tile held -dU^T)
                }
                tile_store16(dWys, cl, t0 + 16 * b, D, a);
                tile_store16(dUts, cl, t0 + 16 * b, D, u);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M3: Kb dWy^T -> C0 ; v dUt^T -> C1 ; dUt^T T -> C3 (dbV^T) ; dWy^T T -> C4 (dbK^T) ;
        //     Kr^T dAqk^T -> C_dQ  (the last three M = D)
        if (tid == 0) {
            tc_fence_after();
            const Tile tT{smem_u32(Ts), 64}, tdW{smem_u32(dWys), D}, tdU{smem_u32(dUts), D};
            mma_tiles(tm + C0, Tile{smem_u32(Kbs), 64}, false, tdW, true, 64, 64, D, false);
            mma_tiles(tm + C1, Tile{smem_u32(Vs), 64}, false, tdU, true, 64, 64, D, false);
            mma_tiles(tm + C3, tdU, false, tT, true, D, 64, 64, false);
            mma_tiles(tm + C4, tdW, false, tT, true, D, 64, 64, false);
            mma_tiles(tm + C_dQ, Tile{smem_u32(Ks), 64}, true, Tile{smem_u32(dAqs), 64}, false, D, 64, 64, false);
            mma_commit(&bar_mma);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        // E4, token rows j: dT^T[j][i] = beta_j (Kb dWy^T + v dUt^T)[j][i], and the key and
        // value parts of dbeta_j = sum_c dbK[j,c] Kb[j,c] + sum_v dbV[j,v] v[j,v]
        //                        = sum_i T[i,j] (dWy Kb^T + dUt v^T)[i,j]
        float dbeta_acc = 0.f;
        {
            // column r2 of T: element (c0 + j, r2) at xr[j] + 128 (c0 + j), c0 a multiple of 8
            uint32_t xr[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) xr[k] = (uint32_t)(((((r2 >> 3) & 7) ^ k) << 4) + (r2 & 7) * 2);
            const float br = beta_s[r2];
#pragma unroll 1
            for (int n = 0; n < 4 / kG; ++n) {
                const int cb = grp + kG * n;
                float a[8], b[8];
                tmem_ld8_x2<8>(tl + C0 + cb * 16, a);
                tmem_ld8_x2<8>(tl + C1 + cb * 16, b);
                tmem_ld_wait();
                const int c0 = cb * 16 + h2 * 8;
                const uint8_t* tcol = Ts + c0 * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float s = a[j] + b[j];
                    const float tij = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16*>(tcol + xr[j] + j * 128));
                    dbeta_acc = fmaf(tij, s, dbeta_acc);
                    a[j] = br * s;
                }
                tile_store8(B8b, r2, c0, 64, a);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M4: X = dT T^T -> C0
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + C0, Tile{smem_u32(B8b), 64}, true, Tile{smem_u32(Ts), 64}, false, 64, 64, 64, false);
            mma_commit(&bar_mma);
        }
        // while M4 runs: dv[j, v] = beta_j dbV^T[v][j], staged in the v / dO tiles (both
        // consumed) and written out
        auto dv_stage = [&](auto f32) {
            constexpr bool F32 = decltype(f32)::value;
#pragma unroll 1
            for (int b = 0; b < kTok / 16; ++b) {
                uint8_t* sb = stage_base(Vs, dOs, F32) + 16 * b * D * (F32 ? 4 : 2);
                float a[16];
                tmem_ld16(tl + C3 + t0 + 16 * b, a);
                tmem_ld_wait();
                if (cl >= 0) {
                    float bt[16];
                    load16(beta_s, 16 * b, bt);
#pragma unroll
                    for (int j = 0; j < 16; ++j) stage_put<D, F32>(sb, j, bt[j] * a[j]);
                }
            }
        };
        if (f32out)
            dv_stage(BoolTag<true>{});
        else
            dv_stage(BoolTag<false>{});
        fence_async_smem();
        __syncthreads();
        if (tstore_v) {
            if (tid == kIssuer) tensor_out(&mgv, Vs, dOs, h, row0);
        } else if (f32out) {
            stage_copy_out<D, true>(p.dv_, Vs, dOs, p, row0, len, h);
        } else {
            stage_copy_out<D, false>(p.dv_, Vs, dOs, p, row0, len, h);
        }
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
#pragma unroll 1
        for (int cb = grp; cb < 4; cb += kG) {
            float a[8];
            tmem_ld8_x2<8>(tl + C0 + cb * 16, a);
            tmem_ld_wait();
            tile_store8(B8a, r2, cb * 16 + h2 * 8, 64, a);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M5: T^T X -> C0 (dA = -it)
        if (tid == 0) {
            tc_fence_after();
            mma_tiles(tm + C0, Tile{smem_u32(Ts), 64}, true, Tile{smem_u32(B8a), 64}, true, 64, 64, 64, false);
            mma_commit(&bar_mma);
        }
        // while M5 runs: dq = (scale dQt + dAqk Kr) e^{Gamma}, staged in the dUt / dWy tiles
        // (consumed), and the dQb Qb - dKC KC part of dGamma.  Tokens past the end of the
        // sequence have zero q and k rows, so they add nothing to dGamma.
        auto dq_stage = [&](auto f32) {
            constexpr bool F32 = decltype(f32)::value;
            const float gc = cl >= 0 ? gcr[cl] : 0.f;  // e^{Gamma_last - Gamma_r}
            uint8_t* sb0 = stage_base(dUts, dWys, F32);
#pragma unroll 1
            for (int b = 0; b < kTok / 8; ++b) {
                uint8_t* sb = sb0 + 8 * b * D * (F32 ? 4 : 2);
                float dq_[8], dkc[8], g[8], e8[8], ei8[8];
                tmem_ld8(tl + C_dQ + t0 + 8 * b, dq_);
                tmem_ld8(tl + C_dKC + t0 + 8 * b, dkc);
                tmem_ld_wait();
                decay8(b, e8, ei8, false);
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = 0.f;
                if (cl >= 0) {
                    float dqt[8];
                    tile_load8(dQs, cl, t0 + 8 * b, D, dqt);
                    const uint8_t* qrow = Qs + 8 * b * 128;
                    const uint8_t* krow = Ks + 8 * b * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float qb = tok(qrow, j), kr = tok(krow, j);
                        const float dQb = fmaf(sc, dqt[j], dq_[j]);
                        const float f = dkc[j] * (kr * gc);
                        g[j] = dQb * qb - f;
                        fsum += f;
                        stage_put<D, F32>(sb, j, dQb * e8[j]);
                    }
                }
                tmem_st8(tl + C1 + t0 + 8 * b, g);
                if (VAR == DR_KDA) tmem_st8(tl + C3 + t0 + 8 * b, e8);  // for the dk stage
            }
            tmem_st_wait();
        };
        if (f32out)
            dq_stage(BoolTag<true>{});
        else
            dq_stage(BoolTag<false>{});
        fence_async_smem();  // the staged dq rows may leave by a tensor store
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        // E6: dA = -T^T X (strictly lower), the A part of dbeta, dG = diag(beta) dA
#pragma unroll 1
        for (int cb = grp; cb < 4; cb += kG) {
            float a[8], gm[8];
            tmem_ld8_x2<8>(tl + C0 + cb * 16, a);
            tmem_ld8_x2<8>(tl + C6 + cb * 16, gm);
            tmem_ld_wait();
            const float br = beta_s[r2];
            const int c0 = cb * 16 + h2 * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool low = c0 + j < r2;  // the Gram above the diagonal may be inf
                const float dA = low ? -a[j] : 0.f;
                if (low) dbeta_acc = fmaf(dA, gm[j], dbeta_acc);
                a[j] = br * dA;  // dG
            }
            tile_store8(B8b, r2, c0, 64, a);
        }
        // the two threads of a row hold the sums over their halves of the columns
        dbeta_acc += __shfl_xor_sync(0xffffffffu, dbeta_acc, 16);
        if (grp > 0 && h2 == 0) part[(grp - 1) * 64 + r2] = dbeta_acc;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // M6 (M = D): Kr^T dG^T -> C6 (dKb') ; Kb^T dG + Qb^T dAqk -> C2 (dKr')
        if (tid == 0) {
            tc_fence_after();
            const Tile tG{smem_u32(B8b), 64};
            mma_tiles(tm + C6, Tile{smem_u32(Ks), 64}, true, tG, false, D, 64, 64, false);
            mma_tiles(tm + C2, Tile{smem_u32(Kbs), 64}, true, tG, true, D, 64, 64, false);
            mma_tiles(tm + C2, Tile{smem_u32(Qs), 64}, true, Tile{smem_u32(dAqs), 64}, true, D, 64, 64, true);
            mma_commit(&bar_mma);
        }
        // while M6 runs: dbeta and the staged dq go out
        if (grp == 0 && h2 == 0 && r2 < len) {
            float db = dbeta_acc;
            for (int q = 1; q < kG; ++q) db += part[(q - 1) * 64 + r2];
            if (PREP) db *= beta_s[r2] * (1.f - beta_s[r2]);  // through beta = sigmoid(b)
            p.dbeta[(size_t)(row0 + r2) * p.H + h] = db;
        }
        if (PREP) {
            // q_hat from the Qb' tile: e^{Gamma_r - Gamma} per row (GDN), 1 / e^{Gamma - Gamma_r}
            // per element (KDA, whose array still holds them), nothing (DeltaNet)
            constexpr int kSrc = VAR == DR_KDA ? 2 : 1;
            const float* rf = VAR == DR_GDN ? Eirow : nullptr;
            if (f32out)
                stage_copy_out_prep<D, true, kSrc>(p.dq, dUts, dWys, p, row0, len, h, nullptr, rq_s, Qs, rf, Gam);
            else
                stage_copy_out_prep<D, false, kSrc>(p.dq, dUts, dWys, p, row0, len, h, nullptr, rq_s, Qs, rf, Gam);
        } else if (tstore) {
            if (tid == kIssuer) tensor_out(&mgq, dUts, dWys, h, row0);
        } else if (f32out) {
            stage_copy_out<D, true>(p.dq, dUts, dWys, p, row0, len, h);
        } else {
            stage_copy_out<D, false>(p.dq, dUts, dWys, p, row0, len, h);
        }
        fence_async_smem();  // generic accesses of the buffers the next item's state goes to
        // the dv and dq stores have read their staging tiles before the next item's state
        // side and the dk stage refill them
        if (tid == kIssuer) bulk_wait_read();
        ok = mma_done();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        // the next item's state side goes into what this item no longer reads (issued by
        // the last warp, which has the least to do in the final epilogue)
        if (tid == kIssuer && next < nitems) issue_state(next, !odd);
        n_st += next < nitems;

        // E7: dk = (dKb' + beta dbK) e^{Gamma} + (dKr' + dKC e^{Gamma_last}) e^{-Gamma}, staged
        // in the v / dO tiles (consumed), and the dKb Kb - dKr Kr part of dGamma
        auto dk_stage = [&](auto f32) {
            constexpr bool F32 = decltype(f32)::value;
            const float gc = cl >= 0 ? gcr[cl] : 0.f;  // e^{Gamma_last - Gamma_r}
            uint8_t* sb0 = stage_base(Vs, dOs, F32);
#pragma unroll 1
            for (int b = 0; b < kTok / 8; ++b) {
                uint8_t* sb = sb0 + 8 * b * D * (F32 ? 4 : 2);
                float dbk[8], dkb[8], dkr[8], dkc[8], g[8], e8[8], ei8[8];
                tmem_ld8(tl + C4 + t0 + 8 * b, dbk);
                tmem_ld8(tl + C6 + t0 + 8 * b, dkb);
                tmem_ld8(tl + C2 + t0 + 8 * b, dkr);
                tmem_ld8(tl + C_dKC + t0 + 8 * b, dkc);
                tmem_ld8(tl + C1 + t0 + 8 * b, g);
                tmem_ld_wait();
                decay8(b, e8, ei8, true);
                if (cl >= 0) {
                    float bt[8];
                    load8(beta_s, 8 * b, bt);
                    const uint8_t* kbrow = Kbs + 8 * b * 128;
                    const uint8_t* krow = Ks + 8 * b * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float kb = tok(kbrow, j), kr = tok(krow, j);
                        const float dKb = fmaf(bt[j], dbk[j], dkb[j]);
                        g[j] += dKb * kb - dkr[j] * kr;
                        stage_put<D, F32>(sb, j, dKb * e8[j] + fmaf(dkc[j], gc, dkr[j]) * ei8[j]);
                    }
                }
                tmem_st8(tl + C1 + t0 + 8 * b, g);
            }
            tmem_st_wait();
        };
        if (f32out)
            dk_stage(BoolTag<true>{});
        else
            dk_stage(BoolTag<false>{});
        fence_async_smem();
        __syncthreads();
        if (tstore) {
            if (tid == kIssuer) tensor_out(&mgk, Vs, dOs, h, row0);
        } else if (PREP) {
            // k_hat from the Kr' tile times e^{Gamma - Gamma_r} per row (GDN) or nothing
            // (DeltaNet); KDA's per-element factors are gone by now (its array already holds
            // the next item's gates), so it re-reads the raw rows
            const __nv_bfloat16* rawk = static_cast<const __nv_bfloat16*>(p.k);
            constexpr int kSrc = VAR == DR_KDA ? 0 : 1;
            const float* rf = VAR == DR_GDN ? Erow : nullptr;
            if (f32out)
                stage_copy_out_prep<D, true, kSrc>(p.dk_, Vs, dOs, p, row0, len, h, rawk, rk_s, Ks, rf, nullptr);
            else
                stage_copy_out_prep<D, false, kSrc>(p.dk_, Vs, dOs, p, row0, len, h, rawk, rk_s, Ks, rf, nullptr);
        } else if (f32out) {
            stage_copy_out<D, true>(p.dk_, Vs, dOs, p, row0, len, h);
        } else {
            stage_copy_out<D, false>(p.dk_, Vs, dOs, p, row0, len, h);
        }
        // the next item's token side goes into the Kb / Kr / staging tiles
        fence_async_smem();
        __syncthreads();
        if (next < nitems) {
            if (tid == kIssuer) {
                bulk_wait_read();  // the dk store has read the staging tiles
                issue_tok(next, !odd);
            }
            load_scalars(next);
            ++n_tok;
        }

        // E8: dg_i = (dgC e^{Gamma_last} + sum_rows dKC KC) + sum_{j >= i} dGamma_j
        float dG[kTok];
        if (VAR != DR_DELTANET) {
            tc_fence_after();
#pragma unroll
            for (int b = 0; b < kTok / 16; ++b) {
                float g16[16];
                tmem_ld16(tl + C1 + t0 + 16 * b, g16);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) dG[16 * b + j] = g16[j];
            }
        }
        if (VAR == DR_KDA) {
            // the token groups of a channel exchange their totals
            float* sgq = Xs;           // [kG][D] sum of dGamma over each group's tokens
            float* fq = Xs + kG * D;   // [kG][D] sum of dKC KC over each group's tokens
            float sg = 0.f;
#pragma unroll
            for (int k = 0; k < kTok; ++k) sg += dG[k];
            if (cl >= 0) {
                sgq[grp * D + cl] = sg;
                fq[grp * D + cl] = fsum;
            }
            __syncthreads();
            if (cl >= 0) {
                float run = dgC_s[cl] * gC_s[cl];
                for (int q = 0; q < kG; ++q) run += fq[q * D + cl];
                for (int q = grp + 1; q < kG; ++q) run += sgq[q * D + cl];
                float sx[PREP ? kTok : 1];  // sigmoid of the raw gate arguments
                if (PREP) {
#pragma unroll
                    for (int k = 0; k < kTok; ++k) {
                        const int i = t0 + k;
                        sx[k] = i < len ? __ldg(p.g + ((size_t)(row0 + i) * p.H + h) * D + cl) : 0.f;
                    }
#pragma unroll
                    for (int k = 0; k < kTok; ++k) sx[k] = prep_sigmoid(sx[k]);
                }
#pragma unroll
                for (int k = kTok - 1; k >= 0; --k) {
                    const int i = t0 + k;
                    run += dG[k];
                    // through g = -softplus(x): dx = -dg sigmoid(x)
                    if (i < len) p.dg[((size_t)(row0 + i) * p.H + h) * D + cl] = PREP ? -run * sx[PREP ? k : 0] : run;
                }
            }
        } else if (VAR == DR_GDN) {
            float* red = Xs;          // [4 channel quarters][64 rows]
            float* fw = Xs + 256;     // [kChunkThreads / 32 warps]
            const float rs = warp_transpose_sum<kTok>(dG);  // row t0 + lane % kTok, this warp's channels
            if (lane < kTok) red[(warp & 3) * 64 + t0 + lane] = rs;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) fsum += __shfl_xor_sync(0xffffffffu, fsum, o);
            if (lane == 0) fw[warp] = fsum;
            __syncthreads();
            if (tid < 64) rowsum[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
            __syncthreads();
            if (warp == 0) {
                float e = 0.f;
                for (int w = 0; w < kChunkThreads / 32; ++w) e += fw[w];
                float ec = 0.f;
                for (int c = lane; c < D; c += 32) ec += dgC_s[c] * gC_s[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ec += __shfl_xor_sync(0xffffffffu, ec, o);
                e += ec;
                const float a0 = 2 * lane < len ? rowsum[2 * lane] : 0.f;
                const float a1 = 2 * lane + 1 < len ? rowsum[2 * lane + 1] : 0.f;
                float x = a0 + a1;  // suffix sum over lanes >= this one
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_down_sync(0xffffffffu, x, o);
                    if (lane + o < 32) x += y;
                }
                const size_t g0 = (size_t)(row0 + 2 * lane) * p.H + h, g1 = g0 + p.H;
                // through g = -softplus(x): dx = -dg sigmoid(x), sigmoid(x) kept by the scan
                if (2 * lane < len) p.dg[g0] = PREP ? -(e + x) * sgx[2 * lane] : e + x;
                if (2 * lane + 1 < len) p.dg[g1] = PREP ? -(e + x - a0) * sgx[2 * lane + 1] : e + x - a0;
            }
        }
        if (next < nitems) map_scalars();  // the next item's (loaded before E8)
        tc_fence_before();
        __syncthreads();  // Xs, TMEM and the small arrays are reused by the next item
    }
    if (!ok) {
        // leave no copy in flight: wait (bounded) for every group issued and not yet waited
        record_timeout(p);
        for (uint32_t q = (uint32_t)it; q < n_st; ++q) mbar_wait(&bar_st, q & 1, kWaitLimitNs);
        for (uint32_t q = (uint32_t)it; q < n_tok; ++q) mbar_wait(&bar_tok, q & 1, kWaitLimitNs);
    }
    if (tid == kIssuer) bulk_wait_all();  // the last item's gradient stores
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// -dU^T of the emitted write's gradient as [D][64] tile images per (chunk, head), the
// form the backward scan adds to its own -dU^T tile (tokens past the end of a
// sequence are zero).  Thread (value channel v, 8 tokens) packs one 16-byte chunk.
template <int D>
__global__ void __launch_bounds__(256) pack_dux_kernel(const Params p, const TcLayout L) {
    const int chunk = blockIdx.x, h = blockIdx.y;
    int seq, row0, len;
    chunk_info(p, chunk, seq, row0, len);
    uint8_t* img = L.dUx + ((size_t)chunk * p.H + h) * (64 * D * 2);
    for (int w = threadIdx.x; w < D * 8; w += blockDim.x) {
        const int v = w % D, j = w / D;
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int i = 8 * j + t;
            x[t] = i < len ? -ld_any(p.dU, ((size_t)(row0 + i) * p.H + h) * D + v, p.io_dtype) : 0.f;
        }
        *reinterpret_cast<uint4*>(img + sw128_offset(v, 8 * j, D)) =
            make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                       pack_bf16(x[6], x[7]));
    }
}

template <int D>
cudaError_t tc_bwd_d(const Params& p, cudaStream_t st, bool reuse) {
    if (!reuse) {
        cudaError_t e = tc_fwd(p, st, false);
        if (e != cudaSuccess) return e;
    }
    const TcLayout L = tc_layout(p);
    const long long rows = (long long)p.B * p.T;
    CUtensorMap mq, mk, mv, mdo, mg;
    if (!make_token_map(&mq, p.q, D, p.H, rows) || !make_token_map(&mk, p.k, D, p.H, rows) ||
        !make_token_map(&mv, p.v, D, p.H, rows) || !make_token_map(&mdo, p.dO, D, p.H, rows))
        return cudaErrorInvalidValue;
    if (p.variant == DR_KDA ? !make_gate_map(&mg, p.g, D, p.H, rows, 64) : !make_token_map(&mg, p.q, D, p.H, rows))
        return cudaErrorInvalidValue;
    CUtensorMap mgq, mgk, mgv;  // dq, dk, dv written by tensor stores
    const bool gf32 = p.grad_dtype == DR_F32;
    if (!make_out_map(&mgq, p.dq, D, p.H, rows, gf32) || !make_out_map(&mgk, p.dk_, D, p.H, rows, gf32) ||
        !make_out_map(&mgv, p.dv_, D, p.H, rows, gf32))
        return cudaErrorInvalidValue;
    if (p.dU && p.num_chunks > 0) {
        TraceScope ts("pack_dux", st);
        pack_dux_kernel<D><<<dim3(p.num_chunks, p.H), 256, 0, st>>>(p, L);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        auto launch_scan = [&](auto kernel, int bv, int smem,
                               std::atomic<unsigned long long>& attr) -> cudaError_t {
            {
                const cudaError_t e = set_smem_once(kernel, smem, attr);
                if (e != cudaSuccess) return e;
            }
            TraceScope ts("tc_scan_bwd", st);
            kernel<<<dim3(p.N * p.H, D / bv), kScanBwdThreads, smem, st>>>(mdo, p, L);
            return cudaGetLastError();
        };
        static std::atomic<unsigned long long> s64{0}, s128{0};
        cudaError_t e;
        if (D == 128 && p.N * p.H >= 120)
            e = launch_scan(tc_scan_bwd_kernel<D, (D == 128 ? 128 : 64)>, D == 128 ? 128 : 64,
                            BScanSmem<D, (D == 128 ? 128 : 64)>::kBytes, s128);
        else
            e = launch_scan(tc_scan_bwd_kernel<D, 64>, 64, BScanSmem<D, 64>::kBytes, s64);
        if (e != cudaSuccess) return e;
    }
    if (p.num_chunks == 0) return cudaSuccess;
    auto chunk_launch = [&](auto kernel, int smem, std::atomic<unsigned long long>& attr) -> cudaError_t {
        {
            const cudaError_t e = set_smem_once(kernel, smem, attr);
            if (e != cudaSuccess) return e;
        }
        // persistent: one CTA per SM of the current device, each taking work items
        // (chunk, head) in a stride
        int dev = 0, nsm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (nsm <= 0) nsm = 1;
        const long long items = (long long)p.num_chunks * p.H;
        const int grid = (int)(items < nsm ? items : nsm);
        {
            TraceScope ts("tc_bwd_chunk", st);
            kernel<<<grid, kChunkThreads, smem, st>>>(mq, mk, mv, mdo, mg, mgq, mgk, mgv, p, L);
        }
        return cudaGetLastError();
    };
    // one attribute flag per instantiation (variant x preparation x gradient type)
    static std::atomic<unsigned long long> attr[12];
    auto pick = [&](auto var, auto prep) -> cudaError_t {
        constexpr int V = decltype(var)::value;
        constexpr bool P = decltype(prep)::value;
        constexpr int slot = (V * 2 + (P ? 1 : 0)) * 2;
        if (p.grad_dtype == DR_F32)
            return chunk_launch(tc_bwd_chunk_kernel<D, V, P, true>, BChunkSmem<D, V>::kBytes, attr[slot + 1]);
        return chunk_launch(tc_bwd_chunk_kernel<D, V, P, false>, BChunkSmem<D, V>::kBytes, attr[slot]);
    };
    using DN = std::integral_constant<int, DR_DELTANET>;
    using GD = std::integral_constant<int, DR_GDN>;
    using KD = std::integral_constant<int, DR_KDA>;
    switch (p.variant * 2 + (p.prepare ? 1 : 0)) {
        case 2 * DR_DELTANET: return pick(DN{}, std::false_type{});
        case 2 * DR_DELTANET + 1: return pick(DN{}, std::true_type{});
        case 2 * DR_GDN: return pick(GD{}, std::false_type{});
        case 2 * DR_GDN + 1: return pick(GD{}, std::true_type{});
        case 2 * DR_KDA: return pick(KD{}, std::false_type{});
        default: return pick(KD{}, std::true_type{});
    }
}

}  // namespace

cudaError_t tc_bwd(const Params& p, cudaStream_t st, bool reuse) {
    return p.dk == 128 ? tc_bwd_d<128>(p, st, reuse) : tc_bwd_d<64>(p, st, reuse);
}

}  // namespace dr
