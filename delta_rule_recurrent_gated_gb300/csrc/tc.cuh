// tc.cuh -- thin inline-PTX layer over the sm_100-family asynchronous units used
// by the kernels of this library: mbarriers, TMA tensor loads
// (cp.async.bulk.tensor), and the 5th-generation tensor cores (tcgen05.mma with
// accumulators in tensor memory, TMEM).
//
// Shared-memory operand format used everywhere ("SW128 K-major tile"): a tile of
// R rows x K bf16 elements is stored as K/64 column blocks; each block holds the
// R rows at 128 bytes per row (64 elements), R/8 swizzle atoms of 8 rows x 128 B
// (1024 B).  Inside an atom the 16-byte chunk j of row r sits at chunk position
// j ^ (r & 7).  This is what a TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a
// box of 64 elements writes, and what the tcgen05 shared-memory descriptor with
// layout "128B swizzle" reads.  Each block starts on a 1024-byte boundary.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// make barrier initialisation visible to the async proxy (TMA, tensor cores)
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on the phase with the given parity.  Returns false if the phase
// did not complete within `limit_ns` nanoseconds (the caller then records an
// error and leaves); never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- proxies
// generic-proxy writes to shared memory -> visible to the async proxy
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Prefetch one box of a tensor map into L2 (no shared memory written, nothing to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- TMEM
// Allocation: one whole warp executes these.  `dst` is a shared-memory word
// that receives the TMEM base address.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major operand: lbo unused (16), sbo = byte distance between 8-row groups.
//   MN-major operand: lbo = byte distance between 64-element MN blocks,
//                     sbo = byte distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major = false,
                                                  bool b_mn_major = false) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- TMEM -> registers
// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp receives
// columns [col, col+16) of TMEM lane (warp_base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 lanes x 32 bits, twice: threads 0..15 of the warp receive columns [col, col+16) of
// TMEM lanes (warp_base + t), threads 16..31 columns [col + OFF, col + OFF + 16) of lanes
// (warp_base + t - 16).  An M = 64 accumulator keeps its rows in lanes 0..15 of each
// warp quarter, so this shape gives every thread of the warp half of a row's columns.
template <int OFF>
__device__ __forceinline__ void tmem_ld16_x2(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr), "n"(OFF));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// The same shape, 8 columns per half: threads 0..15 columns [col, col+8), threads 16..31
// columns [col + OFF, col + OFF + 8).
template <int OFF>
__device__ __forceinline__ void tmem_ld8_x2(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr), "n"(OFF));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 8 consecutive columns of the warp's 32 lanes (thread t: lane warp_base + t).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// registers -> TMEM, the same shape: thread t writes 8 consecutive columns of lane
// (warp_base + t); complete for a later tcgen05.ld of the thread after tmem_st_wait().
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- SW128 tile addressing
// Byte offset of element (row, k) inside an SW128 K-major tile with `rows` rows.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
    const int blk = k >> 6;           // 64-element column block
    const int kk = k & 63;
    const int chunk = kk >> 3;        // 16-byte chunk inside the 128-byte row
    const int within = (kk & 7) * 2;  // byte inside the chunk
    return (uint32_t)(blk * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + within);
}

// Reciprocal through the hardware approximation (about 1 ulp): used for e^{-Gamma}
// from e^{Gamma}, where the result is rounded to bf16 or multiplies bf16 data.
__device__ __forceinline__ float fast_rcp(float x) { return __fdividef(1.f, x); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace tc

namespace tc {

// ---------------------------------------------------------------- bulk copy (untiled)
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-aligned),
// completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, 16-aligned) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- operand tiles
// An SW128 tile in shared memory: `rows` x `cols` bf16, cols a multiple of 64.
struct Tile {
    uint32_t saddr;
    int rows;
};
// Descriptor of the 16-wide K slice starting at kk when the tile is used
// K-major (the tile's columns are the contraction index).
__device__ __forceinline__ uint64_t desc_kmajor(const Tile& t, int kk) {
    return sdesc_sw128(t.saddr + (uint32_t)((kk >> 6) * (t.rows * 128) + (kk & 63) * 2), 16, 1024);
}
// Descriptor of the 16-row K slice starting at kk when the tile is used
// MN-major (the tile's rows are the contraction index).
__device__ __forceinline__ uint64_t desc_mnmajor(const Tile& t, int kk) {
    return sdesc_sw128(t.saddr + (uint32_t)(kk * 128), (uint32_t)(t.rows * 128), 1024);
}
// D[tmem] (+)= op(A) op(B), M x N, contraction K (multiple of 16).
//   a_rows_are_k == false: A tile is [M][K];  true: A tile is [K][M] (uses A^T).
//   b_rows_are_k == false: B tile is [N][K];  true: B tile is [K][N].
// i.e. with both false D = A B^T.  Issued by a single thread.
__device__ __forceinline__ void mma_tiles(uint32_t d_tmem, const Tile& A, bool a_rows_are_k,
                                          const Tile& B, bool b_rows_are_k, int M, int N, int K,
                                          bool accumulate) {
    const uint32_t idesc = idesc_bf16(M, N, a_rows_are_k, b_rows_are_k);
    for (int kk = 0; kk < K; kk += 16) {
        const uint64_t ad = a_rows_are_k ? desc_mnmajor(A, kk) : desc_kmajor(A, kk);
        const uint64_t bd = b_rows_are_k ? desc_mnmajor(B, kk) : desc_kmajor(B, kk);
        mma_bf16(d_tmem, ad, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ __nv_bfloat16* tile_elem(uint8_t* base, int row, int col, int rows) {
    return reinterpret_cast<__nv_bfloat16*>(base + sw128_offset(row, col, rows));
}
// Write 16 consecutive values (col0 multiple of 16) of one tile row as bf16.
__device__ __forceinline__ void tile_store16(uint8_t* base, int row, int col0, int rows,
                                             const float (&v)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 u;
        u.x = pack_bf16(v[8 * h + 0], v[8 * h + 1]);
        u.y = pack_bf16(v[8 * h + 2], v[8 * h + 3]);
        u.z = pack_bf16(v[8 * h + 4], v[8 * h + 5]);
        u.w = pack_bf16(v[8 * h + 6], v[8 * h + 7]);
        *reinterpret_cast<uint4*>(base + sw128_offset(row, col0 + 8 * h, rows)) = u;
    }
}
// Write 8 consecutive values (col0 multiple of 8) of one tile row as bf16.
__device__ __forceinline__ void tile_store8(uint8_t* base, int row, int col0, int rows,
                                            const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16(v[0], v[1]);
    u.y = pack_bf16(v[2], v[3]);
    u.z = pack_bf16(v[4], v[5]);
    u.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(base + sw128_offset(row, col0, rows)) = u;
}
// Read 16 consecutive values (col0 multiple of 16) of one tile row.
__device__ __forceinline__ void tile_load16(const uint8_t* base, int row, int col0, int rows,
                                            float (&v)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 u =
            *reinterpret_cast<const uint4*>(base + sw128_offset(row, col0 + 8 * h, rows));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
            v[8 * h + 2 * j] = __low2float(b);
            v[8 * h + 2 * j + 1] = __high2float(b);
        }
    }
}
// Read 8 consecutive values (col0 multiple of 8) of one tile row.
__device__ __forceinline__ void tile_load8(const uint8_t* base, int row, int col0, int rows,
                                           float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(base + sw128_offset(row, col0, rows));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
        v[2 * j] = __low2float(b);
        v[2 * j + 1] = __high2float(b);
    }
}
// Unpack 8 bf16 held in a uint4.
__device__ __forceinline__ void unpack8(const uint4& u, float* v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
        v[2 * j] = __low2float(b);
        v[2 * j + 1] = __high2float(b);
    }
}

// TMEM lane base of the calling warp (32 lanes per warp quarter)
__device__ __forceinline__ uint32_t warp_lane_base(uint32_t tmem) {
    return tmem + ((uint32_t)((threadIdx.x >> 5) & 3) * 32u << 16);
}
// Row of an M = 64 accumulator that tmem_ld16_x2 gives this thread (both halves of the
// warp read rows 16w..16w+15 of warp quarter w), and which half of the columns.
__device__ __forceinline__ int m64_row_x2() {
    return (int)((threadIdx.x >> 5) & 3) * 16 + (int)(threadIdx.x & 15);
}
__device__ __forceinline__ int m64_half_x2() { return (int)((threadIdx.x >> 4) & 1); }
// Row of the accumulator held by this thread for an M = 64 product (rows
// 16w..16w+15 sit in lanes 0..15 of warp quarter w), or -1.
__device__ __forceinline__ int m64_row() {
    const int lane = threadIdx.x & 31;
    return lane < 16 ? (int)((threadIdx.x >> 5) & 3) * 16 + lane : -1;
}

}  // namespace tc

namespace tc {
// ---------------------------------------------------------------- bulk copy shared -> global
// Untiled copy of `bytes` (multiple of 16, 16-aligned) from shared to global
// memory through the bulk-copy engine, tracked as a bulk async-group of the
// issuing thread.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until the sources of all committed bulk stores have been read
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the same, except for the most recently committed group
__device__ __forceinline__ void bulk_wait_read_but_newest() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Tiled store of one box of a tensor map from shared memory (the box's layout, including
// its swizzle, as a load of the same map writes it), tracked as a bulk async-group of the
// issuing thread.  c0 * element size must be a multiple of 16 bytes; no negative
// coordinate.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1,
                                             int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
// wait until all committed bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
}  // namespace tc
