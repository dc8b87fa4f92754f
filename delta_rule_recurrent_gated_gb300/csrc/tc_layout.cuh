// tc_layout.cuh -- workspace layout of the bf16 tensor-core path.
//
// Every per-chunk intermediate is kept per (chunk, head) record rec = chunk*H + h.
// "Tile images" are byte-for-byte copies of SW128 shared-memory tiles (see
// tc.cuh) so a kernel fetches one with a single untiled bulk copy.
//   Wy, Qt, KC        : [64 tokens][D] tile images             (64*D*2 bytes)
//   Ut, Ot, U         : [64 tokens][D value channels] tile images
//   dU                : [D value channels][64 tokens] tile image of -dU^T
//   T                 : [64][64] tile image of the UT inverse  (8 KB)
//   S, dS             : [D rows = value channel][D cols = key channel] tile images
//                       (W layout) of the state at the chunk start / of dL/d(state
//                       at the chunk end)                       (D*D*2 bytes)
//   gC                : [D] fp32, e^{Gamma} at the chunk's last token
//   dUx               : [D][64] tile image of -dU^T for the gradient of the emitted
//                       write (dr_bwd_u), packed before the backward scan
//   RN (with DR_FLAG_PREPARE_INPUTS only)
//                     : [2][64] fp32, rsqrt(sum x^2 + eps) of the chunk's raw q and k rows,
//                       written by tc_prep, read by tc_bwd_chunk
#pragma once
#include <cstdint>

#include "common.cuh"

namespace dr {

struct TcLayout {
    uint8_t *Wy, *Qt, *KC, *U, *dU, *Ut, *Ot, *T, *S, *dS, *dUx;
    float* gC;
    float* RN;
};

__host__ __device__ inline size_t tc_align(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Byte offsets of the arrays for `recs` records of head size D, starting at 0.
struct TcSizes {
    size_t kd, dd, cc, g;
    __host__ __device__ explicit TcSizes(int D)
        : kd((size_t)64 * D * 2), dd((size_t)D * D * 2), cc(64 * 64 * 2), g((size_t)D * 4) {}
};

__host__ inline size_t tc_layout_bytes(size_t recs, int D, bool prep) {
    TcSizes s(D);
    return tc_align(recs * s.kd) * 8 + tc_align(recs * s.cc) + tc_align(recs * s.dd) * 2 +
           tc_align(recs * s.g) + (prep ? tc_align(recs * 512) : 0);
}

__host__ inline TcLayout tc_layout_at(uint8_t* base, size_t recs, int D, bool prep) {
    TcSizes s(D);
    TcLayout L;
    uint8_t* p = base;
    auto take = [&](size_t n) { uint8_t* r = p; p += tc_align(n); return r; };
    L.Wy = take(recs * s.kd);
    L.Qt = take(recs * s.kd);
    L.KC = take(recs * s.kd);
    L.U = take(recs * s.kd);
    L.dU = take(recs * s.kd);
    L.Ut = take(recs * s.kd);
    L.Ot = take(recs * s.kd);
    L.T = take(recs * s.cc);
    L.S = take(recs * s.dd);
    L.dS = take(recs * s.dd);
    L.dUx = take(recs * s.kd);
    L.gC = reinterpret_cast<float*>(take(recs * s.g));
    L.RN = prep ? reinterpret_cast<float*>(take(recs * 512)) : nullptr;
    return L;
}

}  // namespace dr
