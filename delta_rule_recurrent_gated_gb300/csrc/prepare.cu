// prepare.cu -- input preparation (DR_FLAG_PREPARE_INPUTS): the caller passes q and k
// before their per-(token, head) L2 normalisation, beta as a logit and the gate as the
// argument of -softplus; the library writes the prepared tensors into its workspace, runs
// the path on them, and chains the path's gradients back to the raw tensors in place.
//
//   qn = q * rsqrt(sum_c q_c^2 + eps)   (the same for k; eps = 1e-6)
//   beta = sigmoid(b)                    g = -softplus(x) = -log(1 + e^x)
// and, on the caller's gradient buffers,
//   dq <- rsqrt(sum q^2 + eps) * (dqn - qn (qn . dqn))      (the same for dk)
//   db <- dbeta * beta (1 - beta)        dx <- -dg * sigmoid(x)
//
// Streaming, HBM-bound kernels.  Rows: a group of L = d_k / E lanes owns one (token, head)
// row, each lane E consecutive values (one 16-byte vector of the io type), so a row moves
// as contiguous 16-byte accesses and its sums need log2(L) shuffles; every lane keeps two
// row groups in flight.  Gates: float4 accesses, two per thread in flight, scalar tails.
#include "common.cuh"
#include "trace.cuh"

namespace dr {
namespace {

constexpr float kNormEps = 1e-6f;
constexpr int kThreads = 256;
constexpr int kUnroll = 2;

template <int BYTES> struct RawVec;
template <> struct RawVec<8> { uint2 v[1]; };
template <> struct RawVec<16> { uint4 v[1]; };
template <> struct RawVec<32> { uint4 v[2]; };

template <typename T, int E> union Pack {
    RawVec<E * sizeof(T)> raw;
    T t[E];
};

template <typename T, int E>
__device__ __forceinline__ void ld_vec(const T* p, float (&x)[E]) {
    Pack<T, E> pk;
    constexpr int B = E * sizeof(T);
    if constexpr (B == 8) {
        pk.raw.v[0] = *reinterpret_cast<const uint2*>(p);
    } else {
#pragma unroll
        for (int i = 0; i < B / 16; ++i) pk.raw.v[i] = reinterpret_cast<const uint4*>(p)[i];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = to_f<T>(pk.t[e]);
}

template <typename T, int E>
__device__ __forceinline__ void st_vec(T* p, const float (&x)[E]) {
    Pack<T, E> pk;
#pragma unroll
    for (int e = 0; e < E; ++e) pk.t[e] = from_f<T>(x[e]);
    constexpr int B = E * sizeof(T);
    if constexpr (B == 8) {
        *reinterpret_cast<uint2*>(p) = pk.raw.v[0];
    } else {
#pragma unroll
        for (int i = 0; i < B / 16; ++i) reinterpret_cast<uint4*>(p)[i] = pk.raw.v[i];
    }
}

// sum over the L lanes of an aligned lane group (L a power of two)
template <int L>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// rows [0, rows) are q's, [rows, 2 rows) k's
template <typename T, int DK>
__global__ void __launch_bounds__(kThreads)
    normalize_rows_kernel(const T* __restrict__ q, const T* __restrict__ k, T* __restrict__ qn,
                          T* __restrict__ kn, long long rows) {
    constexpr int E = 16 / sizeof(T), L = DK / E, RPW = 32 / L;
    static_assert(L >= 1 && L <= 32 && DK % E == 0, "row split");
    const int lane = threadIdx.x & 31, sub = lane / L, li = lane % L;
    const long long total = 2 * rows;
    const long long nw = (long long)gridDim.x * (kThreads / 32);
    for (long long r0 = (blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5)) * RPW * kUnroll;
         r0 < total; r0 += nw * RPW * kUnroll) {
        float x[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long r = r0 + u * RPW + sub;
            if (r < total) {
                const T* src = r < rows ? q + r * DK : k + (r - rows) * DK;
                ld_vec<T, E>(src + li * E, x[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(x[u][e], x[u][e], ss);
            const float rinv = rsqrtf(group_sum<L>(ss) + kNormEps);
#pragma unroll
            for (int e = 0; e < E; ++e) x[u][e] *= rinv;
            const long long r = r0 + u * RPW + sub;
            if (r < total) st_vec<T, E>((r < rows ? qn + r * DK : kn + (r - rows) * DK) + li * E, x[u]);
        }
    }
}

// in place on dq (rows [0, rows)) and dk (rows [rows, 2 rows)), from the raw q, k
template <typename TI, typename TG, int DK>
__global__ void __launch_bounds__(kThreads)
    chain_rows_kernel(const TI* __restrict__ q, const TI* __restrict__ k, TG* __restrict__ dq,
                      TG* __restrict__ dk, long long rows) {
    constexpr int E = 16 / sizeof(TI), L = DK / E, RPW = 32 / L;
    static_assert(L >= 1 && L <= 32 && DK % E == 0, "row split");
    const int lane = threadIdx.x & 31, sub = lane / L, li = lane % L;
    const long long total = 2 * rows;
    const long long nw = (long long)gridDim.x * (kThreads / 32);
    for (long long r0 = (blockIdx.x * (long long)(kThreads / 32) + (threadIdx.x >> 5)) * RPW * kUnroll;
         r0 < total; r0 += nw * RPW * kUnroll) {
        float x[kUnroll][E], dn[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long r = r0 + u * RPW + sub;
            if (r < total) {
                const bool is_q = r < rows;
                const long long row = is_q ? r : r - rows;
                ld_vec<TI, E>((is_q ? q : k) + row * DK + li * E, x[u]);
                ld_vec<TG, E>((is_q ? dq : dk) + row * DK + li * E, dn[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] = dn[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float ss = 0.f, xd = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ss = fmaf(x[u][e], x[u][e], ss);
                xd = fmaf(x[u][e], dn[u][e], xd);
            }
            ss = group_sum<L>(ss);
            xd = group_sum<L>(xd);
            const float rinv = rsqrtf(ss + kNormEps);
            const float dot = xd * rinv;  // qn . dqn
#pragma unroll
            for (int e = 0; e < E; ++e) dn[u][e] = rinv * (dn[u][e] - x[u][e] * rinv * dot);
            const long long r = r0 + u * RPW + sub;
            if (r < total) {
                const bool is_q = r < rows;
                st_vec<TG, E>((is_q ? dq : dk) + (is_q ? r : r - rows) * DK + li * E, dn[u]);
            }
        }
    }
}

__device__ __forceinline__ float sigmoid(float b) { return 1.f / (1.f + expf(-b)); }
__device__ __forceinline__ float neg_softplus(float x) {
    return -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
}

// OP 0: dst = sigmoid(src); 1: dst = -softplus(src);
//    2: dst *= s (1 - s), s = sigmoid(src);  3: dst *= -sigmoid(src)
template <int OP>
__device__ __forceinline__ float gate_op(float src, float dst) {
    if constexpr (OP == 0) return sigmoid(src);
    if constexpr (OP == 1) return neg_softplus(src);
    if constexpr (OP == 2) {
        const float s = sigmoid(src);
        return dst * s * (1.f - s);
    }
    return -dst * sigmoid(src);
}

// n values; src and dst 16-byte aligned
template <int OP>
__device__ __forceinline__ void map_range(const float* __restrict__ src, float* __restrict__ dst,
                                          long long n, long long tid, long long nthreads) {
    const long long n4 = n / 4;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst);
    for (long long i = tid; i < n4; i += kUnroll * nthreads) {
        float4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long j = i + u * nthreads;
            if (j < n4) {
                a[u] = s4[j];
                if constexpr (OP >= 2) b[u] = d4[j];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long j = i + u * nthreads;
            if (j < n4) {
                float4 o;
                o.x = gate_op<OP>(a[u].x, OP >= 2 ? b[u].x : 0.f);
                o.y = gate_op<OP>(a[u].y, OP >= 2 ? b[u].y : 0.f);
                o.z = gate_op<OP>(a[u].z, OP >= 2 ? b[u].z : 0.f);
                o.w = gate_op<OP>(a[u].w, OP >= 2 ? b[u].w : 0.f);
                d4[j] = o;
            }
        }
    }
    for (long long i = n4 * 4 + tid; i < n; i += nthreads) dst[i] = gate_op<OP>(src[i], dst[i]);
}

// forward (CHAIN false): beta_out = sigmoid(b), g_out = -softplus(x)
// backward (CHAIN true): dbeta *= beta (1 - beta), dg *= -sigmoid(x), in place
template <bool CHAIN>
__global__ void __launch_bounds__(kThreads)
    gates_kernel(const float* __restrict__ b, const float* __restrict__ x, float* beta_out,
                 float* g_out, long long nb, long long ng) {
    const long long tid = blockIdx.x * (long long)kThreads + threadIdx.x;
    const long long nthreads = (long long)gridDim.x * kThreads;
    map_range<CHAIN ? 2 : 0>(b, beta_out, nb, tid, nthreads);
    if (ng) map_range<CHAIN ? 3 : 1>(x, g_out, ng, tid, nthreads);
}

// One block per slice of the work: blocks that finish make room for new ones, so loads
// of new blocks overlap the stores of finishing ones (the loops above still stride the
// grid, should the work ever exceed the grid limit).
int stream_grid(long long blocks_needed) {
    const long long cap = 0x7fffffffll;
    return (int)(blocks_needed < 1 ? 1 : (blocks_needed < cap ? blocks_needed : cap));
}

long long gate_count(const Params& p) {
    const long long th = (long long)p.B * p.T * p.H;
    return p.variant == DR_DELTANET ? 0 : p.variant == DR_GDN ? th : th * p.dk;
}

template <typename T, int DK>
cudaError_t launch_normalize(const Params& p, void* qn, void* kn, long long rows, cudaStream_t st) {
    constexpr int E = 16 / sizeof(T), RPW = 32 / (DK / E);
    const long long per_block = (long long)(kThreads / 32) * RPW * kUnroll;
    normalize_rows_kernel<T, DK><<<stream_grid((2 * rows + per_block - 1) / per_block), kThreads, 0,
                                   st>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k),
                                         static_cast<T*>(qn), static_cast<T*>(kn), rows);
    return cudaGetLastError();
}

template <typename TI, typename TG, int DK>
cudaError_t launch_chain(const Params& p, long long rows, cudaStream_t st) {
    constexpr int E = 16 / sizeof(TI), RPW = 32 / (DK / E);
    const long long per_block = (long long)(kThreads / 32) * RPW * kUnroll;
    chain_rows_kernel<TI, TG, DK><<<stream_grid((2 * rows + per_block - 1) / per_block), kThreads, 0,
                                    st>>>(static_cast<const TI*>(p.q), static_cast<const TI*>(p.k),
                                          static_cast<TG*>(p.dq), static_cast<TG*>(p.dk_), rows);
    return cudaGetLastError();
}

// d_k in {16, 32, 64, 128} (the supported sets of both paths); others are refused
template <typename T>
cudaError_t normalize_dk(const Params& p, void* qn, void* kn, long long rows, cudaStream_t st) {
    switch (p.dk) {
        case 16: return launch_normalize<T, 16>(p, qn, kn, rows, st);
        case 32: return launch_normalize<T, 32>(p, qn, kn, rows, st);
        case 64: return launch_normalize<T, 64>(p, qn, kn, rows, st);
        case 128: return launch_normalize<T, 128>(p, qn, kn, rows, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TI, typename TG>
cudaError_t chain_dk(const Params& p, long long rows, cudaStream_t st) {
    switch (p.dk) {
        case 16: return launch_chain<TI, TG, 16>(p, rows, st);
        case 32: return launch_chain<TI, TG, 32>(p, rows, st);
        case 64: return launch_chain<TI, TG, 64>(p, rows, st);
        case 128: return launch_chain<TI, TG, 128>(p, rows, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gates(const Params& p, const float* b, const float* x, float* bo, float* go,
                         bool chain, cudaStream_t st) {
    const long long th = (long long)p.B * p.T * p.H, ng = gate_count(p);
    const long long vec = (th > ng ? th : ng) / 4 + 1;
    const int grid = stream_grid((vec + (long long)kThreads * kUnroll - 1) / (kThreads * kUnroll));
    if (chain) gates_kernel<true><<<grid, kThreads, 0, st>>>(b, x, bo, go, th, ng);
    else gates_kernel<false><<<grid, kThreads, 0, st>>>(b, x, bo, go, th, ng);
    return cudaGetLastError();
}

}  // namespace

size_t prepare_bytes(const Params& p) {
    const long long th = (long long)p.B * p.T * p.H;
    const size_t s = p.io_dtype == DR_F32 ? 4 : 2;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return 2 * al(th * p.dk * s) + al(th * 4) + al(gate_count(p) * 4);
}

// Points p at the prepared q, k, beta, g in `area` (written by prepare_inputs).
void use_prepared(Params& p, uint8_t* area) {
    const long long th = (long long)p.B * p.T * p.H;
    const size_t s = p.io_dtype == DR_F32 ? 4 : 2;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    uint8_t* kn = area + al(th * p.dk * s);
    float* bn = reinterpret_cast<float*>(kn + al(th * p.dk * s));
    p.q = area;
    p.k = kn;
    p.beta = bn;
    if (gate_count(p)) p.g = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bn) + al(th * 4));
}

// Writes the prepared q, k, beta, g into `area` and points p at them.
cudaError_t prepare_inputs(Params& p, uint8_t* area, cudaStream_t st) {
    const long long th = (long long)p.B * p.T * p.H;
    Params prepared = p;
    use_prepared(prepared, area);
    cudaError_t e;
    {
        TraceScope ts("prepare_rows", st);
        void* qn = const_cast<void*>(prepared.q);
        void* kn = const_cast<void*>(prepared.k);
        e = p.io_dtype == DR_F32 ? normalize_dk<float>(p, qn, kn, th, st)
                                 : normalize_dk<__nv_bfloat16>(p, qn, kn, th, st);
    }
    if (e != cudaSuccess) return e;
    {
        TraceScope ts("prepare_gates", st);
        e = launch_gates(p, p.beta, p.g, const_cast<float*>(prepared.beta),
                         const_cast<float*>(prepared.g), false, st);
    }
    if (e != cudaSuccess) return e;
    p = prepared;
    return cudaSuccess;
}

// p holds the caller's raw q, k, beta, g and its gradient buffers (already written by the
// path's backward for the prepared tensors).
cudaError_t chain_prepared_grads(const Params& p, cudaStream_t st) {
    const long long th = (long long)p.B * p.T * p.H;
    cudaError_t e;
    {
        TraceScope ts("chain_rows", st);
        const bool gi = p.io_dtype == DR_F32, gg = p.grad_dtype == DR_F32;
        e = gi ? (gg ? chain_dk<float, float>(p, th, st) : chain_dk<float, __nv_bfloat16>(p, th, st))
               : (gg ? chain_dk<__nv_bfloat16, float>(p, th, st)
                     : chain_dk<__nv_bfloat16, __nv_bfloat16>(p, th, st));
    }
    if (e != cudaSuccess) return e;
    {
        TraceScope ts("chain_gates", st);
        e = launch_gates(p, p.beta, p.g, p.dbeta, p.dg, true, st);
    }
    return e;
}

}  // namespace dr
