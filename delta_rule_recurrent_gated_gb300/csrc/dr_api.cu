// dr_api.cu -- the C ABI of libdr.so (declared in include/dr.h): argument
// validation, workspace sizing, the packed-sequence chunk plan, and dispatch
// to the bf16 tensor-core path (tc_*.cu) or the fp32 CUDA-core path (simt.cu).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "dr.h"

namespace dr {
size_t simt_workspace_bytes(int units, int num_chunks, int H, int dk, int dv, int C);
cudaError_t simt_fwd(const Params& p, cudaStream_t st);
cudaError_t simt_bwd(const Params& p, cudaStream_t st);
size_t tc_workspace_bytes(const Params& p);
cudaError_t tc_fwd(const Params& p, cudaStream_t st, bool write_o);
cudaError_t tc_bwd(const Params& p, cudaStream_t st, bool reuse);
cudaError_t state_passthrough(const float* src, float* dst, size_t n, cudaStream_t st);
int simt_noalloc_max_units(int C, int dk, int dv);
cudaError_t simt_fwd_noalloc(const Params& p, cudaStream_t st);
cudaError_t decode(const Params& p, float* state, cudaStream_t st, bool prepare);
size_t prepare_bytes(const Params& p);
cudaError_t prepare_inputs(Params& p, uint8_t* area, cudaStream_t st);
void use_prepared(Params& p, uint8_t* area);
cudaError_t chain_prepared_grads(const Params& p, cudaStream_t st);
size_t gdn2_workspace_bytes(int units, int num_chunks, int H, int dk, int dv, long long th);
cudaError_t gdn2_fwd(const Params& p, cudaStream_t st);
cudaError_t gdn2_bwd(const Params& p, cudaStream_t st, bool reuse);
cudaError_t wait_selftest(int* err, int arrive, unsigned long long limit_ns, cudaStream_t st);
}  // namespace dr

using dr::Params;

namespace {

constexpr size_t kHeader = 256;  // error word + padding at the start of the workspace

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

enum class Path { kNone, kTensor, kSimt, kGdn2 };

// Structural validity (DR_ERR_INVALID_ARG) and support (DR_ERR_UNSUPPORTED).
int check_desc(const dr_desc* d, Path* path) {
    if (!d) return DR_ERR_INVALID_ARG;
    if (d->B < 0 || d->T < 0 || d->H < 1 || d->d_k < 1 || d->d_v < 1 || d->chunk < 1)
        return DR_ERR_INVALID_ARG;
    if (d->variant < DR_DELTANET || d->variant > DR_GDN2) return DR_ERR_INVALID_ARG;
    for (int t : {d->io_dtype, d->out_dtype, d->grad_dtype})
        if (t != DR_BF16 && t != DR_F32) return DR_ERR_INVALID_ARG;
    if (!std::isfinite(d->scale)) return DR_ERR_INVALID_ARG;
    if (d->flags & ~(DR_FLAG_REUSE_FWD | DR_FLAG_PREPARE_INPUTS)) return DR_ERR_INVALID_ARG;
    if ((long long)d->B * d->T * d->H * (d->d_k > d->d_v ? d->d_k : d->d_v) >= (1ll << 40))
        return DR_ERR_INVALID_ARG;
    if (d->cu_seqlens) {
        if (d->B != 1 || d->num_seqs < 0 || d->num_chunks < 0) return DR_ERR_INVALID_ARG;
        if (d->num_seqs > 0 && !d->chunk_offsets) return DR_ERR_INVALID_ARG;
        if (d->num_chunks > 0 && !d->chunk_table) return DR_ERR_INVALID_ARG;
    } else {
        if (d->num_seqs != d->B) return DR_ERR_INVALID_ARG;
        if (d->chunk_table || d->chunk_offsets) return DR_ERR_INVALID_ARG;
    }
    *path = Path::kNone;
    auto small = [](int x) { return x == 16 || x == 32 || x == 64; };
    if (d->variant == DR_GDN2) {
        if (d->flags & DR_FLAG_PREPARE_INPUTS) return DR_ERR_UNSUPPORTED;
        if (small(d->d_k) && small(d->d_v) && small(d->chunk)) *path = Path::kGdn2;
        return *path == Path::kNone ? DR_ERR_UNSUPPORTED : DR_OK;
    }
    if (d->io_dtype == DR_BF16) {
        if (d->d_k == d->d_v && (d->d_k == 64 || d->d_k == 128) && d->chunk == 64)
            *path = Path::kTensor;
    } else {
        auto dim = [&](int x) { return small(x) || x == 128; };
        if (dim(d->d_k) && dim(d->d_v) && small(d->chunk)) *path = Path::kSimt;
    }
    return *path == Path::kNone ? DR_ERR_UNSUPPORTED : DR_OK;
}

Params make_params(const dr_desc* d) {
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.B = d->B; p.T = d->T; p.H = d->H; p.dk = d->d_k; p.dv = d->d_v; p.C = d->chunk;
    p.variant = d->variant; p.io_dtype = d->io_dtype; p.out_dtype = d->out_dtype;
    p.grad_dtype = d->grad_dtype; p.scale = d->scale;
    if (d->cu_seqlens) {
        p.N = d->num_seqs;
        p.num_chunks = d->num_chunks;
        p.chunks_per_seq = 0;
        p.cu = d->cu_seqlens; p.ctab = d->chunk_table; p.coff = d->chunk_offsets;
    } else {
        p.N = d->B;
        p.chunks_per_seq = (d->T + d->chunk - 1) / d->chunk;
        p.num_chunks = p.N * p.chunks_per_seq;
    }
    return p;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The path's own workspace: header, then the path's residuals and scratch.
size_t path_ws_bytes(const Params& p, Path path) {
    if (path == Path::kGdn2)
        return kHeader + dr::gdn2_workspace_bytes(p.N * p.H, p.num_chunks, p.H, p.dk, p.dv,
                                                  (long long)p.B * p.T * p.H);
    if (path == Path::kSimt)
        return kHeader + dr::simt_workspace_bytes(p.N * p.H, p.num_chunks, p.H, p.dk, p.dv, p.C);
    return kHeader + dr::tc_workspace_bytes(p);
}

// With DR_FLAG_PREPARE_INPUTS on the fp32 CUDA-core path the prepared q, k, beta, g
// follow the path's area; the tensor-core kernels prepare their inputs on the fly.
size_t ws_bytes(const Params& p, Path path, int flags) {
    if (path == Path::kTensor) {  // with preparation the tensor-core path keeps the row norms
        Params q = p;
        q.prepare = (flags & DR_FLAG_PREPARE_INPUTS) ? 1 : 0;
        return path_ws_bytes(q, path);
    }
    const size_t base = path_ws_bytes(p, path);
    if (!(flags & DR_FLAG_PREPARE_INPUTS)) return base;
    return align256(base) + dr::prepare_bytes(p);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DR_OK : DR_ERR_CUDA; }

}  // namespace

extern "C" {

const char* dr_error_string(int code) {
    switch (code) {
        case DR_OK: return "DR_OK";
        case DR_ERR_INVALID_ARG: return "DR_ERR_INVALID_ARG: invalid argument";
        case DR_ERR_UNSUPPORTED: return "DR_ERR_UNSUPPORTED: outside the supported set";
        case DR_ERR_WORKSPACE: return "DR_ERR_WORKSPACE: workspace missing or too small";
        case DR_ERR_ALIGNMENT: return "DR_ERR_ALIGNMENT: pointer not 16-byte aligned";
        case DR_ERR_CUDA: return "DR_ERR_CUDA: CUDA launch or runtime failure";
        case DR_ERR_TIMEOUT: return "DR_ERR_TIMEOUT: a bounded device wait ran out";
        case DR_ERR_SCRATCH_LIMIT:
            return "DR_ERR_SCRATCH_LIMIT: problem larger than the library's static scratch "
                   "(dr_fwd_noalloc)";
        default: return "unknown dr status code";
    }
}

size_t dr_workspace_bytes(const dr_desc* desc) {
    Path path;
    if (check_desc(desc, &path) != DR_OK) return 0;
    return ws_bytes(make_params(desc), path, desc->flags);
}

int dr_plan_varlen(const int32_t* cu, int num_seqs, int chunk, int32_t* table, int32_t* offsets,
                   int max_chunks, int* num_chunks) {
    if (!cu || num_seqs < 0 || chunk < 1 || !num_chunks) return DR_ERR_INVALID_ARG;
    if (cu[0] != 0) return DR_ERR_INVALID_ARG;
    long long total = 0;
    for (int n = 0; n < num_seqs; ++n) {
        const long long len = (long long)cu[n + 1] - cu[n];
        if (len < 0) return DR_ERR_INVALID_ARG;
        total += (len + chunk - 1) / chunk;
    }
    if (total > 0x7fffffffll) return DR_ERR_INVALID_ARG;
    *num_chunks = (int)total;
    if (!table && !offsets) return DR_OK;
    if (total > max_chunks) return DR_ERR_INVALID_ARG;
    int c = 0;
    for (int n = 0; n < num_seqs; ++n) {
        if (offsets) offsets[n] = c;
        for (int32_t t = cu[n]; t < cu[n + 1]; t += chunk, ++c) {
            if (table) { table[2 * c] = n; table[2 * c + 1] = t; }
        }
    }
    if (offsets) offsets[num_seqs] = c;
    return DR_OK;
}

}  // extern "C"

namespace {

int fwd_impl(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
             const float* g, const float* h0, void* o, float* hT, void* u, void* ws,
             size_t ws_size, void* stream) {
    Path path;
    int rc = check_desc(desc, &path);
    if (rc != DR_OK) return rc;
    if (path == Path::kGdn2) return DR_ERR_INVALID_ARG;  // its gates go through dr_gdn2_fwd
    Params p = make_params(desc);
    const long long tokens = (long long)p.B * p.T;
    if (tokens > 0 && (!q || !k || !v || !beta || !o)) return DR_ERR_INVALID_ARG;
    if (tokens > 0 && ((p.variant == DR_DELTANET) != (g == nullptr))) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, beta, g, h0, o, hT, u, ws};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    const size_t need = ws_bytes(p, path, desc->flags);
    if (!ws || ws_size < need) return DR_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.o = o; p.hT = hT;
    p.u = u;
    p.ws = static_cast<uint8_t*>(ws);
    p.err = static_cast<int*>(ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return DR_ERR_CUDA;
    if (tokens == 0) {
        if (hT) return cuda_status(dr::state_passthrough(h0, hT, (size_t)p.N * p.H * p.dk * p.dv, st));
        return DR_OK;
    }
    if (desc->flags & DR_FLAG_PREPARE_INPUTS) {
        if (path == Path::kTensor) {
            p.prepare = 1;  // the tensor-core kernels normalise and map on the fly
        } else {
            cudaError_t e = dr::prepare_inputs(p, p.ws + align256(path_ws_bytes(p, path)), st);
            if (e != cudaSuccess) return DR_ERR_CUDA;
        }
    }
    if (path == Path::kSimt) return cuda_status(dr::simt_fwd(p, st));
    return cuda_status(dr::tc_fwd(p, st, true));
}

int bwd_impl(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
             const float* g, const float* h0, const void* dO, const float* dhT, const void* dU,
             void* dq, void* dk, void* dv, float* dbeta, float* dg, float* dh0, void* ws,
             size_t ws_size, void* stream) {
    Path path;
    int rc = check_desc(desc, &path);
    if (rc != DR_OK) return rc;
    if (path == Path::kGdn2) return DR_ERR_INVALID_ARG;  // its gates go through dr_gdn2_bwd
    Params p = make_params(desc);
    const long long tokens = (long long)p.B * p.T;
    if (tokens > 0 && (!q || !k || !v || !beta || !dO || !dq || !dk || !dv || !dbeta))
        return DR_ERR_INVALID_ARG;
    if (tokens > 0 && ((p.variant == DR_DELTANET) != (g == nullptr))) return DR_ERR_INVALID_ARG;
    if (tokens > 0 && ((p.variant == DR_DELTANET) != (dg == nullptr))) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, beta, g, h0, dO, dhT, dU, dq, dk, dv, dbeta, dg, dh0, ws};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    const size_t need = ws_bytes(p, path, desc->flags);
    if (!ws || ws_size < need) return DR_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0;
    p.dO = dO; p.dhT = dhT; p.dU = dU; p.dq = dq; p.dk_ = dk; p.dv_ = dv; p.dbeta = dbeta; p.dg = dg;
    p.dh0 = dh0;
    p.ws = static_cast<uint8_t*>(ws);
    p.err = static_cast<int*>(ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return DR_ERR_CUDA;
    if (tokens == 0) {
        if (dh0) return cuda_status(dr::state_passthrough(dhT, dh0, (size_t)p.N * p.H * p.dk * p.dv, st));
        return DR_OK;
    }
    const bool reuse = (desc->flags & DR_FLAG_REUSE_FWD) != 0;
    if ((desc->flags & DR_FLAG_PREPARE_INPUTS) && path == Path::kTensor) {
        // the tensor-core kernels normalise and map the raw inputs on the fly and chain
        // their gradients back to them before writing
        p.prepare = 1;
        return cuda_status(dr::tc_bwd(p, st, reuse));
    }
    const bool prepare = (desc->flags & DR_FLAG_PREPARE_INPUTS) != 0;
    Params raw = p;
    if (prepare) {
        // the path runs on the prepared tensors, then its gradients are chained back
        // to the raw ones in place; with DR_FLAG_REUSE_FWD the forward's prepared
        // tensors are still in the workspace
        uint8_t* area = p.ws + align256(path_ws_bytes(p, path));
        if (reuse) {
            dr::use_prepared(p, area);
        } else {
            cudaError_t e = dr::prepare_inputs(p, area, st);
            if (e != cudaSuccess) return DR_ERR_CUDA;
        }
    }
    cudaError_t e = path == Path::kSimt ? dr::simt_bwd(p, st) : dr::tc_bwd(p, st, reuse);
    if (e != cudaSuccess) return DR_ERR_CUDA;
    if (prepare) return cuda_status(dr::chain_prepared_grads(raw, st));
    return DR_OK;
}

}  // namespace

extern "C" {

int dr_fwd(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
           const float* g, const float* h0, void* o, float* hT, void* ws, size_t ws_size,
           void* stream) {
    return fwd_impl(desc, q, k, v, beta, g, h0, o, hT, nullptr, ws, ws_size, stream);
}

int dr_fwd_u(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
             const float* g, const float* h0, void* o, float* hT, void* u, void* ws,
             size_t ws_size, void* stream) {
    return fwd_impl(desc, q, k, v, beta, g, h0, o, hT, u, ws, ws_size, stream);
}

int dr_bwd(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
           const float* g, const float* h0, const void* dO, const float* dhT, void* dq, void* dk,
           void* dv, float* dbeta, float* dg, float* dh0, void* ws, size_t ws_size,
           void* stream) {
    return bwd_impl(desc, q, k, v, beta, g, h0, dO, dhT, nullptr, dq, dk, dv, dbeta, dg, dh0, ws,
                    ws_size, stream);
}

int dr_bwd_u(const dr_desc* desc, const void* q, const void* k, const void* v, const float* beta,
             const float* g, const float* h0, const void* dO, const float* dhT, const void* dU,
             void* dq, void* dk, void* dv, float* dbeta, float* dg, float* dh0, void* ws,
             size_t ws_size, void* stream) {
    return bwd_impl(desc, q, k, v, beta, g, h0, dO, dhT, dU, dq, dk, dv, dbeta, dg, dh0, ws,
                    ws_size, stream);
}

namespace {
// Host checks shared by dr_decode and dr_gdn2_decode (sizes, layout, flags, state).
int check_decode(const dr_desc& d, const float* state) {
    if (d.B < 0 || d.T < 0 || d.H < 1 || d.d_k < 1 || d.d_v < 1 || d.chunk < 1)
        return DR_ERR_INVALID_ARG;
    for (int t : {d.io_dtype, d.out_dtype})
        if (t != DR_BF16 && t != DR_F32) return DR_ERR_INVALID_ARG;
    if (!std::isfinite(d.scale)) return DR_ERR_INVALID_ARG;
    if (d.flags & ~(DR_FLAG_REUSE_FWD | DR_FLAG_PREPARE_INPUTS)) return DR_ERR_INVALID_ARG;
    if (d.cu_seqlens || d.chunk_table || d.chunk_offsets || d.num_seqs != d.B)
        return DR_ERR_INVALID_ARG;
    if ((long long)d.B * d.T * d.H * (d.d_k > d.d_v ? d.d_k : d.d_v) >= (1ll << 40))
        return DR_ERR_INVALID_ARG;
    auto size_ok = [](int x) { return x == 16 || x == 32 || x == 64 || x == 128; };
    if (!size_ok(d.d_k) || !size_ok(d.d_v)) return DR_ERR_UNSUPPORTED;
    if (d.B > 0 && !state) return DR_ERR_INVALID_ARG;
    return DR_OK;
}
}  // namespace

int dr_gdn2_decode(const dr_desc* desc, const void* q, const void* k, const void* v,
                   const float* erase, const float* write, const float* g, float* state,
                   void* o, void* stream) {
    if (!desc) return DR_ERR_INVALID_ARG;
    const dr_desc& d = *desc;
    if (d.variant != DR_GDN2) return DR_ERR_INVALID_ARG;
    int rc = check_decode(d, state);
    if (rc != DR_OK) return rc;
    if (d.flags & DR_FLAG_PREPARE_INPUTS) return DR_ERR_UNSUPPORTED;
    const long long tokens = (long long)d.B * d.T;
    if (tokens > 0 && (!q || !k || !v || !erase || !write || !g || !o)) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, erase, write, g, state, o};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    Params p = make_params(desc);
    p.q = q; p.k = k; p.v = v; p.erase = erase; p.write = write; p.g = g; p.o = o;
    return cuda_status(dr::decode(p, state, static_cast<cudaStream_t>(stream), false));
}

int dr_decode(const dr_desc* desc, const void* q, const void* k, const void* v,
              const float* beta, const float* g, float* state, void* o, void* stream) {
    if (!desc) return DR_ERR_INVALID_ARG;
    const dr_desc& d = *desc;
    if (d.variant < DR_DELTANET || d.variant > DR_KDA) return DR_ERR_INVALID_ARG;
    int rc = check_decode(d, state);
    if (rc != DR_OK) return rc;
    const long long tokens = (long long)d.B * d.T;
    if (tokens > 0 && (!q || !k || !v || !beta || !o)) return DR_ERR_INVALID_ARG;
    if (tokens > 0 && ((d.variant == DR_DELTANET) != (g == nullptr))) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, beta, g, state, o};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    Params p = make_params(desc);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.o = o;
    return cuda_status(dr::decode(p, state, static_cast<cudaStream_t>(stream),
                                  (d.flags & DR_FLAG_PREPARE_INPUTS) != 0));
}

int dr_fwd_noalloc(const dr_desc* desc, const void* q, const void* k, const void* v,
                   const float* beta, const float* g, const float* h0, void* o, float* hT,
                   void* stream) {
    Path path;
    int rc = check_desc(desc, &path);
    if (rc != DR_OK) return rc;
    if (path != Path::kSimt || (desc->flags & DR_FLAG_PREPARE_INPUTS)) return DR_ERR_UNSUPPORTED;
    Params p = make_params(desc);
    const long long tokens = (long long)p.B * p.T;
    if (tokens > 0 && (!q || !k || !v || !beta || !o)) return DR_ERR_INVALID_ARG;
    if (tokens > 0 && ((p.variant == DR_DELTANET) != (g == nullptr))) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, beta, g, h0, o, hT};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    if ((long long)p.N * p.H > dr::simt_noalloc_max_units(p.C, p.dk, p.dv)) return DR_ERR_SCRATCH_LIMIT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.o = o; p.hT = hT;
    if (tokens == 0) {
        if (hT) return cuda_status(dr::state_passthrough(h0, hT, (size_t)p.N * p.H * p.dk * p.dv, st));
        return DR_OK;
    }
    return cuda_status(dr::simt_fwd_noalloc(p, st));
}

int dr_gdn2_fwd(const dr_desc* desc, const void* q, const void* k, const void* v,
                const float* erase, const float* write, const float* g, const float* h0, void* o,
                float* hT, void* ws, size_t ws_size, void* stream) {
    Path path;
    int rc = check_desc(desc, &path);
    if (rc != DR_OK) return rc;
    if (path != Path::kGdn2) return DR_ERR_INVALID_ARG;
    Params p = make_params(desc);
    const long long tokens = (long long)p.B * p.T;
    if (tokens > 0 && (!q || !k || !v || !erase || !write || !g || !o)) return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, erase, write, g, h0, o, hT, ws};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    const size_t need = ws_bytes(p, path, desc->flags);
    if (!ws || ws_size < need) return DR_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.q = q; p.k = k; p.v = v; p.erase = erase; p.write = write; p.g = g; p.h0 = h0;
    p.o = o; p.hT = hT;
    p.ws = static_cast<uint8_t*>(ws);
    p.err = static_cast<int*>(ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return DR_ERR_CUDA;
    if (tokens == 0) {
        if (hT) return cuda_status(dr::state_passthrough(h0, hT, (size_t)p.N * p.H * p.dk * p.dv, st));
        return DR_OK;
    }
    return cuda_status(dr::gdn2_fwd(p, st));
}

int dr_gdn2_bwd(const dr_desc* desc, const void* q, const void* k, const void* v,
                const float* erase, const float* write, const float* g, const float* h0,
                const void* dO, const float* dhT, void* dq, void* dk, void* dv, float* derase,
                float* dwrite, float* dg, float* dh0, void* ws, size_t ws_size, void* stream) {
    Path path;
    int rc = check_desc(desc, &path);
    if (rc != DR_OK) return rc;
    if (path != Path::kGdn2) return DR_ERR_INVALID_ARG;
    Params p = make_params(desc);
    const long long tokens = (long long)p.B * p.T;
    if (tokens > 0 && (!q || !k || !v || !erase || !write || !g || !dO || !dq || !dk || !dv ||
                       !derase || !dwrite || !dg))
        return DR_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, erase, write, g, h0, dO, dhT, dq, dk, dv, derase, dwrite, dg,
                          dh0, ws};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DR_ERR_ALIGNMENT;
    const size_t need = ws_bytes(p, path, desc->flags);
    if (!ws || ws_size < need) return DR_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.q = q; p.k = k; p.v = v; p.erase = erase; p.write = write; p.g = g; p.h0 = h0;
    p.dO = dO; p.dhT = dhT; p.dq = dq; p.dk_ = dk; p.dv_ = dv; p.derase = derase;
    p.dwrite = dwrite; p.dg = dg; p.dh0 = dh0;
    p.ws = static_cast<uint8_t*>(ws);
    p.err = static_cast<int*>(ws);
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return DR_ERR_CUDA;
    if (tokens == 0) {
        if (dh0) return cuda_status(dr::state_passthrough(dhT, dh0, (size_t)p.N * p.H * p.dk * p.dv, st));
        return DR_OK;
    }
    return cuda_status(dr::gdn2_bwd(p, st, (desc->flags & DR_FLAG_REUSE_FWD) != 0));
}

int dr_selftest_wait(void* ws, int arrive, long long limit_ns, void* stream) {
    if (!ws || !aligned16(ws) || limit_ns < 0 || limit_ns > 100000000ll) return DR_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return DR_ERR_CUDA;
    return cuda_status(dr::wait_selftest(static_cast<int*>(ws), arrive ? 1 : 0,
                                         (unsigned long long)limit_ns, st));
}

int dr_check_status(const void* ws, void* stream) {
    if (!ws) return DR_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return DR_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DR_ERR_CUDA;
    return word == 0 ? DR_OK : DR_ERR_TIMEOUT;
}

}  // extern "C"
