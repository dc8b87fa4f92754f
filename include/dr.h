/*
 * dr.h -- C ABI of libdr.so: chunkwise-parallel forward and backward of the
 * delta-rule recurrent memory (DeltaNet, Gated DeltaNet, Kimi Delta Attention)
 * on one GB300 GPU (sm_103a).
 *
 * The operation (page "Linear Attention Architectures: Mechanisms, Trade-offs,
 * and Cross-Layer Routing", section "Metodologia y Marco de Trabajo", item 1,
 * the unified recurrent-memory notation and its three variant bullets): per
 * (sequence, head) a memory matrix W (d_v x d_k) is, token by token,
 *   decayed   Wd_t = W_{t-1} diag(a_t)       a_t = 1 (DeltaNet), exp(g_t) * 1 (Gated
 *                                            DeltaNet, one scalar gate), exp(g_t) per
 *                                            key channel (Kimi Delta Attention)
 *   corrected r_t  = v_t - Wd_t k_t          (the delta-rule residual r = v - vbar)
 *   written   W_t  = Wd_t + beta_t r_t k_t^T
 *   read      o_t  = scale * W_t q_t
 * The gate enters as its logarithm g = log(alpha) <= 0.  beta_t, the read after
 * the write and `scale` are the standard delta-rule reading of that notation.
 * Also here: the recurrent step for inference (dr_decode), the emitted write
 * u = beta r with its gradient (dr_fwd_u / dr_bwd_u), input preparation inside the
 * library (DR_FLAG_PREPARE_INPUTS), and Gated DeltaNet-2, the fourth variant of the
 * same section (dr_gdn2_*, separate erase and write gates; its equations are a
 * reading, stated at its entry points).
 *
 * Memory: the caller allocates every buffer (device memory unless stated) and
 * the workspace; the library never allocates, frees or synchronises inside
 * dr_fwd / dr_bwd.  All work is enqueued on `stream` (a cudaStream_t passed as
 * void*, NULL = legacy default stream) in stream order.  Calls are re-entrant;
 * two calls that run concurrently must not share a workspace.
 *
 * Layouts (row-major, contiguous, every pointer 16-byte aligned):
 *   q, k, dq, dk   [B, T, H, d_k]       io dtype (grad dtype for dq, dk)
 *   v, dO, dv      [B, T, H, d_v]       io dtype (grad dtype for dv)
 *   o              [B, T, H, d_v]       out dtype
 *   beta, dbeta    [B, T, H]            fp32, beta in [0, 1]
 *   g, dg          Gated DeltaNet [B, T, H]; KDA [B, T, H, d_k]; fp32; NULL for DeltaNet
 *   h0, hT, dhT, dh0  [N, H, d_k, d_v]  fp32, the state S = W^T (d_v contiguous)
 * N = B for dense batches.  For packed ragged sequences B == 1, T is the total
 * length and cu_seqlens (N + 1 offsets) splits the T axis; every sequence
 * starts from its own h0[n] (zero when h0 is NULL) and ends in hT[n].
 *
 * Errors: every entry point returns a dr_status_code.  When the host detects
 * an error nothing is launched and no output is touched.  A launch failure is
 * DR_ERR_CUDA.  Device-side waits are bounded: a wait that runs out records
 * DR_ERR_TIMEOUT in the workspace, which dr_check_status reports.
 */
#ifndef DR_H
#define DR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum dr_status_code {
    DR_OK = 0,
    DR_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, bad cu_seqlens */
    DR_ERR_UNSUPPORTED = 2,   /* valid but outside the supported set (below)         */
    DR_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than dr_workspace_bytes   */
    DR_ERR_ALIGNMENT = 4,     /* a pointer is not 16-byte aligned                    */
    DR_ERR_CUDA = 5,          /* a CUDA call or launch failed                        */
    DR_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out                  */
    DR_ERR_SCRATCH_LIMIT = 7  /* dr_fwd_noalloc: problem larger than its static scratch */
};

enum dr_variant { DR_DELTANET = 0, DR_GDN = 1, DR_KDA = 2, DR_GDN2 = 3 /* dr_gdn2_* only */ };
enum dr_dtype { DR_BF16 = 0, DR_F32 = 1 };

/* dr_desc.flags */
#define DR_FLAG_REUSE_FWD 1  /* dr_bwd: the workspace still holds the residuals
                                written by dr_fwd for the same desc and inputs;
                                skip their recomputation */
/*
 * DR_FLAG_PREPARE_INPUTS: q, k, beta and g arrive as the projections produce them,
 * and the library applies the input maps of these layers itself.  The pages give
 * the recurrence on prepared inputs only (q, k unit-norm keys, beta in [0, 1],
 * g = log alpha <= 0); the maps below are the standard ones the workloads use to
 * produce them (q, k L2-normalised per head, beta through a sigmoid, log alpha
 * through -softplus), with eps = 1e-6 guarding the zero vector:
 *   q_hat = q * rsqrt(sum_c q_c^2 + 1e-6)   per (token, head); the same for k
 *   beta  = sigmoid(b)                       b: the beta argument, a logit
 *   g     = -softplus(x) = -log(1 + e^x)     x: the g argument (GDN, KDA)
 * dr_bwd / dr_bwd_u take the same raw tensors and return gradients with respect to
 * them (dq, dk, dbeta, dg chained through the three maps).  On the bf16 tensor-core
 * path the kernels apply the maps on the fly, in fp32, to the raw tiles they load
 * (forward and backward alike; the prepared values are never stored, only the two
 * inverse row norms per token and head, 8 bytes, which dr_workspace_bytes counts and
 * the backward reads back) and chain the gradients before writing them.  On the fp32 CUDA-core path dr_fwd / dr_fwd_u write
 * q_hat, k_hat (io_dtype), beta and g (fp32) into the workspace (dr_workspace_bytes
 * counts them) and run on those; with DR_FLAG_REUSE_FWD the backward reuses them (the
 * same raw inputs must be passed).  dr_decode applies the maps in its own kernel.
 * dr_fwd_noalloc does not take the flag (DR_ERR_UNSUPPORTED).
 */
#define DR_FLAG_PREPARE_INPUTS 2

/*
 * Problem descriptor.  Supported set:
 *   io bf16: d_k = d_v in {64, 128}, chunk = 64  (tensor-core path)
 *   io fp32: d_k, d_v in {16, 32, 64, 128}, chunk in {16, 32, 64}  (fp32 CUDA-core path)
 *   any T >= 0 (a partial last chunk is fine), B >= 0, H >= 1.
 */
typedef struct dr_desc {
    int B, T, H;
    int d_k, d_v;
    int chunk;                    /* tokens per chunk of the chunkwise form            */
    int variant;                  /* enum dr_variant                                   */
    int io_dtype;                 /* q, k, v, dO                                       */
    int out_dtype;                /* o                                                 */
    int grad_dtype;               /* dq, dk, dv                                        */
    float scale;                  /* read scale (1.0 = the plain read o = W q)         */
    int flags;                    /* DR_FLAG_*                                          */
    int num_seqs;                 /* N: B for dense batches, or the packed count       */
    const int32_t* cu_seqlens;    /* device [N+1] or NULL (dense)                      */
    const int32_t* chunk_table;   /* device [num_chunks][2] = (sequence, first token),
                                     from dr_plan_varlen; NULL for dense batches      */
    const int32_t* chunk_offsets; /* device [N+1]: first chunk of each sequence        */
    int num_chunks;               /* total chunks (packed layout only)                 */
} dr_desc;

/* Bytes of workspace dr_fwd and dr_bwd need for `desc` (the same for both).
   Returns 0 when desc is invalid or unsupported. */
size_t dr_workspace_bytes(const dr_desc* desc);

/*
 * Host-side chunk plan of packed ragged sequences (no GPU work).
 * cu_seqlens_host: N + 1 non-decreasing offsets starting at 0.  Writes, for
 * every chunk of every sequence in order, (sequence, first token) into
 * chunk_table_host[2*i], [2*i+1] (chunks never straddle a sequence boundary;
 * the last chunk of a sequence may be short; an empty sequence has none), and
 * the index of each sequence's first chunk into chunk_offsets_host[0..N]
 * (chunk_offsets_host[N] = total).  *num_chunks receives the total; when it
 * exceeds max_chunks nothing is written and DR_ERR_INVALID_ARG is returned.
 * chunk_table_host / chunk_offsets_host may be NULL to query the count only.
 */
int dr_plan_varlen(const int32_t* cu_seqlens_host, int num_seqs, int chunk,
                   int32_t* chunk_table_host, int32_t* chunk_offsets_host, int max_chunks,
                   int* num_chunks);

/*
 * Forward: o (and hT when non-NULL) from q, k, v, beta, g, h0 (h0 NULL = zero
 * state).  Also leaves in the workspace the residuals dr_bwd can reuse
 * (DR_FLAG_REUSE_FWD).
 */
int dr_fwd(const dr_desc* desc, const void* q, const void* k, const void* v,
           const float* beta, const float* g, const float* h0, void* o, float* hT,
           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: gradients of L = sum(dO * o) + sum(dhT * hT) with respect to q, k,
 * v, beta, g (the log-gate) and h0.  dhT NULL means a zero final-state
 * gradient; dh0 may be NULL when not needed; dg must be NULL for DeltaNet and
 * non-NULL otherwise.  Gradients are with respect to the tensors as passed
 * (q, k already normalised, beta after its sigmoid, g = log alpha; with
 * DR_FLAG_PREPARE_INPUTS the raw tensors before those maps).
 */
int dr_bwd(const dr_desc* desc, const void* q, const void* k, const void* v,
           const float* beta, const float* g, const float* h0, const void* dO,
           const float* dhT, void* dq, void* dk, void* dv, float* dbeta, float* dg,
           float* dh0, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The write of every token, for routing it to another layer ("Linear Attention
 * Architectures: Mechanisms, Trade-offs, and Cross-Layer Routing", section
 * "Metodologia y Marco de Trabajo", item 3, CLER: the delta-rule write error of a
 * layer is forwarded to the next one).
 * dr_fwd_u is dr_fwd that also writes u_t = beta_t r_t, r_t = v_t - (decayed W) k_t
 * (the write the recurrence adds to the memory), to u: [B][T][H][d_v] in out_dtype
 * (packed layout as o), or nothing when u is NULL.
 * dr_bwd_u is dr_bwd for L = sum(dO * o) + sum(dhT * hT) + sum(dU * u): dU has the
 * layout of u in io_dtype; NULL means zero (dr_bwd).  With DR_FLAG_REUSE_FWD the
 * workspace may come from dr_fwd or dr_fwd_u.
 * Same supported set, ownership and errors as dr_fwd / dr_bwd (u and dU 16-byte
 * aligned).
 */
int dr_fwd_u(const dr_desc* desc, const void* q, const void* k, const void* v,
             const float* beta, const float* g, const float* h0, void* o, float* hT,
             void* u, void* workspace, size_t workspace_bytes, void* stream);
int dr_bwd_u(const dr_desc* desc, const void* q, const void* k, const void* v,
             const float* beta, const float* g, const float* h0, const void* dO,
             const float* dhT, const void* dU, void* dq, void* dk, void* dv, float* dbeta,
             float* dg, float* dh0, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward for callers that cannot allocate device memory.  The paper has no
 * counterpart; this is an interface convenience of the library.
 *
 * Some callers cannot call cudaMalloc where they run this layer (a plugin
 * handed only its input and output buffers by its host framework, or code
 * that must not trigger an allocation and the device synchronisation it may
 * bring).  dr_fwd_noalloc computes the same o and hT as dr_fwd, with the
 * fp32 CUDA-core kernel (io fp32 only; the supported set of dr_fwd for fp32
 * inputs), but takes no workspace: its scratch is a 16 MiB array that the
 * library keeps in the global memory of every GPU that loads it, for the life
 * of the process.  It allocates nothing itself.
 *   - Size limit: N * H (sequences times heads) must not exceed 46 when d_k,
 *     d_v and chunk are at most 64, or 11 when d_k or d_v is 128; larger
 *     problems return DR_ERR_SCRATCH_LIMIT and launch nothing.
 *   - The first call on each device looks up the array's device address with
 *     that device current (a runtime symbol query); make that first call
 *     before any stream capture on the device.  The address is cached per
 *     device ordinal for the rest of the process: it belongs to the device's
 *     primary context (the one the CUDA runtime uses), is not valid after a
 *     cudaDeviceReset of that device, and must not be used from another
 *     context made current on it.
 *   - Every call shares the one array: calls whose kernels can overlap on the
 *     GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller.  Contents left by an earlier call are never
 *     read before being overwritten.
 *   - It writes no workspace, so dr_bwd cannot reuse its residuals.
 * Errors as dr_fwd, plus DR_ERR_UNSUPPORTED for bf16 inputs.
 */
int dr_fwd_noalloc(const dr_desc* desc, const void* q, const void* k, const void* v,
                   const float* beta, const float* g, const float* h0, void* o, float* hT,
                   void* stream);

/*
 * Recurrent step for inference (decode): the delta-rule recurrence applied
 * token by token, without chunks, to a state that the caller keeps between
 * calls ("The Delta Rule and its gated forms", the per-token update with the
 * decay applied before the residual and the read after the write).
 *   For every sequence n < desc->B, head h and token t < desc->T in order:
 *     S~ = D_t S;  r = v_t - S~^T k_t;  S = S~ + beta_t k_t r^T;  o_t = scale S^T q_t
 *   with S = W^T and D_t = I (DeltaNet), e^{g_t} I (GDN) or diag(e^{g_t}) (KDA).
 * state: [B][H][d_k][d_v] fp32 (the layout of h0 / hT), read at entry and
 *   overwritten with the state after the last token; device memory owned by
 *   the caller, never NULL.
 * q, k: [B][T][H][d_k]; v, o: [B][T][H][d_v] in io_dtype / out_dtype;
 *   beta [B][T][H] fp32; g as for dr_fwd (NULL for DeltaNet).  Dense batches
 *   only (cu_seqlens NULL); desc->chunk is ignored (any value >= 1).
 * desc->flags: DR_FLAG_PREPARE_INPUTS (q, k normalised, beta and g mapped inside
 *   the kernel, as for dr_fwd); DR_FLAG_REUSE_FWD is ignored.
 * Supported: d_k, d_v in {16, 32, 64, 128}, io bf16 or fp32.  No workspace,
 *   nothing allocated, no device synchronisation; stream-ordered on `stream`.
 * Errors: DR_ERR_INVALID_ARG (bad desc, NULL state or input, packed layout),
 *   DR_ERR_UNSUPPORTED (sizes), DR_ERR_ALIGNMENT (pointers not 16-byte
 *   aligned), DR_ERR_CUDA (launch failure).  Nothing is launched on error.
 */
int dr_decode(const dr_desc* desc, const void* q, const void* k, const void* v,
              const float* beta, const float* g, float* state, void* o, void* stream);

/*
 * Gated DeltaNet-2: separate per-channel erase and write gates ("Linear Attention
 * Architectures: Mechanisms, Trade-offs, and Cross-Layer Routing", section "Metodologia
 * y Marco de Trabajo", item 1, the Gated DeltaNet-2 bullet, which describes it in words
 * only).  The library reads it as Gated DeltaNet's scalar decay followed by an erase
 * along the gated key channels and a write of the gated value channels:
 *   Wd_t = alpha_t W_{t-1};  p_t = Wd_t k_t;
 *   W_t  = Wd_t - p_t (erase_t . k_t)^T + (write_t . v_t) k_t^T;  o_t = scale W_t q_t
 * ("." elementwise), which is Gated DeltaNet when erase_t = write_t = beta_t.
 * desc->variant must be DR_GDN2.  Inputs as dr_fwd / dr_bwd with beta replaced by
 *   erase [B, T, H, d_k] fp32 (gate per key channel, normally in [0, 1]) and
 *   write [B, T, H, d_v] fp32 (gate per value channel, normally in [0, 1]);
 *   g [B, T, H] fp32 = log alpha, never NULL.
 * dr_gdn2_bwd returns dq, dk, dv (grad dtype), derase, dwrite, dg (fp32) and dh0
 * (optional) for L = sum(dO * o) + sum(dhT * hT).
 * Supported: d_k, d_v, chunk in {16, 32, 64}; io bf16 or fp32 (fp32 arithmetic on the
 * CUDA cores for both); dense or packed layout as dr_fwd.  dr_workspace_bytes sizes the
 * workspace (same value for both calls); dr_gdn2_fwd leaves the chunk-start states in
 * it, and dr_gdn2_bwd with DR_FLAG_REUSE_FWD reads them instead of recomputing them
 * (the same desc, inputs and workspace as the forward).  DR_FLAG_PREPARE_INPUTS is
 * DR_ERR_UNSUPPORTED.  Errors as dr_fwd / dr_bwd; dr_fwd and
 * dr_bwd refuse DR_GDN2 with DR_ERR_INVALID_ARG.
 */
int dr_gdn2_fwd(const dr_desc* desc, const void* q, const void* k, const void* v,
                const float* erase, const float* write, const float* g, const float* h0,
                void* o, float* hT, void* workspace, size_t workspace_bytes, void* stream);
int dr_gdn2_bwd(const dr_desc* desc, const void* q, const void* k, const void* v,
                const float* erase, const float* write, const float* g, const float* h0,
                const void* dO, const float* dhT, void* dq, void* dk, void* dv, float* derase,
                float* dwrite, float* dg, float* dh0, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * Recurrent step of Gated DeltaNet-2 (the update of dr_gdn2_fwd token by token, as
 * dr_decode for the other variants): for every sequence, head and token in order,
 *   S~ = e^{g_t} S;  p = S~^T k_t;  S = S~ - (erase_t . k_t) p^T + k_t (write_t . v_t)^T;
 *   o_t = scale S^T q_t
 * on the caller's fp32 state [B][H][d_k][d_v], updated in place.  desc->variant must be
 * DR_GDN2; erase [B][T][H][d_k], write [B][T][H][d_v], g [B][T][H] fp32, none NULL when
 * there are tokens.  Sizes, dtypes, layout and errors as dr_decode;
 * DR_FLAG_PREPARE_INPUTS is DR_ERR_UNSUPPORTED.
 */
int dr_gdn2_decode(const dr_desc* desc, const void* q, const void* k, const void* v,
                   const float* erase, const float* write, const float* g, float* state,
                   void* o, void* stream);

/*
 * Self-test of the device failure path (no counterpart on the pages).  Launches one
 * warp that waits, with the bounded wait every tensor-core kernel uses, on an mbarrier
 * phase that only completes when `arrive` is non-zero (the warp completes it itself);
 * a wait that runs out after limit_ns records DR_ERR_TIMEOUT in the workspace error
 * word, as the kernels do.  The workspace needs only its first 16 bytes (16-byte
 * aligned, device memory).  limit_ns in [0, 1e8].  Read the outcome with
 * dr_check_status: DR_ERR_TIMEOUT without `arrive`, DR_OK with it.  Nothing is copied
 * and no tensor memory is held, so the expired wait leaves nothing in flight.
 * Errors: DR_ERR_INVALID_ARG (NULL or misaligned workspace, limit out of range),
 * DR_ERR_CUDA (launch).
 */
int dr_selftest_wait(void* workspace, int arrive, long long limit_ns, void* stream);

/* Synchronise `stream` and report any device-side error recorded in the
   workspace by the last call that used it (DR_OK or DR_ERR_TIMEOUT), or
   DR_ERR_CUDA when the stream itself failed. */
int dr_check_status(const void* workspace, void* stream);

/*
 * Kernel-level timing.  dr_trace_enable(n) (n > 0) creates n pairs of CUDA
 * events; while enabled, each of the next n kernel launches made by dr_fwd /
 * dr_bwd is bracketed by an event pair recorded on the call's stream.
 * dr_trace_enable(0) disables tracing and destroys the events;
 * dr_trace_reset() reuses them from the first slot.  dr_trace_get(i, ...)
 * waits for launch i to finish and returns its kernel name and device
 * duration in milliseconds.  Host-global state: not for concurrent callers.
 */
int dr_trace_enable(int max_launches);
int dr_trace_count(void);
void dr_trace_reset(void);
int dr_trace_get(int index, const char** kernel_name, float* milliseconds);

/* Human-readable name of a dr_status_code. */
const char* dr_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* DR_H */
