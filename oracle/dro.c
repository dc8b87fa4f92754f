/*
 * dro.c -- sequential fp64 oracle of the delta-rule recurrent memory
 * (DeltaNet, Gated DeltaNet, Kimi Delta Attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the CPU baseline leg
 * of the benchmark do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (page "Linear Attention Architectures: Mechanisms,
 * Trade-offs, and Cross-Layer Routing", section "Metodologia y Marco de
 * Trabajo", item 1 "Notacion Unificada"): a memory matrix W (d_v x d_k) per
 * (sequence, head) that is, for every token t in order,
 *
 *   decayed       Wd_t = W_{t-1} diag(a_t)          (DeltaNet: a_t = 1;
 *                                                    Gated DeltaNet: a_t = alpha_t * 1,
 *                                                    one scalar gate, applied before the
 *                                                    residual is formed;
 *                                                    Kimi Delta Attention: a_t is a
 *                                                    vector, one decay per key channel)
 *   residual      r_t  = v_t - Wd_t k_t             (the delta-rule error "r = v - vbar")
 *   written       W_t  = Wd_t + beta_t r_t k_t^T    (write strength beta_t)
 *   read          o_t  = scale * W_t q_t            (read after the write)
 *
 * Optionally the forward also returns the write u_t = beta_t r_t, the delta-rule
 * write error scaled by its write strength (section "Metodologia y Marco de
 * Trabajo", item 3, "Enrutamiento entre Capas", CLER: the write error of one
 * layer is forwarded to the next), and the backward then accepts dL/du_t.
 *
 * The gate enters as g = log(alpha) (fp64 here), so a_t = exp(g_t).
 * The write strength beta_t, the read o = W q and the read-after-write order
 * are the standard delta-rule reading of that notation; the pages name a
 * write control and a read but print no formula for either.
 *
 * The backward pass is the reverse-time recurrence derived by hand from the
 * four lines above (chain rule through one token step, applied from t = L
 * down to 1).  With G = dL/dW_t (d_v x d_k), initialised to dL/dW_L:
 *
 *   G   += scale * dO_t q_t^T          dq_t = scale * W_t^T dO_t
 *   dr   = beta_t (G k_t + du_t)       dbeta_t = r_t . (G k_t + du_t)   dv_t = dr
 *          (du_t = dL/du_t of the emitted write, zero when it is not used)
 *   dk_t = beta_t G^T r_t - Wd_t^T dr
 *   dWd  = G - dr k_t^T
 *   dg_t[c] = a_t[c] * sum_i dWd[i][c] * W_{t-1}[i][c]   (KDA, per channel;
 *                                                          GDN: summed over c)
 *   G    = dWd diag(a_t)
 *
 * and dL/dW_0 = G at the end.  W_{t-1} is recomputed forward from
 * checkpoints stored every CKPT tokens; the decay is never inverted.
 *
 * Layouts (row-major, contiguous):
 *   q, k   [B, T, H, dk]        v, o, dO  [B, T, H, dv]
 *   beta   [B, T, H]            g: GDN [B, T, H], KDA [B, T, H, dk], DeltaNet unused
 *   h0, hT, dhT, dh0            [N, H, dk, dv]   (the state S = W^T, d_v contiguous)
 * With cu_seqlens (int32, N+1 offsets, B == 1) sequence n is tokens
 * [cu[n], cu[n+1]) of batch row 0 and starts from its own h0[n]; otherwise
 * sequence n is batch row n (N == B) of length T.
 *
 * A "unit" is one (sequence, head) pair, u = n * H + h.  A NULL unit list
 * means all N*H units; otherwise only the listed units are computed and only
 * their outputs are written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

enum { DRO_DELTANET = 0, DRO_GDN = 1, DRO_KDA = 2 };

typedef struct {
    int B, T, H, dk, dv, variant;
    double scale;
    const int32_t *cu;
    int N;
} shape_t;

/* token range and batch row of sequence n */
static void seq_range(const shape_t *s, int n, int64_t *row0, int64_t *len)
{
    if (s->cu) {
        *row0 = s->cu[n];
        *len = (int64_t)s->cu[n + 1] - s->cu[n];
    } else {
        *row0 = (int64_t)n * s->T;
        *len = s->T;
    }
}

/* a_t[c] = exp(g_t[c]) for the token at flat row `row` (= b*T + t) */
static void decay_of(const shape_t *s, const double *g, int64_t row, int h, double *a)
{
    int c;
    if (s->variant == DRO_DELTANET) {
        for (c = 0; c < s->dk; ++c) a[c] = 1.0;
    } else if (s->variant == DRO_GDN) {
        double x = exp(g[row * s->H + h]);
        for (c = 0; c < s->dk; ++c) a[c] = x;
    } else {
        const double *gr = g + (row * s->H + h) * s->dk;
        for (c = 0; c < s->dk; ++c) a[c] = exp(gr[c]);
    }
}

/* One forward token step, in place on W (dv x dk).  r receives the residual. */
static void step(const shape_t *s, double *W, const double *a, const double *kt,
                 const double *vt, double bt, double *r)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    for (i = 0; i < dv; ++i) {
        double *w = W + (int64_t)i * dk;
        double p = 0.0;
        for (c = 0; c < dk; ++c) {
            w[c] *= a[c];
            p += w[c] * kt[c];
        }
        r[i] = vt[i] - p;
    }
    for (i = 0; i < dv; ++i) {
        double *w = W + (int64_t)i * dk;
        double br = bt * r[i];
        for (c = 0; c < dk; ++c) w[c] += br * kt[c];
    }
}

static void load_state(const shape_t *s, const double *h, int n, int hd, double *W)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    if (!h) {
        memset(W, 0, sizeof(double) * dk * dv);
        return;
    }
    const double *src = h + ((int64_t)n * s->H + hd) * dk * dv;
    for (c = 0; c < dk; ++c)
        for (i = 0; i < dv; ++i) W[(int64_t)i * dk + c] = src[(int64_t)c * dv + i];
}

static void store_state(const shape_t *s, double *h, int n, int hd, const double *W)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    double *dst = h + ((int64_t)n * s->H + hd) * dk * dv;
    for (c = 0; c < dk; ++c)
        for (i = 0; i < dv; ++i) dst[(int64_t)c * dv + i] = W[(int64_t)i * dk + c];
}

static int check_shape(const shape_t *s)
{
    if (s->B < 0 || s->T < 0 || s->H <= 0 || s->dk <= 0 || s->dv <= 0) return 1;
    if (s->variant < 0 || s->variant > 2) return 1;
    if (s->cu) {
        int n;
        if (s->B != 1 || s->N < 0 || s->cu[0] != 0 || s->cu[s->N] != s->T) return 1;
        for (n = 0; n < s->N; ++n)
            if (s->cu[n + 1] < s->cu[n]) return 1;
    } else if (s->N != s->B) {
        return 1;
    }
    return 0;
}

static void fwd_unit(const shape_t *s, int u, const double *q, const double *k,
                     const double *v, const double *beta, const double *g,
                     const double *h0, double *o, double *hT, double *uw)
{
    const int dk = s->dk, dv = s->dv, H = s->H;
    const int n = u / H, hd = u % H;
    int64_t row0, len, t;
    int i, c;
    double *W = (double *)malloc(sizeof(double) * dk * dv);
    double *a = (double *)malloc(sizeof(double) * dk);
    double *r = (double *)malloc(sizeof(double) * dv);
    seq_range(s, n, &row0, &len);
    load_state(s, h0, n, hd, W);
    for (t = 0; t < len; ++t) {
        const int64_t row = row0 + t;
        const double *kt = k + (row * H + hd) * dk;
        const double *qt = q + (row * H + hd) * dk;
        const double *vt = v + (row * H + hd) * dv;
        decay_of(s, g, row, hd, a);
        step(s, W, a, kt, vt, beta[row * H + hd], r);
        if (uw) {
            double *ut = uw + (row * H + hd) * dv;
            for (i = 0; i < dv; ++i) ut[i] = beta[row * H + hd] * r[i];
        }
        if (o) {
            double *ot = o + (row * H + hd) * dv;
            for (i = 0; i < dv; ++i) {
                const double *w = W + (int64_t)i * dk;
                double acc = 0.0;
                for (c = 0; c < dk; ++c) acc += w[c] * qt[c];
                ot[i] = s->scale * acc;
            }
        }
    }
    if (hT) store_state(s, hT, n, hd, W);
    free(W);
    free(a);
    free(r);
}

static void bwd_unit(const shape_t *s, int u, const double *q, const double *k,
                     const double *v, const double *beta, const double *g,
                     const double *h0, const double *dO, const double *dhT,
                     const double *dU, double *dq, double *dkk, double *dvv, double *dbeta,
                     double *dg, double *dh0)
{
    const int dk = s->dk, dv = s->dv, H = s->H;
    const int n = u / H, hd = u % H;
    const int64_t S = (int64_t)dk * dv;
    int64_t row0, len, t, seg, nseg;
    int i, c;
    seq_range(s, n, &row0, &len);
    nseg = (len + CKPT - 1) / CKPT;

    double *ck = (double *)malloc(sizeof(double) * S * (nseg > 0 ? nseg : 1));
    double *Wp = (double *)malloc(sizeof(double) * S * CKPT); /* W_{t-1} in a segment */
    double *W = (double *)malloc(sizeof(double) * S);
    double *G = (double *)malloc(sizeof(double) * S);
    double *a = (double *)malloc(sizeof(double) * dk);
    double *r = (double *)malloc(sizeof(double) * dv);
    double *Gk = (double *)malloc(sizeof(double) * dv);
    double *dr = (double *)malloc(sizeof(double) * dv);
    double *Wt = (double *)malloc(sizeof(double) * S);
    double *dgc = (double *)malloc(sizeof(double) * dk);

    /* checkpoints: the state before the first token of each segment */
    load_state(s, h0, n, hd, W);
    for (seg = 0; seg < nseg; ++seg) {
        const int64_t t1 = (seg + 1) * CKPT < len ? (seg + 1) * CKPT : len;
        memcpy(ck + seg * S, W, sizeof(double) * S);
        for (t = seg * CKPT; t < t1; ++t) {
            const int64_t row = row0 + t;
            decay_of(s, g, row, hd, a);
            step(s, W, a, k + (row * H + hd) * dk, v + (row * H + hd) * dv,
                 beta[row * H + hd], r);
        }
    }

    /* G = dL/dW_L */
    if (dhT) {
        const double *src = dhT + ((int64_t)n * H + hd) * S;
        for (c = 0; c < dk; ++c)
            for (i = 0; i < dv; ++i) G[(int64_t)i * dk + c] = src[(int64_t)c * dv + i];
    } else {
        memset(G, 0, sizeof(double) * S);
    }

    for (seg = nseg - 1; seg >= 0; --seg) {
        const int64_t t0 = seg * CKPT;
        const int64_t t1 = (seg + 1) * CKPT < len ? (seg + 1) * CKPT : len;
        /* recompute W_{t-1} for t in [t0, t1) */
        memcpy(W, ck + seg * S, sizeof(double) * S);
        for (t = t0; t < t1; ++t) {
            const int64_t row = row0 + t;
            memcpy(Wp + (t - t0) * S, W, sizeof(double) * S);
            decay_of(s, g, row, hd, a);
            step(s, W, a, k + (row * H + hd) * dk, v + (row * H + hd) * dv,
                 beta[row * H + hd], r);
        }
        for (t = t1 - 1; t >= t0; --t) {
            const int64_t row = row0 + t;
            const double *Wprev = Wp + (t - t0) * S;
            const double *kt = k + (row * H + hd) * dk;
            const double *qt = q + (row * H + hd) * dk;
            const double *vt = v + (row * H + hd) * dv;
            const double *dot = dO + (row * H + hd) * dv;
            const double bt = beta[row * H + hd];
            double db = 0.0;
            decay_of(s, g, row, hd, a);
            /* Wt := decayed memory Wd_t, r := residual */
            for (i = 0; i < dv; ++i) {
                double p = 0.0;
                for (c = 0; c < dk; ++c) {
                    const double w = Wprev[(int64_t)i * dk + c] * a[c];
                    Wt[(int64_t)i * dk + c] = w;
                    p += w * kt[c];
                }
                r[i] = vt[i] - p;
            }
            /* the read: G += scale dO q^T ; dq = scale W_t^T dO, W_t = Wd + beta r k^T */
            for (i = 0; i < dv; ++i) {
                const double sd = s->scale * dot[i];
                for (c = 0; c < dk; ++c) G[(int64_t)i * dk + c] += sd * qt[c];
            }
            for (c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (i = 0; i < dv; ++i)
                    acc += (Wt[(int64_t)i * dk + c] + bt * r[i] * kt[c]) * dot[i];
                dq[(row * H + hd) * dk + c] = s->scale * acc;
            }
            /* the write and the residual (plus the gradient of the emitted write) */
            for (i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (c = 0; c < dk; ++c) acc += G[(int64_t)i * dk + c] * kt[c];
                if (dU) acc += dU[(row * H + hd) * dv + i];
                Gk[i] = acc;
                dr[i] = bt * acc;
                db += r[i] * acc;
            }
            dbeta[row * H + hd] = db;
            for (i = 0; i < dv; ++i) dvv[(row * H + hd) * dv + i] = dr[i];
            for (c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (i = 0; i < dv; ++i)
                    acc += bt * G[(int64_t)i * dk + c] * r[i] - Wt[(int64_t)i * dk + c] * dr[i];
                dkk[(row * H + hd) * dk + c] = acc;
            }
            /* dWd = G - dr k^T ; gate gradient ; G = dWd diag(a) */
            for (c = 0; c < dk; ++c) dgc[c] = 0.0;
            for (i = 0; i < dv; ++i) {
                double *gr = G + (int64_t)i * dk;
                const double *wp = Wprev + (int64_t)i * dk;
                for (c = 0; c < dk; ++c) {
                    const double dwd = gr[c] - dr[i] * kt[c];
                    dgc[c] += dwd * wp[c];
                    gr[c] = dwd * a[c];
                }
            }
            if (s->variant == DRO_GDN) {
                double acc = 0.0;
                for (c = 0; c < dk; ++c) acc += a[c] * dgc[c];
                dg[row * H + hd] = acc;
            } else if (s->variant == DRO_KDA) {
                for (c = 0; c < dk; ++c) dg[(row * H + hd) * dk + c] = a[c] * dgc[c];
            }
        }
    }
    if (dh0) {
        double *dst = dh0 + ((int64_t)n * H + hd) * S;
        for (c = 0; c < dk; ++c)
            for (i = 0; i < dv; ++i) dst[(int64_t)c * dv + i] = G[(int64_t)i * dk + c];
    }
    free(ck); free(Wp); free(W); free(G); free(a); free(r); free(Gk); free(dr);
    free(Wt); free(dgc);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Returns 0 on success, 1 on a bad shape. */
int dro_forward(int B, int T, int H, int dk, int dv, int variant, double scale,
                const int32_t *cu_seqlens, int N, const int32_t *units, int n_units,
                const double *q, const double *k, const double *v, const double *beta,
                const double *g, const double *h0, double *o, double *hT, double *u,
                int nthreads)
{
    shape_t s = {B, T, H, dk, dv, variant, scale, cu_seqlens, N};
    int64_t j, nu;
    if (check_shape(&s)) return 1;
    if (variant != DRO_DELTANET && !g) return 1;
    nu = units ? n_units : (int64_t)N * H;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (j = 0; j < nu; ++j) {
        const int un = units ? units[j] : (int)j;
        fwd_unit(&s, un, q, k, v, beta, g, h0, o, hT, u);
    }
    return 0;
}

int dro_backward(int B, int T, int H, int dk, int dv, int variant, double scale,
                 const int32_t *cu_seqlens, int N, const int32_t *units, int n_units,
                 const double *q, const double *k, const double *v, const double *beta,
                 const double *g, const double *h0, const double *dO, const double *dhT,
                 const double *dU, double *dq, double *dk_out, double *dv_out, double *dbeta,
                 double *dg, double *dh0, int nthreads)
{
    shape_t s = {B, T, H, dk, dv, variant, scale, cu_seqlens, N};
    int64_t j, nu;
    if (check_shape(&s)) return 1;
    if (variant != DRO_DELTANET && (!g || !dg)) return 1;
    nu = units ? n_units : (int64_t)N * H;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (j = 0; j < nu; ++j) {
        const int u = units ? units[j] : (int)j;
        bwd_unit(&s, u, q, k, v, beta, g, h0, dO, dhT, dU, dq, dk_out, dv_out, dbeta, dg, dh0);
    }
    return 0;
}

int dro_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
