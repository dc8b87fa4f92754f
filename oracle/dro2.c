/*
 * dro2.c -- sequential fp64 oracle of Gated DeltaNet-2 (separate erase and write
 * gates).
 *
 * TEST INFRASTRUCTURE ONLY, like dro.c: nothing in the product path links, loads or
 * calls it, and it shares no code with the CUDA library.
 *
 * The pages ("Linear Attention Architectures: Mechanisms, Trade-offs, and Cross-Layer
 * Routing", section "Metodologia y Marco de Trabajo", item 1, the Gated DeltaNet-2
 * bullet) describe this variant in words only: it decouples the delta-rule update of
 * Gated DeltaNet further, with separate per-channel gates for erasing (which key
 * channels are removed) and for writing (which value channels are stored).  They print
 * no equation.  The reading taken here, the plainest one that keeps everything else of
 * the Gated DeltaNet bullet (scalar decay applied before the residual) and reduces to
 * it when both gates equal beta:
 *
 *   decayed   Wd_t = alpha_t W_{t-1}                    alpha_t = exp(g_t), one scalar
 *   predicted p_t  = Wd_t k_t                           (the memory's value for k_t)
 *   erased    Wd_t - p_t (e_t . k_t)^T                  e_t in [0,1]^{d_k}, per key channel
 *   written   W_t  = Wd_t - p_t (e_t . k_t)^T + (w_t . v_t) k_t^T
 *                                                       w_t in [0,1]^{d_v}, per value channel
 *   read      o_t  = scale * W_t q_t
 *
 * ("." is the elementwise product.)  With e_t = beta_t 1 and w_t = beta_t 1 this is
 * Gated DeltaNet: Wd + beta_t (v_t - p_t) k_t^T.
 *
 * Backward: the reverse-time recurrence derived by hand from those lines.  With
 * G = dL/dW_t (d_v x d_k), b_t = e_t . k_t, vw_t = w_t . v_t:
 *
 *   G   += scale * dO_t q_t^T           dq_t = scale * W_t^T dO_t
 *   dvw  = G k_t        dv_t = w_t . dvw     dw_t = v_t . dvw
 *   db   = -G^T p_t     de_t = k_t . db      dk_t = G^T vw_t + e_t . db
 *   dp   = -G b_t
 *   dWd  = G + dp k_t^T                      dk_t += Wd_t^T dp
 *   dg_t = alpha_t * sum(dWd . W_{t-1})
 *   G    = alpha_t dWd
 *
 * and dL/dW_0 = G at the end.  W_{t-1} is recomputed from checkpoints every CKPT2
 * tokens.  Layouts as dro.c; erase [B,T,H,d_k], write [B,T,H,d_v], g [B,T,H].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT2 64

typedef struct {
    int B, T, H, dk, dv;
    double scale;
    const int32_t *cu;
    int N;
} shape2_t;

static int check2(const shape2_t *s)
{
    if (s->B < 0 || s->T < 0 || s->H <= 0 || s->dk <= 0 || s->dv <= 0) return 1;
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

static void range2(const shape2_t *s, int n, int64_t *row0, int64_t *len)
{
    if (s->cu) {
        *row0 = s->cu[n];
        *len = (int64_t)s->cu[n + 1] - s->cu[n];
    } else {
        *row0 = (int64_t)n * s->T;
        *len = s->T;
    }
}

/* W (dv x dk) from the stored state S = W^T [dk][dv] (zero when h is NULL) */
static void load2(const shape2_t *s, const double *h, int n, int hd, double *W)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    if (!h) {
        memset(W, 0, sizeof(double) * dk * dv);
        return;
    }
    h += ((int64_t)n * s->H + hd) * dk * dv;
    for (c = 0; c < dk; ++c)
        for (i = 0; i < dv; ++i) W[(int64_t)i * dk + c] = h[(int64_t)c * dv + i];
}

static void store2(const shape2_t *s, double *h, int n, int hd, const double *W)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    h += ((int64_t)n * s->H + hd) * dk * dv;
    for (c = 0; c < dk; ++c)
        for (i = 0; i < dv; ++i) h[(int64_t)c * dv + i] = W[(int64_t)i * dk + c];
}

/* One token step in place on W; p receives the prediction Wd k. */
static void step2(const shape2_t *s, double *W, double alpha, const double *kt,
                  const double *vt, const double *et, const double *wt, double *p)
{
    const int dk = s->dk, dv = s->dv;
    int i, c;
    for (i = 0; i < dv; ++i) {
        double *w = W + (int64_t)i * dk;
        double acc = 0.0;
        for (c = 0; c < dk; ++c) {
            w[c] *= alpha;
            acc += w[c] * kt[c];
        }
        p[i] = acc;
    }
    for (i = 0; i < dv; ++i) {
        double *w = W + (int64_t)i * dk;
        const double vw = wt[i] * vt[i];
        for (c = 0; c < dk; ++c) w[c] += vw * kt[c] - p[i] * et[c] * kt[c];
    }
}

static void fwd2_unit(const shape2_t *s, int u, const double *q, const double *k,
                      const double *v, const double *er, const double *wr, const double *g,
                      const double *h0, double *o, double *hT)
{
    const int dk = s->dk, dv = s->dv, H = s->H, n = u / H, hd = u % H;
    int64_t row0, len, t;
    int i, c;
    double *W = (double *)malloc(sizeof(double) * dk * dv);
    double *p = (double *)malloc(sizeof(double) * dv);
    range2(s, n, &row0, &len);
    load2(s, h0, n, hd, W);
    for (t = 0; t < len; ++t) {
        const int64_t row = row0 + t, rk = (row * H + hd) * dk, rv = (row * H + hd) * dv;
        step2(s, W, exp(g[row * H + hd]), k + rk, v + rv, er + rk, wr + rv, p);
        if (o) {
            for (i = 0; i < dv; ++i) {
                const double *w = W + (int64_t)i * dk;
                double acc = 0.0;
                for (c = 0; c < dk; ++c) acc += w[c] * q[rk + c];
                o[rv + i] = s->scale * acc;
            }
        }
    }
    if (hT) store2(s, hT, n, hd, W);
    free(W);
    free(p);
}

static void bwd2_unit(const shape2_t *s, int u, const double *q, const double *k,
                      const double *v, const double *er, const double *wr, const double *g,
                      const double *h0, const double *dO, const double *dhT, double *dq,
                      double *dk_o, double *dv_o, double *de_o, double *dw_o, double *dg_o,
                      double *dh0)
{
    const int dk = s->dk, dv = s->dv, H = s->H, n = u / H, hd = u % H;
    const int64_t SZ = (int64_t)dk * dv;
    int64_t row0, len, t, nck, seg;
    int i, c;
    range2(s, n, &row0, &len);
    nck = (len + CKPT2 - 1) / CKPT2;
    double *ck = (double *)malloc(sizeof(double) * SZ * (nck > 0 ? nck : 1));
    double *Wseg = (double *)malloc(sizeof(double) * SZ * (CKPT2 + 1)); /* W_{t-1}, .., W_t */
    double *Pseg = (double *)malloc(sizeof(double) * dv * CKPT2);
    double *W = (double *)malloc(sizeof(double) * SZ);
    double *G = (double *)malloc(sizeof(double) * SZ);
    double *dvw = (double *)malloc(sizeof(double) * dv);
    double *dp = (double *)malloc(sizeof(double) * dv);
    double *db = (double *)malloc(sizeof(double) * dk);
    /* checkpoints: the state at the start of every segment */
    load2(s, h0, n, hd, W);
    for (t = 0; t < len; ++t) {
        const int64_t row = row0 + t, rk = (row * H + hd) * dk, rv = (row * H + hd) * dv;
        if (t % CKPT2 == 0) memcpy(ck + (t / CKPT2) * SZ, W, sizeof(double) * SZ);
        step2(s, W, exp(g[row * H + hd]), k + rk, v + rv, er + rk, wr + rv, dvw);
    }
    /* G = dL/dW_L */
    if (dhT) {
        load2(s, dhT, n, hd, G);
    } else {
        memset(G, 0, sizeof(double) * SZ);
    }
    for (seg = nck - 1; seg >= 0; --seg) {
        const int64_t t0 = seg * CKPT2, t1 = (t0 + CKPT2 < len) ? t0 + CKPT2 : len;
        /* recompute W_{t0-1} .. W_{t1-1} and the predictions of the segment */
        memcpy(Wseg, ck + seg * SZ, sizeof(double) * SZ);
        for (t = t0; t < t1; ++t) {
            const int64_t row = row0 + t, rk = (row * H + hd) * dk, rv = (row * H + hd) * dv;
            double *Wn = Wseg + (t - t0 + 1) * SZ;
            memcpy(Wn, Wseg + (t - t0) * SZ, sizeof(double) * SZ);
            step2(s, Wn, exp(g[row * H + hd]), k + rk, v + rv, er + rk, wr + rv,
                  Pseg + (t - t0) * dv);
        }
        for (t = t1 - 1; t >= t0; --t) {
            const int64_t row = row0 + t, rk = (row * H + hd) * dk, rv = (row * H + hd) * dv;
            const double *Wprev = Wseg + (t - t0) * SZ, *Wt = Wseg + (t - t0 + 1) * SZ;
            const double *p = Pseg + (t - t0) * dv;
            const double *kt = k + rk, *qt = q + rk, *et = er + rk;
            const double *vt = v + rv, *wt = wr + rv, *dot = dO + rv;
            const double alpha = exp(g[row * H + hd]);
            double dgt = 0.0;
            /* read: G += scale dO q^T; dq = scale W_t^T dO */
            for (i = 0; i < dv; ++i)
                for (c = 0; c < dk; ++c) G[(int64_t)i * dk + c] += s->scale * dot[i] * qt[c];
            for (c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (i = 0; i < dv; ++i) acc += Wt[(int64_t)i * dk + c] * dot[i];
                dq[rk + c] = s->scale * acc;
            }
            /* write and erase terms */
            for (i = 0; i < dv; ++i) {
                double a1 = 0.0, a2 = 0.0;
                for (c = 0; c < dk; ++c) {
                    a1 += G[(int64_t)i * dk + c] * kt[c];
                    a2 += G[(int64_t)i * dk + c] * et[c] * kt[c];
                }
                dvw[i] = a1;
                dp[i] = -a2;
                dv_o[rv + i] = wt[i] * a1;
                dw_o[rv + i] = vt[i] * a1;
            }
            for (c = 0; c < dk; ++c) {
                double gv = 0.0, gp = 0.0, wdp = 0.0;
                for (i = 0; i < dv; ++i) {
                    const double Gic = G[(int64_t)i * dk + c];
                    gv += Gic * wt[i] * vt[i];
                    gp += Gic * p[i];
                    wdp += alpha * Wprev[(int64_t)i * dk + c] * dp[i];
                }
                db[c] = -gp;
                de_o[rk + c] = kt[c] * db[c];
                dk_o[rk + c] = gv + et[c] * db[c] + wdp;
            }
            /* dWd = G + dp k^T;  dg = alpha sum(dWd . W_{t-1});  G = alpha dWd */
            for (i = 0; i < dv; ++i)
                for (c = 0; c < dk; ++c) {
                    const int64_t ix = (int64_t)i * dk + c;
                    const double dWd = G[ix] + dp[i] * kt[c];
                    dgt += dWd * Wprev[ix];
                    G[ix] = alpha * dWd;
                }
            dg_o[row * H + hd] = alpha * dgt;
        }
    }
    if (dh0) store2(s, dh0, n, hd, G);
    free(ck); free(Wseg); free(Pseg); free(W); free(G); free(dvw); free(dp); free(db);
}

static void threads2(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Returns 0 on success, 1 on a bad shape.  units: NULL = all N*H (sequence, head) pairs. */
int dro2_forward(int B, int T, int H, int dk, int dv, double scale, const int32_t *cu_seqlens,
                 int N, const int32_t *units, int n_units, const double *q, const double *k,
                 const double *v, const double *erase, const double *write, const double *g,
                 const double *h0, double *o, double *hT, int nthreads)
{
    shape2_t s = {B, T, H, dk, dv, scale, cu_seqlens, N};
    int64_t j, nu;
    if (check2(&s) || !g || !erase || !write) return 1;
    nu = units ? n_units : (int64_t)N * H;
    threads2(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (j = 0; j < nu; ++j)
        fwd2_unit(&s, units ? units[j] : (int)j, q, k, v, erase, write, g, h0, o, hT);
    return 0;
}

int dro2_backward(int B, int T, int H, int dk, int dv, double scale, const int32_t *cu_seqlens,
                  int N, const int32_t *units, int n_units, const double *q, const double *k,
                  const double *v, const double *erase, const double *write, const double *g,
                  const double *h0, const double *dO, const double *dhT, double *dq,
                  double *dk_out, double *dv_out, double *derase, double *dwrite, double *dg,
                  double *dh0, int nthreads)
{
    shape2_t s = {B, T, H, dk, dv, scale, cu_seqlens, N};
    int64_t j, nu;
    if (check2(&s) || !g || !erase || !write) return 1;
    nu = units ? n_units : (int64_t)N * H;
    threads2(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (j = 0; j < nu; ++j)
        bwd2_unit(&s, units ? units[j] : (int)j, q, k, v, erase, write, g, h0, dO, dhT, dq,
                  dk_out, dv_out, derase, dwrite, dg, dh0);
    return 0;
}
