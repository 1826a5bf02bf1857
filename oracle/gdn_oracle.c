/*
 * gdn_oracle.c -- plain fp64 CPU oracle for Gated DeltaNet (GDN) prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file.  It exists so that tests/, the smoke check and the
 * benchmark's CPU-baseline leg have an independent, obviously correct answer
 * to compare the CUDA kernels against.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it computes
 * ----------------
 * The pages ("FlashQLA是什么" on ollai.cn, section "FlashQLA的主要功能";
 * "Открыт FlashQLA" on aivizor, first paragraph) name the method -- the
 * forward and backward passes of GDN chunked prefill -- but never print the
 * recurrence.  The recurrence is the gated delta rule of Yang, Kautz and
 * Hatamizadeh ("Gated Delta Networks", ICLR 2025):
 *
 *     S_t = exp(g_t) * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t (scale * q_t),            scale = K^-1/2 unless given
 *
 * with S_t a V x K matrix.  The oracle keeps H_t = S_t^T (K x V, the key
 * index first), which turns one step into
 *
 *     Hbar = exp(g_t) H_{t-1}
 *     r_t  = v_t - Hbar^T k_t
 *     H_t  = Hbar + beta_t k_t r_t^T
 *     o_t  = scale * H_t^T q_t
 *
 * Chunking is a reformulation that reaches exactly this result (up to the
 * order of rounding), so the oracle runs the plain token-by-token recurrence
 * and does not emulate chunks.
 *
 * Backward: the reverse-mode recurrence of the step above, derived by hand
 * (chain rule through the four lines, last token first).  With dH the
 * gradient with respect to H_t:
 *
 *     dH   += scale q_t do_t^T          (o_t depends on H_t)
 *     dq_t  = scale H_t do_t
 *     dbeta_t = k_t^T dH r_t
 *     dr    = beta_t dH^T k_t
 *     dk_t  = beta_t dH r_t - Hbar dr
 *     dv_t  = dr
 *     dHbar = dH - k_t dr^T
 *     dg_t  = <dHbar, Hbar>_F
 *     dH    = exp(g_t) dHbar            (gradient with respect to H_{t-1})
 *
 * and d(initial_state) is dH after the first token.  States inside the
 * sequence are recomputed from checkpoints taken every CKPT tokens, so the
 * memory is O(K*V*T/CKPT) per (sequence, head).
 *
 * Optional L2 normalisation of q and k (the pages' prep step is silent on
 * it; the reading taken is x_hat = x * (sum x^2 + eps)^-1/2), and its
 * backward dx = (dx_hat - x_hat <x_hat, dx_hat>) * (sum x^2 + eps)^-1/2.
 *
 * Layouts (all row-major, token-major):
 *   q, k : [B, T, Hh, K]     v, o, do : [B, T, Hh, V]
 *   g, beta, dg, dbeta : [B, T, Hh]
 *   states (h0, hT, dhT, dh0) : [N, Hh, K, V]
 * With cu_seqlens (int32, N+1 entries), B must be 1 and sequence n covers
 * tokens cu_seqlens[n] .. cu_seqlens[n+1]-1; otherwise N = B.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0, *dout, *dht;
    const int32_t *cu_seqlens;
    int B, T, Hh, K, V;
    double scale, eps;
    int use_l2norm;
    double *o, *ht, *dq, *dk, *dv, *dg, *dbeta, *dh0;
} oracle_problem;

/* Token range [bos, bos+len) of sequence n. */
static void seq_range(const oracle_problem *p, int n, long *bos, long *len) {
    if (p->cu_seqlens) {
        *bos = p->cu_seqlens[n];
        *len = (long)p->cu_seqlens[n + 1] - p->cu_seqlens[n];
    } else {
        *bos = (long)n * p->T;
        *len = p->T;
    }
}

/* x_hat = x * (sum x^2 + eps)^-1/2 when normalising, else a plain copy.
 * Returns the factor (sum x^2 + eps)^-1/2 (1 when not normalising). */
static double load_vec(const double *x, int n, int normalise, double eps, double *out) {
    double s = 1.0;
    if (normalise) {
        double ss = 0.0;
        for (int i = 0; i < n; ++i) ss += x[i] * x[i];
        s = 1.0 / sqrt(ss + eps);
    }
    for (int i = 0; i < n; ++i) out[i] = x[i] * s;
    return s;
}

/* One forward step of the recurrence on H (K x V), in place.
 * Leaves Hbar^T k in r's complement: on return r = v - Hbar^T k. */
static void step_forward(double *H, int K, int V, double alpha, double beta,
                         const double *kt, const double *vt, double *r) {
    for (int i = 0; i < K * V; ++i) H[i] *= alpha;           /* Hbar */
    for (int j = 0; j < V; ++j) r[j] = vt[j];
    for (int i = 0; i < K; ++i) {
        const double ki = kt[i];
        const double *row = H + (long)i * V;
        for (int j = 0; j < V; ++j) r[j] -= row[j] * ki;     /* r = v - Hbar^T k */
    }
    for (int i = 0; i < K; ++i) {
        const double bk = beta * kt[i];
        double *row = H + (long)i * V;
        for (int j = 0; j < V; ++j) row[j] += bk * r[j];     /* H = Hbar + beta k r^T */
    }
}

static void output_row(const double *H, int K, int V, double scale, const double *qt, double *ot) {
    for (int j = 0; j < V; ++j) ot[j] = 0.0;
    for (int i = 0; i < K; ++i) {
        const double qi = qt[i];
        const double *row = H + (long)i * V;
        for (int j = 0; j < V; ++j) ot[j] += row[j] * qi;
    }
    for (int j = 0; j < V; ++j) ot[j] *= scale;
}

static void forward_unit(const oracle_problem *p, int n, int h) {
    const int K = p->K, V = p->V, Hh = p->Hh;
    long bos, len;
    seq_range(p, n, &bos, &len);
    double *H = (double *)malloc(sizeof(double) * K * V);
    double *qt = (double *)malloc(sizeof(double) * K);
    double *kt = (double *)malloc(sizeof(double) * K);
    double *r = (double *)malloc(sizeof(double) * V);
    const long sidx = ((long)n * Hh + h) * K * V;
    if (p->h0) memcpy(H, p->h0 + sidx, sizeof(double) * K * V);
    else memset(H, 0, sizeof(double) * K * V);
    for (long t = 0; t < len; ++t) {
        const long tok = bos + t;
        const long th = tok * Hh + h;
        load_vec(p->q + th * K, K, p->use_l2norm, p->eps, qt);
        load_vec(p->k + th * K, K, p->use_l2norm, p->eps, kt);
        step_forward(H, K, V, exp(p->g[th]), p->beta[th], kt, p->v + th * V, r);
        if (p->o) output_row(H, K, V, p->scale, qt, p->o + th * V);
    }
    if (p->ht) memcpy(p->ht + sidx, H, sizeof(double) * K * V);
    free(H); free(qt); free(kt); free(r);
}

static void backward_unit(const oracle_problem *p, int n, int h) {
    const int K = p->K, V = p->V, Hh = p->Hh;
    const long KV = (long)K * V;
    long bos, len;
    seq_range(p, n, &bos, &len);
    const long sidx = ((long)n * Hh + h) * KV;
    const long nck = (len + CKPT - 1) / CKPT;

    /* ckpt[c] = state before token c*CKPT. */
    double *ckpt = (double *)malloc(sizeof(double) * KV * (nck > 0 ? nck : 1));
    double *seg = (double *)malloc(sizeof(double) * KV * (CKPT + 1));
    double *dH = (double *)malloc(sizeof(double) * KV);
    double *Hbar = (double *)malloc(sizeof(double) * KV);
    double *qt = (double *)malloc(sizeof(double) * K);
    double *kt = (double *)malloc(sizeof(double) * K);
    double *dqh = (double *)malloc(sizeof(double) * K);
    double *dkh = (double *)malloc(sizeof(double) * K);
    double *r = (double *)malloc(sizeof(double) * V);
    double *dr = (double *)malloc(sizeof(double) * V);

    double *H = seg;  /* scratch for the checkpoint pass */
    if (p->h0) memcpy(H, p->h0 + sidx, sizeof(double) * KV);
    else memset(H, 0, sizeof(double) * KV);
    for (long t = 0; t < len; ++t) {
        if (t % CKPT == 0) memcpy(ckpt + (t / CKPT) * KV, H, sizeof(double) * KV);
        const long th = (bos + t) * Hh + h;
        load_vec(p->k + th * K, K, p->use_l2norm, p->eps, kt);
        step_forward(H, K, V, exp(p->g[th]), p->beta[th], kt, p->v + th * V, r);
    }

    if (p->dht) memcpy(dH, p->dht + sidx, sizeof(double) * KV);
    else memset(dH, 0, sizeof(double) * KV);

    for (long c = nck - 1; c >= 0; --c) {
        const long t0 = c * CKPT;
        const long t1 = (t0 + CKPT < len) ? t0 + CKPT : len;
        /* seg[i] = state after token t0+i-1 (seg[0] = state before t0). */
        memcpy(seg, ckpt + c * KV, sizeof(double) * KV);
        for (long t = t0; t < t1; ++t) {
            const long th = (bos + t) * Hh + h;
            double *next = seg + (t - t0 + 1) * KV;
            memcpy(next, seg + (t - t0) * KV, sizeof(double) * KV);
            load_vec(p->k + th * K, K, p->use_l2norm, p->eps, kt);
            step_forward(next, K, V, exp(p->g[th]), p->beta[th], kt, p->v + th * V, r);
        }
        for (long t = t1 - 1; t >= t0; --t) {
            const long th = (bos + t) * Hh + h;
            const double *Hprev = seg + (t - t0) * KV;
            const double *Ht = seg + (t - t0 + 1) * KV;
            const double alpha = exp(p->g[th]);
            const double beta = p->beta[th];
            const double sq = load_vec(p->q + th * K, K, p->use_l2norm, p->eps, qt);
            const double sk = load_vec(p->k + th * K, K, p->use_l2norm, p->eps, kt);
            const double *vt = p->v + th * V;
            const double *dot = p->dout + th * V;

            for (long i = 0; i < KV; ++i) Hbar[i] = alpha * Hprev[i];
            for (int j = 0; j < V; ++j) r[j] = vt[j];
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) r[j] -= Hbar[(long)i * V + j] * kt[i];

            /* dH += scale q do^T */
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) dH[(long)i * V + j] += p->scale * qt[i] * dot[j];
            /* dq = scale H_t do */
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j < V; ++j) s += Ht[(long)i * V + j] * dot[j];
                dqh[i] = p->scale * s;
            }
            /* dbeta = k^T dH r ; dr = beta dH^T k */
            double dbeta = 0.0;
            for (int j = 0; j < V; ++j) dr[j] = 0.0;
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j < V; ++j) {
                    s += dH[(long)i * V + j] * r[j];
                    dr[j] += dH[(long)i * V + j] * kt[i];
                }
                dbeta += kt[i] * s;
                dkh[i] = beta * s;                     /* beta dH r */
            }
            for (int j = 0; j < V; ++j) dr[j] *= beta;
            /* dk -= Hbar dr */
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j < V; ++j) s += Hbar[(long)i * V + j] * dr[j];
                dkh[i] -= s;
            }
            /* dHbar = dH - k dr^T ; dg = <dHbar, Hbar> ; dH = alpha dHbar */
            double dg = 0.0;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) {
                    const long ij = (long)i * V + j;
                    const double dhb = dH[ij] - kt[i] * dr[j];
                    dg += dhb * Hbar[ij];
                    dH[ij] = alpha * dhb;
                }

            /* Chain through the optional L2 normalisation. */
            double *dq_out = p->dq + th * K, *dk_out = p->dk + th * K;
            if (p->use_l2norm) {
                double pq = 0.0, pk = 0.0;
                for (int i = 0; i < K; ++i) { pq += qt[i] * dqh[i]; pk += kt[i] * dkh[i]; }
                for (int i = 0; i < K; ++i) {
                    dq_out[i] = (dqh[i] - qt[i] * pq) * sq;
                    dk_out[i] = (dkh[i] - kt[i] * pk) * sk;
                }
            } else {
                for (int i = 0; i < K; ++i) { dq_out[i] = dqh[i]; dk_out[i] = dkh[i]; }
            }
            memcpy(p->dv + th * V, dr, sizeof(double) * V);
            p->dg[th] = dg;
            p->dbeta[th] = dbeta;
        }
    }
    if (p->dh0) memcpy(p->dh0 + sidx, dH, sizeof(double) * KV);
    free(ckpt); free(seg); free(dH); free(Hbar); free(qt); free(kt);
    free(dqh); free(dkh); free(r); free(dr);
}

static int check_problem(const oracle_problem *p, int N) {
    if (!p->q || !p->k || !p->v || !p->g || !p->beta) return 1;
    if (p->B <= 0 || p->T < 0 || p->Hh <= 0 || p->K <= 0 || p->V <= 0 || N < 0) return 1;
    if (p->cu_seqlens) {
        if (p->B != 1 || p->cu_seqlens[0] != 0 || p->cu_seqlens[N] != p->T) return 1;
        for (int n = 0; n < N; ++n)
            if (p->cu_seqlens[n + 1] < p->cu_seqlens[n]) return 1;
    }
    return 0;
}

/* Runs `fn` over the listed (sequence, head) units, unit u = n*Hh + h.
 * unit_list == NULL means every unit. */
static void run_units(const oracle_problem *p, int N, const int32_t *unit_list, int n_units,
                      int nthreads, void (*fn)(const oracle_problem *, int, int)) {
    const int total = unit_list ? n_units : N * p->Hh;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int i = 0; i < total; ++i) {
        const int u = unit_list ? unit_list[i] : i;
        fn(p, u / p->Hh, u % p->Hh);
    }
    (void)nthreads;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward.  o may be NULL (states only); ht may be NULL. Returns 0 on success. */
int gdn_oracle_fwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *h0, const int32_t *cu_seqlens, int N,
                   int B, int T, int Hh, int K, int V, double scale, int use_l2norm, double eps,
                   double *o, double *ht, const int32_t *unit_list, int n_units, int nthreads) {
    oracle_problem p;
    memset(&p, 0, sizeof p);
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.Hh = Hh; p.K = K; p.V = V; p.scale = scale; p.eps = eps;
    p.use_l2norm = use_l2norm; p.o = o; p.ht = ht;
    if (!cu_seqlens) N = B;
    if (check_problem(&p, N)) return 1;
    run_units(&p, N, unit_list, n_units, nthreads, forward_unit);
    return 0;
}

/* Backward.  dht and h0 may be NULL (zeros); dh0 may be NULL. */
int gdn_oracle_bwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *h0, const int32_t *cu_seqlens, int N,
                   int B, int T, int Hh, int K, int V, double scale, int use_l2norm, double eps,
                   const double *dout, const double *dht, double *dq, double *dk, double *dv,
                   double *dg, double *dbeta, double *dh0, const int32_t *unit_list, int n_units,
                   int nthreads) {
    oracle_problem p;
    memset(&p, 0, sizeof p);
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.Hh = Hh; p.K = K; p.V = V; p.scale = scale; p.eps = eps;
    p.use_l2norm = use_l2norm; p.dout = dout; p.dht = dht;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dh0 = dh0;
    if (!cu_seqlens) N = B;
    if (check_problem(&p, N) || !dout || !dq || !dk || !dv || !dg || !dbeta) return 1;
    run_units(&p, N, unit_list, n_units, nthreads, backward_unit);
    return 0;
}

/*
 * Gate preprocessing (the pages' "gate preprocessing" ahead of the kernels,
 * aivizor, FLA-flow paragraph; its form is the GDN layer's decay gate):
 * the log decay of token t, head h is g = -a_h * softplus(x_t,h) from a raw
 * gate logit x and a positive per-head scale a_h, softplus(x) = log(1 + e^x).
 * Its backward: dx = dg * (-a_h * sigmoid(x)), da_h = sum_t dg * (-softplus(x)).
 * x, g, dg, dx: [n_tok, Hh];  a, da: [Hh].
 */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

int gdn_oracle_gate(const double *x, const double *a, long n_tok, int Hh, double *g) {
    if (!x || !a || !g || n_tok < 0 || Hh <= 0) return 1;
    for (long t = 0; t < n_tok; ++t)
        for (int h = 0; h < Hh; ++h) g[t * Hh + h] = -a[h] * softplus(x[t * Hh + h]);
    return 0;
}

int gdn_oracle_gate_bwd(const double *x, const double *a, const double *dg, long n_tok, int Hh,
                        double *dx, double *da) {
    if (!x || !a || !dg || !dx || n_tok < 0 || Hh <= 0) return 1;
    for (int h = 0; h < Hh; ++h) {
        double acc = 0.0;
        for (long t = 0; t < n_tok; ++t) {
            const double xv = x[t * Hh + h], d = dg[t * Hh + h];
            dx[t * Hh + h] = -a[h] * d / (1.0 + exp(-xv));
            acc -= d * softplus(xv);
        }
        if (da) da[h] = acc;
    }
    return 0;
}
