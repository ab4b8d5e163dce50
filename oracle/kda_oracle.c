/*
 * fp64 CPU oracle for the Kimi Delta Attention (KDA) gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links or calls this
 * file; only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark load it.
 *
 * What it computes (flashinfer "kda_backward" page, "Supported contract";
 * FLA chunk_kda call contract on the Kimi-K3 "fused_chunk" page):
 *   value-first state S in R^{V x K} per (sequence, head);
 *   q^ = q / sqrt(|q|^2 + eps), k^ likewise, eps = 1e-6;
 *   beta = sigmoid(beta_raw);
 *   g_c = lb * sigmoid(exp(A_log) * (g_raw_c + dt_bias_c)), decay exp(g_c),
 *   one decay per KEY channel c (the kda-neuron-kernels log, fix T-KDA-02:
 *   decaying per value column is the bug);
 *   S_t = S_{t-1} diag(exp(g_t)) (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T;
 *   o_t = scale * S_t q^_t.
 * The recurrence is evaluated token by token, exactly as written, in fp64.
 *
 * The reverse mode is derived by hand from the same step (chain rule through
 * the rank-one write, the residual r = v - S' k^, the per-key decay, the
 * gate, the beta sigmoid and the L2 norms); the flashinfer page lists the
 * gradients it returns: q, k, v, raw gate, raw beta, A_log, dt_bias and the
 * initial state. The loss seen by the backward is
 *   L = sum_t <o_t, dO_t> + <h_T, dh_T>.
 *
 * Two modes:
 *   raw  (mode 1): q, k are normalised here; g_raw, beta_raw, A_log, dt_bias
 *                  go through the gate and the sigmoid.
 *   core (mode 0): q^, k^ are taken as given (no normalisation), the
 *                  log-decay g and beta are given directly. Used to pin the
 *                  recurrence on exact special cases (beta = 0 or 1, g = 0).
 *
 * The backward recomputes the states of each 64-token segment from an fp64
 * checkpoint at the segment start; the recomputation repeats the forward's
 * operations in the same order, so the states are bitwise the forward's.
 *
 * Units (sequence, head) are independent and run on POSIX threads. The
 * parameter gradients are written per unit and summed by the caller in a
 * fixed order.
 *
 * Grouped value heads (the FlashKDA CPU-reference proposal lists them): with
 * G value heads per query/key head, value head h reads q, k of head h / G
 * (q, k hold H / G heads); every other tensor is per value head. dq and dk are
 * written per value head and summed over each group by the caller, in a fixed
 * order. G = 1 is the plain layout.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t N, H, K, V;
    const int64_t *cu;          /* [N+1] token offsets, host */
    double scale, lb, eps;
    int mode;                   /* 1 raw, 0 core */
    int nthreads;
    /* forward inputs, packed over tokens */
    const double *q, *k;        /* [T,H/G,K] */
    const double *v;            /* [T,H,V] */
    const double *gx;           /* raw: g_raw [T,H,K]; core: log-decay g [T,H,K] */
    const double *bx;           /* raw: beta_raw [T,H]; core: beta [T,H] */
    const double *A_log;        /* [H] (raw) */
    const double *dt_bias;      /* [H,K] (raw) */
    const double *h0;           /* [N,H,V,K] or NULL (= 0) */
    /* forward outputs */
    double *o;                  /* [T,H,V] or NULL */
    double *hT;                 /* [N,H,V,K] or NULL */
    /* backward inputs */
    const double *dO;           /* [T,H,V] */
    const double *dhT;          /* [N,H,V,K] or NULL (= 0) */
    /* backward outputs */
    double *dq, *dk;            /* [T,H,K] per value head (raw: wrt q,k; core: wrt q^,k^) */
    double *dv;                 /* [T,H,V] */
    double *dgx;                /* raw: wrt g_raw; core: wrt g. [T,H,K] */
    double *dbx;                /* raw: wrt beta_raw; core: wrt beta. [T,H] */
    double *dA_log_unit;        /* [N,H] per-unit partial (raw) */
    double *ddt_bias_unit;      /* [N,H,K] per-unit partial (raw) */
    double *dh0;                /* [N,H,V,K] or NULL */
    int64_t G;                  /* value heads per query/key head (q, k: [T,H/G,K]); 1 = none */
} kda_oracle_args;

enum { SEG = 64 };

/* Test hook: the oracle's own tests rebuild it with KDA_ORACLE_MUTATION = n to
 * plant one plausible mistake and check that the pins catch it. 0 = none. */
#ifndef KDA_ORACLE_MUTATION
#define KDA_ORACLE_MUTATION 0
#endif
#define MUT(n) (KDA_ORACLE_MUTATION == (n))

/* Per-token quantities of the step, in the pages' notation. */
typedef struct {
    double *qh, *kh, *g, *alpha;   /* [K] */
    double *s;                     /* [K] sigmoid of the gate pre-activation (raw) */
    double beta, nq, nk;           /* nq, nk: sqrt(|x|^2 + eps) (raw) */
} tok_t;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Gate, beta and L2 norm of token t, head h (flashinfer page, contract). */
static void prep_token(const kda_oracle_args *a, int64_t t, int64_t h, tok_t *x)
{
    const int64_t K = a->K, H = a->H, G = a->G > 0 ? a->G : 1;
    const int64_t hk = MUT(11) ? h % (H / G) : h / G;   /* the query/key head of value head h */
    const double *q = a->q + (t * (H / G) + hk) * K;
    const double *k = a->k + (t * (H / G) + hk) * K;
    const double *gx = a->gx + (t * H + h) * K;
    const double bx = a->bx[t * H + h];
    if (a->mode == 1) {
        double sq = 0.0, sk = 0.0;
        for (int64_t c = 0; c < K; ++c) { sq += q[c] * q[c]; sk += k[c] * k[c]; }
        x->nq = MUT(4) ? sqrt(sq) + a->eps : sqrt(sq + a->eps);
        x->nk = sqrt(sk + a->eps);
        const double am = exp(a->A_log[h]);
        for (int64_t c = 0; c < K; ++c) {
            x->qh[c] = q[c] / x->nq;
            x->kh[c] = k[c] / x->nk;
            x->s[c] = sigmoid(am * (gx[c] + a->dt_bias[h * K + c]));
            x->g[c] = (MUT(3) ? -a->lb : a->lb) * x->s[c];
            x->alpha[c] = exp(x->g[c]);
        }
        x->beta = sigmoid(bx);
    } else {
        x->nq = x->nk = 1.0;
        for (int64_t c = 0; c < K; ++c) {
            x->qh[c] = q[c];
            x->kh[c] = k[c];
            x->s[c] = 0.0;
            x->g[c] = gx[c];
            x->alpha[c] = exp(gx[c]);
        }
        x->beta = bx;
    }
}

/* One forward step S_{t-1} -> S_t in place; r receives v - S' k^.
 * Writes o_t = scale * S_t q^ when o != NULL. */
static void step_fwd(const kda_oracle_args *a, const tok_t *x, const double *vt,
                     double *S, double *r, double *o)
{
    const int64_t K = a->K, V = a->V;
    for (int64_t i = 0; i < V; ++i) {
        double *row = S + i * K;
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            row[c] *= MUT(1) ? x->alpha[i % K] : x->alpha[c];   /* S' = S diag(exp(g)) */
            acc += row[c] * x->kh[c];
        }
        r[i] = vt[i] - acc;                   /* r = v - S' k^ */
        if (MUT(10)) r[i] = vt[i] - (i < K ? S[i * K + i] : 0.0) * x->kh[i % K] - acc;
        const double br = x->beta * r[i];
        double oi = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            if (MUT(2)) oi += row[c] * x->qh[c];
            row[c] += br * x->kh[c];          /* S = S' + beta r k^T */
            if (!MUT(2)) oi += row[c] * x->qh[c];
        }
        if (o) o[i] = a->scale * oi;          /* o = scale S q^ */
    }
}

typedef struct {
    const kda_oracle_args *a;
    int64_t next;               /* shared unit counter */
    pthread_mutex_t mu;
    int backward;
} pool_t;

static int64_t take_unit(pool_t *p)
{
    pthread_mutex_lock(&p->mu);
    int64_t u = p->next++;
    pthread_mutex_unlock(&p->mu);
    return u;
}

typedef struct {
    double *S, *r, *buf;
    tok_t x;
} scratch_t;

static void scratch_init(scratch_t *w, int64_t K, int64_t V, size_t extra)
{
    w->S = (double *)calloc((size_t)(V * K), sizeof(double));
    w->r = (double *)calloc((size_t)V, sizeof(double));
    w->buf = (double *)calloc((size_t)(5 * K) + extra, sizeof(double));
    w->x.qh = w->buf;
    w->x.kh = w->buf + K;
    w->x.g = w->buf + 2 * K;
    w->x.alpha = w->buf + 3 * K;
    w->x.s = w->buf + 4 * K;
}

static void scratch_free(scratch_t *w) { free(w->S); free(w->r); free(w->buf); }

static void unit_forward(const kda_oracle_args *a, int64_t n, int64_t h, scratch_t *w)
{
    const int64_t K = a->K, V = a->V, H = a->H;
    const size_t sz = (size_t)(V * K);
    if (a->h0) memcpy(w->S, a->h0 + (n * H + h) * V * K, sz * sizeof(double));
    else memset(w->S, 0, sz * sizeof(double));
    for (int64_t t = a->cu[n]; t < a->cu[n + 1]; ++t) {
        prep_token(a, t, h, &w->x);
        step_fwd(a, &w->x, a->v + (t * H + h) * V, w->S, w->r,
                 a->o ? a->o + (t * H + h) * V : NULL);
    }
    if (a->hT) memcpy(a->hT + (n * H + h) * V * K, w->S, sz * sizeof(double));
}

static void unit_backward(const kda_oracle_args *a, int64_t n, int64_t h, scratch_t *w)
{
    const int64_t K = a->K, V = a->V, H = a->H;
    const size_t sz = (size_t)(V * K);
    const int64_t t0 = a->cu[n], t1 = a->cu[n + 1], L = t1 - t0;
    const int64_t nseg = (L + SEG - 1) / SEG;

    /* checkpoints: state at the start of each segment */
    double *ck = (double *)malloc((size_t)(nseg > 0 ? nseg : 1) * sz * sizeof(double));
    /* states S_{t-1} for every step of one segment, plus the state after it */
    double *st = (double *)malloc((size_t)(SEG + 1) * sz * sizeof(double));
    double *dS = (double *)calloc(sz, sizeof(double));
    double *dSp = (double *)calloc(sz, sizeof(double));
    double *Sp = (double *)calloc(sz, sizeof(double));
    double *dqh = (double *)calloc((size_t)K, sizeof(double));
    double *dkh = (double *)calloc((size_t)K, sizeof(double));
    double *dal = (double *)calloc((size_t)K, sizeof(double));
    double *dr = (double *)calloc((size_t)V, sizeof(double));
    double *ddt = a->mode == 1 ? a->ddt_bias_unit + (n * H + h) * K : NULL;
    double dA = 0.0;

    if (a->h0) memcpy(w->S, a->h0 + (n * H + h) * V * K, sz * sizeof(double));
    else memset(w->S, 0, sz * sizeof(double));
    for (int64_t sg = 0; sg < nseg; ++sg) {
        memcpy(ck + sg * sz, w->S, sz * sizeof(double));
        const int64_t e = (sg + 1) * SEG < L ? (sg + 1) * SEG : L;
        for (int64_t t = t0 + sg * SEG; t < t0 + e; ++t) {
            prep_token(a, t, h, &w->x);
            step_fwd(a, &w->x, a->v + (t * H + h) * V, w->S, w->r, NULL);
        }
    }
    if (a->dhT) memcpy(dS, a->dhT + (n * H + h) * V * K, sz * sizeof(double));
    if (ddt) memset(ddt, 0, (size_t)K * sizeof(double));

    for (int64_t sg = nseg - 1; sg >= 0; --sg) {
        const int64_t b = sg * SEG, e = (sg + 1) * SEG < L ? (sg + 1) * SEG : L;
        /* recompute the segment: st[j] = S before step b+j */
        memcpy(st, ck + sg * sz, sz * sizeof(double));
        for (int64_t j = 0; j < e - b; ++j) {
            const int64_t t = t0 + b + j;
            memcpy(st + (j + 1) * sz, st + j * sz, sz * sizeof(double));
            prep_token(a, t, h, &w->x);
            step_fwd(a, &w->x, a->v + (t * H + h) * V, st + (j + 1) * sz, w->r, NULL);
        }
        for (int64_t j = e - b - 1; j >= 0; --j) {
            const int64_t t = t0 + b + j;
            const double *Sprev = st + j * sz;      /* S_{t-1} */
            const double *St = st + (j + 1) * sz;    /* S_t */
            const double *vt = a->v + (t * H + h) * V;
            const double *dOt = a->dO + (t * H + h) * V;
            tok_t *x = &w->x;
            prep_token(a, t, h, x);
            /* S' = S_{t-1} diag(alpha), r = v - S' k^ */
            for (int64_t i = 0; i < V; ++i) {
                double acc = 0.0;
                for (int64_t c = 0; c < K; ++c) {
                    Sp[i * K + c] = Sprev[i * K + c] * x->alpha[c];
                    acc += Sp[i * K + c] * x->kh[c];
                }
                w->r[i] = vt[i] - acc;
            }
            /* output: o = scale S_t q^ */
            for (int64_t c = 0; c < K; ++c) dqh[c] = 0.0;
            for (int64_t i = 0; i < V; ++i) {
                const double sd = a->scale * dOt[i];
                for (int64_t c = 0; c < K; ++c) {
                    dS[i * K + c] += sd * x->qh[c];
                    dqh[c] += sd * St[i * K + c];
                }
            }
            /* rank-one write S_t = S' + beta r k^T */
            double dbeta = 0.0;
            for (int64_t c = 0; c < K; ++c) dkh[c] = 0.0;
            for (int64_t i = 0; i < V; ++i) {
                double dsk = 0.0;
                for (int64_t c = 0; c < K; ++c) dsk += dS[i * K + c] * x->kh[c];
                dbeta += w->r[i] * dsk;
                dr[i] = x->beta * dsk;
                for (int64_t c = 0; c < K; ++c) dkh[c] += x->beta * dS[i * K + c] * w->r[i];
            }
            /* residual r = v - S' k^ */
            for (int64_t i = 0; i < V; ++i) {
                if (a->dv) a->dv[(t * H + h) * V + i] = dr[i];
                for (int64_t c = 0; c < K; ++c) {
                    dSp[i * K + c] = dS[i * K + c] - dr[i] * x->kh[c];
                    if (!MUT(5)) dkh[c] -= Sp[i * K + c] * dr[i];
                }
            }
            /* decay S' = S_{t-1} diag(alpha) */
            for (int64_t c = 0; c < K; ++c) dal[c] = 0.0;
            for (int64_t i = 0; i < V; ++i)
                for (int64_t c = 0; c < K; ++c) {
                    dal[c] += dSp[i * K + c] * Sprev[i * K + c];
                    dS[i * K + c] = MUT(6) ? dSp[i * K + c] : dSp[i * K + c] * x->alpha[c];
                }
            /* gate, beta and norm chains */
            double *dgo = a->dgx + (t * H + h) * K;
            if (a->mode == 1) {
                const double am = exp(a->A_log[h]);
                const double *graw = a->gx + (t * H + h) * K;
                for (int64_t c = 0; c < K; ++c) {
                    const double dg = dal[c] * x->alpha[c];
                    const double du = dg * a->lb * x->s[c] * (MUT(7) ? 1.0 : (1.0 - x->s[c]));
                    dgo[c] = du * am;
                    ddt[c] += du * am;
                    dA += du * (MUT(8) ? 1.0 : am) * (graw[c] + a->dt_bias[h * K + c]);
                }
                a->dbx[t * H + h] = dbeta * x->beta * (1.0 - x->beta);
                double pq = 0.0, pk = 0.0;
                for (int64_t c = 0; c < K; ++c) { pq += x->qh[c] * dqh[c]; pk += x->kh[c] * dkh[c]; }
                for (int64_t c = 0; c < K; ++c) {
                    a->dq[(t * H + h) * K + c] = (dqh[c] - (MUT(9) ? 0.0 : x->qh[c] * pq)) / x->nq;
                    a->dk[(t * H + h) * K + c] = (dkh[c] - x->kh[c] * pk) / x->nk;
                }
            } else {
                for (int64_t c = 0; c < K; ++c) {
                    dgo[c] = dal[c] * x->alpha[c];
                    a->dq[(t * H + h) * K + c] = dqh[c];
                    a->dk[(t * H + h) * K + c] = dkh[c];
                }
                a->dbx[t * H + h] = dbeta;
            }
        }
    }
    if (a->dh0) memcpy(a->dh0 + (n * H + h) * V * K, dS, sz * sizeof(double));
    if (a->mode == 1) a->dA_log_unit[n * H + h] = dA;
    free(ck); free(st); free(dS); free(dSp); free(Sp);
    free(dqh); free(dkh); free(dal); free(dr);
}

static void *worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    const kda_oracle_args *a = p->a;
    scratch_t w;
    scratch_init(&w, a->K, a->V, 0);
    const int64_t units = a->N * a->H;
    for (;;) {
        const int64_t u = take_unit(p);
        if (u >= units) break;
        const int64_t n = u / a->H, h = u % a->H;
        if (p->backward) unit_backward(a, n, h, &w);
        else unit_forward(a, n, h, &w);
    }
    scratch_free(&w);
    return NULL;
}

static int run_pool(const kda_oracle_args *a, int backward)
{
    pool_t p;
    p.a = a;
    p.next = 0;
    p.backward = backward;
    pthread_mutex_init(&p.mu, NULL);
    int nt = a->nthreads > 0 ? a->nthreads : 1;
    if ((int64_t)nt > a->N * a->H) nt = (int)(a->N * a->H > 0 ? a->N * a->H : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, worker, &p);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&p.mu);
    return 0;
}

/* Forward: o (nullable) and hT (nullable). */
int kda_oracle_forward(const kda_oracle_args *a) { return run_pool(a, 0); }

/* Backward: every gradient of L = sum <o, dO> + <hT, dhT>. */
int kda_oracle_backward(const kda_oracle_args *a) { return run_pool(a, 1); }

size_t kda_oracle_args_size(void) { return sizeof(kda_oracle_args); }
