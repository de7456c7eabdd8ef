/*
 * Oracle for the Q-Delta / QED / EDA forwards, the Q-Delta backward and the decode
 * steps: plain fp64 sequential recurrences on the CPU.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the bench's
 * CPU-baseline / reference leg load this library.  It shares no code with the
 * CUDA path (no headers, helpers or tables) and the CUDA path never calls it.
 *
 * It computes the definition, not the chunked algorithm: one token at a time,
 * in the order the pages state the steps, with no blocking or reordering.
 *
 *  - Q-Delta, gated recurrence: "Q-Delta: Beyond Key-Value Associative State
 *    Evolution", Sec. 3.3.1, Eqs. 17-20 (the boxed gated form and the teaching
 *    pseudocode under it).  State S is d_v x d_k, output o_t = S_t q_t.
 *      x = k + lambda q;  S_prior = alpha S;  e = v - S_prior x;
 *      S = S_prior + beta e k^T;  o = S q.
 *    Absent alpha means 1 and absent lambda means 0 (Gated DeltaNet, DeltaNet).
 *    No 1+lambda normalisation of the residual (same section).
 *  - QED over GDN-2: "The Query Knows What to Forget", Sec. 2 Eqs. 4 and 8
 *    (GDN-2 update) and Sec. 3.1 Eq. 6 (erase vector).  State S is K x V,
 *    output o_t = S_t^T q_t.
 *      Sbar = Diag(exp g) S;  u = b*q;  d = u - k (k^T u);  a = b*k + lambda_h d;
 *      r = w*v - Sbar^T a;  S = Sbar + k r^T;  o = S^T q.
 *    d is formed with the given k as it is (the pages' projection assumes
 *    |k| = 1; no renormalisation is done here).
 *  - QED ablation arms: same page, Sec. 3.2 (Table 1), each a different term
 *    added to the base erase vector b*k:
 *      full          lambda_h P(b*q)          (the method above)
 *      nogate        lambda_h P(q)            (the gate b removed from the new term only)
 *      nogate-noproj lambda_h q               (no gate, no projection)
 *      rand          lambda_h P(b*z_h)        (z_h a fixed unit vector per head)
 *    with P(u) = u - k (k^T u).
 *  - Decode steps: one iteration of the Q-Delta or the QED loop per call, the
 *    state carried in and out in place.
 *  - Backward of the Q-Delta forward (and of the forward from projections, through the
 *    prologue's maps by the chain rule): the gradients of the scalar
 *    L = sum_t <dO_t, o_t> + <dS_final, S_T> with respect to q, k, v, alpha, beta,
 *    lambda and S0, by reverse-mode differentiation of the sequential recurrence
 *    above, one step at a time in reverse (the pages train the layer end to end,
 *    "Parallelizing Linear Transformers with the Delta Rule over Sequence Length",
 *    sec. 3, but print no backward; this is the adjoint of the stated forward).
 *    Rows of S evolve independently given a token's q, k and gates, so each row's
 *    states are recorded and walked back on their own; the row contributions to the
 *    shared gradients are summed.
 *  - EDA, erase-then-delta ("Erase-then-Delta Attention", core method, the two
 *    steps of its update): with the memory M (K x V), an erase direction e, then
 *    the Delta write along the key,
 *      M <- M - e (e^T M)                  (targeted erase; the printed "(e^T M) e" read
 *                                           as the outer product that fits the shapes)
 *      M <- M - beta k (k^T M - v^T)       (Delta write; the page's unit step is beta = 1)
 *      o = M^T q                           (read-out after both steps)
 *    Stored here as S = M^T ([dv][dk]): S <- S - (S e) e^T, S <- S - beta (S k - v) k^T,
 *    o = S q.  e is used as given (the page's default e = q/|q| is the caller's).
 *  - Prologue (the feature map and gates computed from the layer's projections):
 *    DeltaNet notes sec. 3.8, q = SiLU(x_q)/|SiLU(x_q)|_2 and the same for k,
 *    beta = sigmoid(x_beta); Q-Delta notes sec. 2.5 (App. B), lambda = sigmoid(x_lambda);
 *    the decay alpha = exp(-softplus(x_alpha)), the parameterisation of the
 *    workloads' decay gate.  Applied token by token, then the recurrence above.
 *
 * Storage of every state buffer, both methods: [B][H][d_v][d_k] row-major.  For
 * Q-Delta that is S itself; for QED it is S^T (QED's K x V state transposed), so
 * both share one format.  Token tensors are [B][T][H][d], gates [B][T][H],
 * QED's per-channel g, b [B][T][H][d_k] and w [B][T][H][d_v], lambda_h [H].
 *
 * Parity pins: see tests/test_oracle_pins.py (worked examples, closed forms,
 * special cases, brute force on tiny inputs).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int B, T, H, dk, dv;
    const double *q, *k, *v, *alpha, *beta, *lam;   /* Q-Delta gates */
    const double *g, *bgate, *w, *lam_h;            /* QED gates */
    int variant;                                     /* QED arm: 0 full, 1 nogate, 2 nogate-noproj, 3 rand */
    const double *z;                                 /* rand arm: z_h [H][dk] */
    const double *S0;
    double *o, *S_final;
    const double *dO, *dS_final;                     /* backward: incoming gradients */
    double *dq, *dk_out, *dv_out, *dalpha, *dbeta, *dlam, *dS0;
    int method;          /* 0 = Q-Delta, 1 = QED, 2 = Q-Delta backward, 3 = EDA */
    int first, stride;   /* this worker's (b,h) streams: first, first+stride, ... */
    int status;
} job_t;

/* One Q-Delta stream (b, h), t = 0..T-1. */
static int qdelta_stream(const job_t *J, int b, int h)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    double *S = malloc(sizeof(double) * (size_t)dv * dk);
    double *x = malloc(sizeof(double) * (size_t)dk);
    double *e = malloc(sizeof(double) * (size_t)dv);
    if (!S || !x || !e) { free(S); free(x); free(e); return 1; }
    const size_t sh = ((size_t)b * H + h) * dv * dk;
    if (J->S0) memcpy(S, J->S0 + sh, sizeof(double) * (size_t)dv * dk);
    else memset(S, 0, sizeof(double) * (size_t)dv * dk);

    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const double *qt = J->q + tok * dk, *kt = J->k + tok * dk, *vt = J->v + tok * dv;
        const double alpha = J->alpha ? J->alpha[tok] : 1.0;
        const double beta = J->beta[tok];
        const double lam = J->lam ? J->lam[tok] : 0.0;
        double *ot = J->o + tok * dv;

        for (int j = 0; j < dk; ++j) x[j] = kt[j] + lam * qt[j];          /* x = k + lambda q */
        for (size_t n = 0; n < (size_t)dv * dk; ++n) S[n] *= alpha;       /* S_prior = alpha S */
        for (int i = 0; i < dv; ++i) {                                     /* e = v - S_prior x */
            const double *Si = S + (size_t)i * dk;
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Si[j] * x[j];
            e[i] = vt[i] - acc;
        }
        for (int i = 0; i < dv; ++i) {                                     /* S += beta e k^T */
            double *Si = S + (size_t)i * dk;
            const double be = beta * e[i];
            for (int j = 0; j < dk; ++j) Si[j] += be * kt[j];
        }
        for (int i = 0; i < dv; ++i) {                                     /* o = S q */
            const double *Si = S + (size_t)i * dk;
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Si[j] * qt[j];
            ot[i] = acc;
        }
    }
    if (J->S_final) memcpy(J->S_final + sh, S, sizeof(double) * (size_t)dv * dk);
    free(S); free(x); free(e);
    return 0;
}

/* Backward of one Q-Delta stream (b, h).  For row i of S (s = S[i][:]):
 *   forward   sbar_t = alpha_t s_{t-1},  e_t = v_t[i] - sbar_t . x_t,
 *             s_t = sbar_t + beta_t e_t k_t,  o_t[i] = s_t . q_t
 *   adjoint   g = dL/ds_t, walked from t = T-1 down to 0:
 *             g += dO_t[i] q_t                       dq_t += dO_t[i] s_t
 *             ge = beta_t (g . k_t)  (dL/de_t)       dbeta_t += e_t (g . k_t)
 *             dk_t += beta_t e_t g                   dv_t[i] = ge
 *             gbar = g - ge x_t      (dL/dsbar_t)    dx = -ge sbar_t
 *             dk_t += dx,  dq_t += lambda_t dx,      dlambda_t += q_t . dx
 *             dalpha_t += gbar . s_{t-1}             g = alpha_t gbar
 *   and dS0[i] = g at the end. */
static int qdelta_bwd_stream(const job_t *J, int b, int h)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    double *hist = malloc(sizeof(double) * (size_t)(T + 1) * dk);   /* s_0 .. s_T of one row */
    double *x = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * dk);
    double *e = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *g = malloc(sizeof(double) * (size_t)dk), *gbar = malloc(sizeof(double) * (size_t)dk);
    if (!hist || !x || !e || !g || !gbar) { free(hist); free(x); free(e); free(g); free(gbar); return 1; }
    const size_t sh = ((size_t)b * H + h) * dv * dk;

    for (int t = 0; t < T; ++t) {                                         /* x_t = k_t + lambda_t q_t */
        const size_t tok = ((size_t)b * T + t) * H + h;
        const double lam = J->lam ? J->lam[tok] : 0.0;
        for (int j = 0; j < dk; ++j) x[(size_t)t * dk + j] = J->k[tok * dk + j] + lam * J->q[tok * dk + j];
    }
    for (int i = 0; i < dv; ++i) {
        /* forward, recording this row's states */
        for (int j = 0; j < dk; ++j) hist[j] = J->S0 ? J->S0[sh + (size_t)i * dk + j] : 0.0;
        for (int t = 0; t < T; ++t) {
            const size_t tok = ((size_t)b * T + t) * H + h;
            const double alpha = J->alpha ? J->alpha[tok] : 1.0;
            const double *sp = hist + (size_t)t * dk, *xt = x + (size_t)t * dk, *kt = J->k + tok * dk;
            double *sn = hist + (size_t)(t + 1) * dk;
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += alpha * sp[j] * xt[j];
            e[t] = J->v[tok * dv + i] - acc;
            for (int j = 0; j < dk; ++j) sn[j] = alpha * sp[j] + J->beta[tok] * e[t] * kt[j];
        }
        /* adjoint, t = T-1 .. 0 */
        for (int j = 0; j < dk; ++j) g[j] = J->dS_final ? J->dS_final[sh + (size_t)i * dk + j] : 0.0;
        for (int t = T - 1; t >= 0; --t) {
            const size_t tok = ((size_t)b * T + t) * H + h;
            const double alpha = J->alpha ? J->alpha[tok] : 1.0;
            const double beta = J->beta[tok];
            const double lam = J->lam ? J->lam[tok] : 0.0;
            const double *qt = J->q + tok * dk, *kt = J->k + tok * dk, *xt = x + (size_t)t * dk;
            const double *sp = hist + (size_t)t * dk, *sn = hist + (size_t)(t + 1) * dk;
            double *dqt = J->dq + tok * dk, *dkt = J->dk_out + tok * dk;
            const double dot = J->dO[tok * dv + i];
            for (int j = 0; j < dk; ++j) {                                /* o_t[i] = s_t . q_t */
                g[j] += dot * qt[j];
                dqt[j] += dot * sn[j];
            }
            double gk = 0.0;
            for (int j = 0; j < dk; ++j) gk += g[j] * kt[j];
            const double ge = beta * gk;                                  /* s_t = sbar + beta e k */
            J->dbeta[tok] += e[t] * gk;
            for (int j = 0; j < dk; ++j) dkt[j] += beta * e[t] * g[j];
            J->dv_out[tok * dv + i] = ge;                                 /* e = v - sbar . x */
            double dlam = 0.0, dal = 0.0;
            for (int j = 0; j < dk; ++j) {
                gbar[j] = g[j] - ge * xt[j];
                const double dx = -ge * alpha * sp[j];
                dkt[j] += dx;                                             /* x = k + lambda q */
                dqt[j] += lam * dx;
                dlam += qt[j] * dx;
                dal += gbar[j] * sp[j];                                   /* sbar = alpha s_{t-1} */
            }
            if (J->dlam) J->dlam[tok] += dlam;
            if (J->dalpha) J->dalpha[tok] += dal;
            for (int j = 0; j < dk; ++j) g[j] = alpha * gbar[j];
        }
        if (J->dS0) for (int j = 0; j < dk; ++j) J->dS0[sh + (size_t)i * dk + j] = g[j];
    }
    free(hist); free(x); free(e); free(g); free(gbar);
    return 0;
}

/* One EDA stream (b, h), S = M^T in [dv][dk]; J->g holds e [B][T][H][dk] and
 * J->beta the write strength (NULL = 1). */
static int eda_stream(const job_t *J, int b, int h)
{
    const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    double *S = malloc(sizeof(double) * (size_t)dv * dk);
    if (!S) return 1;
    const size_t sh = ((size_t)b * H + h) * dv * dk;
    if (J->S0) memcpy(S, J->S0 + sh, sizeof(double) * (size_t)dv * dk);
    else memset(S, 0, sizeof(double) * (size_t)dv * dk);
    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const double *qt = J->q + tok * dk, *kt = J->k + tok * dk, *et = J->g + tok * dk, *vt = J->v + tok * dv;
        const double beta = J->beta ? J->beta[tok] : 1.0;
        for (int i = 0; i < dv; ++i) {
            double *Si = S + (size_t)i * dk;
            double p = 0.0;                                                /* erase: (S e)_i */
            for (int j = 0; j < dk; ++j) p += Si[j] * et[j];
            for (int j = 0; j < dk; ++j) Si[j] -= p * et[j];
            double r = -vt[i];                                             /* write: (S k - v)_i */
            for (int j = 0; j < dk; ++j) r += Si[j] * kt[j];
            for (int j = 0; j < dk; ++j) Si[j] -= beta * r * kt[j];
            double acc = 0.0;                                              /* o = S q */
            for (int j = 0; j < dk; ++j) acc += Si[j] * qt[j];
            J->o[tok * dv + i] = acc;
        }
    }
    if (J->S_final) memcpy(J->S_final + sh, S, sizeof(double) * (size_t)dv * dk);
    free(S);
    return 0;
}

/* One QED stream (b, h).  S is held K x V here (S[c*dv + j], c over keys). */
static int qed_stream(const job_t *J, int b, int h)
{
    const int T = J->T, H = J->H, K = J->dk, V = J->dv;
    double *S = malloc(sizeof(double) * (size_t)K * V);
    double *u = malloc(sizeof(double) * (size_t)K);
    double *a = malloc(sizeof(double) * (size_t)K);
    double *r = malloc(sizeof(double) * (size_t)V);
    if (!S || !u || !a || !r) { free(S); free(u); free(a); free(r); return 1; }
    const size_t sh = ((size_t)b * H + h) * K * V;
    for (int c = 0; c < K; ++c)                   /* stored [V][K] = S^T -> S[c][j] */
        for (int j = 0; j < V; ++j)
            S[(size_t)c * V + j] = J->S0 ? J->S0[sh + (size_t)j * K + c] : 0.0;
    const double lam_h = J->lam_h[h];

    for (int t = 0; t < T; ++t) {
        const size_t tok = ((size_t)b * T + t) * H + h;
        const double *qt = J->q + tok * K, *kt = J->k + tok * K, *vt = J->v + tok * V;
        const double *gt = J->g + tok * K, *bt = J->bgate + tok * K, *wt = J->w + tok * V;
        double *ot = J->o + tok * V;

        for (int c = 0; c < K; ++c) {                                      /* Sbar = Diag(exp g) S */
            const double dc = exp(gt[c]);
            double *Sc = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) Sc[j] *= dc;
        }
        /* the new term's input: b*q (full), q (nogate, nogate-noproj), b*z_h (rand) */
        const double *zh = J->variant == 3 ? J->z + (size_t)h * K : NULL;
        double ku = 0.0;
        for (int c = 0; c < K; ++c) {
            const double x = zh ? zh[c] : qt[c];
            u[c] = (J->variant == 1 || J->variant == 2) ? x : bt[c] * x;
            ku += kt[c] * u[c];                                            /* k^T u */
        }
        for (int c = 0; c < K; ++c) {
            const double d = J->variant == 2 ? u[c] : u[c] - kt[c] * ku;   /* d = u - k (k^T u) */
            a[c] = bt[c] * kt[c] + lam_h * d;                              /* a = b*k + lambda_h d */
        }
        for (int j = 0; j < V; ++j) {                                      /* r = w*v - Sbar^T a */
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += S[(size_t)c * V + j] * a[c];
            r[j] = wt[j] * vt[j] - acc;
        }
        for (int c = 0; c < K; ++c) {                                      /* S = Sbar + k r^T */
            double *Sc = S + (size_t)c * V;
            for (int j = 0; j < V; ++j) Sc[j] += kt[c] * r[j];
        }
        for (int j = 0; j < V; ++j) {                                      /* o = S^T q */
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += S[(size_t)c * V + j] * qt[c];
            ot[j] = acc;
        }
    }
    if (J->S_final)
        for (int c = 0; c < K; ++c)
            for (int j = 0; j < V; ++j)
                J->S_final[sh + (size_t)j * K + c] = S[(size_t)c * V + j];
    free(S); free(u); free(a); free(r);
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int n = J->B * J->H;
    for (int s = J->first; s < n; s += J->stride) {
        const int b = s / J->H, h = s % J->H;
        int rc = J->method == 0 ? qdelta_stream(J, b, h)
               : J->method == 1 ? qed_stream(J, b, h)
               : J->method == 2 ? qdelta_bwd_stream(J, b, h) : eda_stream(J, b, h);
        if (rc) J->status = rc;
    }
    return NULL;
}

/* Runs the streams of one call over `nthreads` threads (<= 0: all cores). */
static int run(job_t *proto, int nthreads)
{
    const int n = proto->B * proto->H;
    if (n <= 0 || proto->T < 0) return 0;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = n;
    job_t *jobs = calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    int status = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].first = i;
        jobs[i].stride = nthreads;
        jobs[i].status = 0;
        if (i > 0 && pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) {
            worker(&jobs[i]);          /* could not spawn: run inline */
            th[i] = 0;
        }
    }
    worker(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (th[i]) pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].status) status = jobs[i].status;
    free(jobs); free(th);
    return status;
}

/* Q-Delta forward.  alpha, lam, S0, S_final may be NULL.  Returns 0 on success. */
int oracle_qdelta_fwd(int B, int T, int H, int dk, int dv,
                      const double *q, const double *k, const double *v,
                      const double *alpha, const double *beta, const double *lam,
                      const double *S0, double *o, double *S_final, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.beta = beta; J.lam = lam;
    J.S0 = S0; J.o = o; J.S_final = S_final; J.method = 0;
    return run(&J, nthreads);
}

/* Q-Delta backward.  dO [B][T][H][dv]; dS_final [B][H][dv][dk] or NULL (= 0).
 * Gradients: dq, dk [B][T][H][dk], dv [B][T][H][dv], dalpha, dbeta, dlam [B][T][H],
 * dS0 [B][H][dv][dk].  dalpha (dlam) must be NULL when alpha (lam) is NULL and is
 * then not computed; dS0 may be NULL.  All outputs are overwritten. */
int oracle_qdelta_bwd(int B, int T, int H, int dk, int dv,
                      const double *q, const double *k, const double *v,
                      const double *alpha, const double *beta, const double *lam, const double *S0,
                      const double *dO, const double *dS_final,
                      double *dq, double *dk_out, double *dv_out, double *dalpha, double *dbeta,
                      double *dlam, double *dS0, int nthreads)
{
    if ((dalpha && !alpha) || (dlam && !lam)) return 2;
    const size_t nt = (size_t)B * T * H;
    memset(dq, 0, sizeof(double) * nt * dk);
    memset(dk_out, 0, sizeof(double) * nt * dk);
    memset(dv_out, 0, sizeof(double) * nt * dv);
    memset(dbeta, 0, sizeof(double) * nt);
    if (dalpha) memset(dalpha, 0, sizeof(double) * nt);
    if (dlam) memset(dlam, 0, sizeof(double) * nt);
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.beta = beta; J.lam = lam; J.S0 = S0;
    J.dO = dO; J.dS_final = dS_final;
    J.dq = dq; J.dk_out = dk_out; J.dv_out = dv_out; J.dalpha = dalpha; J.dbeta = dbeta; J.dlam = dlam;
    J.dS0 = dS0; J.method = 2;
    return run(&J, nthreads);
}

/* EDA forward: q, k, e [B][T][H][dk], v [B][T][H][dv], beta [B][T][H] or NULL (= 1),
 * S0, S_final [B][H][dv][dk] (M^T) or NULL. */
int oracle_eda_fwd(int B, int T, int H, int dk, int dv,
                   const double *q, const double *k, const double *v, const double *e, const double *beta,
                   const double *S0, double *o, double *S_final, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.g = e; J.beta = beta;
    J.S0 = S0; J.o = o; J.S_final = S_final; J.method = 3;
    return run(&J, nthreads);
}

/* QED forward over GDN-2.  S0, S_final may be NULL; stored as [B][H][dv][dk]. */
int oracle_qed_fwd(int B, int T, int H, int dk, int dv,
                   const double *q, const double *k, const double *v,
                   const double *g, const double *b, const double *w, const double *lam_h,
                   const double *S0, double *o, double *S_final, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.g = g; J.bgate = b; J.w = w; J.lam_h = lam_h;
    J.S0 = S0; J.o = o; J.S_final = S_final; J.method = 1;
    return run(&J, nthreads);
}

/* QED forward for one of the ablation arms (variant 0 full, 1 nogate,
 * 2 nogate-noproj, 3 rand with z_h [H][dk]).  Variant 0 is oracle_qed_fwd. */
int oracle_qed_fwd_variant(int B, int T, int H, int dk, int dv,
                           const double *q, const double *k, const double *v,
                           const double *g, const double *b, const double *w, const double *lam_h,
                           int variant, const double *z, const double *S0, double *o, double *S_final,
                           int nthreads)
{
    if (variant < 0 || variant > 3 || (variant == 3 && !z)) return 2;
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.g = g; J.bgate = b; J.w = w; J.lam_h = lam_h;
    J.variant = variant; J.z = z;
    J.S0 = S0; J.o = o; J.S_final = S_final; J.method = 1;
    return run(&J, nthreads);
}

/* The prologue for one token-head: q = SiLU(x)/|SiLU(x)|, sigmoid and
 * exp(-softplus) gates.  The norm of an all-zero SiLU row is taken as 1. */
static void feature_map(const double *x, double *y, int d)
{
    double ss = 0.0;
    for (int j = 0; j < d; ++j) {
        y[j] = x[j] / (1.0 + exp(-x[j]));                  /* SiLU(x) = x sigmoid(x) */
        ss += y[j] * y[j];
    }
    const double inv = ss > 0.0 ? 1.0 / sqrt(ss) : 1.0;
    for (int j = 0; j < d; ++j) y[j] *= inv;
}
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double exp_neg_softplus(double x) { return exp(-log1p(exp(x))); }

/* Q-Delta forward from the layer's projections: q_raw, k_raw [B][T][H][dk] go
 * through the feature map, the gate logits [B][T][H] through their gates (NULL
 * alpha / lambda logits: alpha = 1 / lambda = 0), then oracle_qdelta_fwd. */
int oracle_qdelta_fwd_prologue(int B, int T, int H, int dk, int dv,
                               const double *q_raw, const double *k_raw, const double *v,
                               const double *a_logit, const double *b_logit, const double *l_logit,
                               const double *S0, double *o, double *S_final, int nthreads)
{
    const size_t nt = (size_t)B * T * H;
    double *q = malloc(sizeof(double) * nt * dk), *k = malloc(sizeof(double) * nt * dk);
    double *al = a_logit ? malloc(sizeof(double) * nt) : NULL, *be = malloc(sizeof(double) * nt);
    double *lm = l_logit ? malloc(sizeof(double) * nt) : NULL;
    int rc = 1;
    if (q && k && be && (!a_logit || al) && (!l_logit || lm)) {
        for (size_t i = 0; i < nt; ++i) {
            feature_map(q_raw + i * dk, q + i * dk, dk);
            feature_map(k_raw + i * dk, k + i * dk, dk);
            be[i] = sigmoid(b_logit[i]);
            if (al) al[i] = exp_neg_softplus(a_logit[i]);
            if (lm) lm[i] = sigmoid(l_logit[i]);
        }
        rc = oracle_qdelta_fwd(B, T, H, dk, dv, q, k, v, al, be, lm, S0, o, S_final, nthreads);
    }
    free(q); free(k); free(al); free(be); free(lm);
    return rc;
}

/* Backward through the prologue's feature map for one token-head row: with
 * s = SiLU(x), n = |s|, y = s / n and the incoming gradient dy, the gradient of x is
 *     ds = (dy - y (y . dy)) / n,   dx = ds * SiLU'(x),  SiLU'(x) = sig(x) (1 + x (1 - sig(x))).
 * An all-zero s (where the forward leaves y = 0) passes no gradient. */
static void feature_map_bwd(const double *x, const double *dy, double *dx, int d)
{
    double ss = 0.0, ydy = 0.0;
    for (int j = 0; j < d; ++j) {
        const double sj = x[j] * sigmoid(x[j]);
        ss += sj * sj;
    }
    if (!(ss > 0.0)) { for (int j = 0; j < d; ++j) dx[j] = 0.0; return; }
    const double n = sqrt(ss);
    for (int j = 0; j < d; ++j) ydy += (x[j] * sigmoid(x[j]) / n) * dy[j];
    for (int j = 0; j < d; ++j) {
        const double sg = sigmoid(x[j]), y = x[j] * sg / n;
        dx[j] = (dy[j] - y * ydy) / n * (sg * (1.0 + x[j] * (1.0 - sg)));
    }
}

/* Backward of oracle_qdelta_fwd_prologue: the inputs through the prologue, the
 * recurrence's backward (oracle_qdelta_bwd) on them, then the chain rule back through
 * the prologue: dq_raw, dk_raw by feature_map_bwd, d b_logit = dbeta beta (1 - beta),
 * d l_logit = dlam lam (1 - lam), d a_logit = -dalpha alpha (1 - alpha) (alpha =
 * exp(-softplus(a)) = sigmoid(-a)).  Outputs as oracle_qdelta_bwd with the logits'
 * gradients in place of the gates'. */
int oracle_qdelta_bwd_prologue(int B, int T, int H, int dk, int dv,
                               const double *q_raw, const double *k_raw, const double *v,
                               const double *a_logit, const double *b_logit, const double *l_logit,
                               const double *S0, const double *dO, const double *dS_final,
                               double *dq_raw, double *dk_raw, double *dv_out, double *da_logit,
                               double *db_logit, double *dl_logit, double *dS0, int nthreads)
{
    if ((da_logit && !a_logit) || (dl_logit && !l_logit)) return 2;
    const size_t nt = (size_t)B * T * H;
    double *q = malloc(sizeof(double) * nt * dk), *k = malloc(sizeof(double) * nt * dk);
    double *dq = malloc(sizeof(double) * nt * dk), *dkk = malloc(sizeof(double) * nt * dk);
    double *al = a_logit ? malloc(sizeof(double) * nt) : NULL, *be = malloc(sizeof(double) * nt);
    double *lm = l_logit ? malloc(sizeof(double) * nt) : NULL;
    double *dal = a_logit ? malloc(sizeof(double) * nt) : NULL, *dbe = malloc(sizeof(double) * nt);
    double *dlm = l_logit ? malloc(sizeof(double) * nt) : NULL;
    int rc = 1;
    if (q && k && dq && dkk && be && dbe && (!a_logit || (al && dal)) && (!l_logit || (lm && dlm))) {
        for (size_t i = 0; i < nt; ++i) {
            feature_map(q_raw + i * dk, q + i * dk, dk);
            feature_map(k_raw + i * dk, k + i * dk, dk);
            be[i] = sigmoid(b_logit[i]);
            if (al) al[i] = exp_neg_softplus(a_logit[i]);
            if (lm) lm[i] = sigmoid(l_logit[i]);
        }
        rc = oracle_qdelta_bwd(B, T, H, dk, dv, q, k, v, al, be, lm, S0, dO, dS_final, dq, dkk, dv_out,
                               dal, dbe, dlm, dS0, nthreads);
        if (!rc)
            for (size_t i = 0; i < nt; ++i) {
                feature_map_bwd(q_raw + i * dk, dq + i * dk, dq_raw + i * dk, dk);
                feature_map_bwd(k_raw + i * dk, dkk + i * dk, dk_raw + i * dk, dk);
                db_logit[i] = dbe[i] * be[i] * (1.0 - be[i]);
                if (da_logit) da_logit[i] = -dal[i] * al[i] * (1.0 - al[i]);
                if (dl_logit) dl_logit[i] = dlm[i] * lm[i] * (1.0 - lm[i]);
            }
    }
    free(q); free(k); free(dq); free(dkk); free(al); free(be); free(lm); free(dal); free(dbe); free(dlm);
    return rc;
}

/* One QED decode step for N sequences x H heads: S [N][H][dv][dk] (QED's state
 * transposed) updated in place, tokens [N][H][d], g, b [N][H][dk], w [N][H][dv],
 * lambda_h [H], o [N][H][dv]; the T = 1 case of the forward. */
int oracle_qed_step(int N, int H, int dk, int dv, double *S,
                    const double *q, const double *k, const double *v,
                    const double *g, const double *b, const double *w, const double *lam_h,
                    int variant, const double *z, double *o, int nthreads)
{
    return oracle_qed_fwd_variant(N, 1, H, dk, dv, q, k, v, g, b, w, lam_h, variant, z, S, o, S, nthreads);
}

/* One Q-Delta decode step for N sequences x H heads: S [N][H][dv][dk] updated in
 * place, tokens [N][H][d], gates [N][H] (alpha, lam may be NULL), o [N][H][dv].
 * It is the T = 1 case of the forward, with the state carried in and out. */
int oracle_qdelta_step(int N, int H, int dk, int dv, double *S,
                       const double *q, const double *k, const double *v,
                       const double *alpha, const double *beta, const double *lam,
                       double *o, int nthreads)
{
    return oracle_qdelta_fwd(N, 1, H, dk, dv, q, k, v, alpha, beta, lam, S, o, S, nthreads);
}
