/*
 * fp64 CPU oracle for the forward pass of causal gated linear attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition, the gated recurrence
 *     S_t = Diag(alpha_t) S_{t-1} + k_t^T v_t,      o_t = q_t S_t,
 * ("Gated Linear Attention Transformers with Hardware-Efficient Training",
 * §4.1 Eq. 3; the ungated case alpha = 1 is §2.1 Eq. 1; the fixed per-head
 * decay alpha = lambda_h is the recurrence "Lightning Attention-2" §3.2.1
 * starts from). S_0 is zero or a caller-given state carried from a previous
 * segment (same GLA paper, §2.2, below Eq. 2). The chunkwise method of
 * §4.2-4.3 reaches exactly this result (up to rounding order), so the
 * oracle is the token-by-token recurrence itself, one token at a time, with
 * no chunking, blocking or reordering.
 *
 * Gate modes (alpha_t in (0,1]^dk is given as log alpha_t):
 *   0  alpha_t = 1                         (log_g unused)
 *   1  alpha_t = exp(log_g[h]) for all t,k (log_g is [H])
 *   2  alpha_t = exp(log_g[b,h,t,:])       (log_g is [B,H,T,dk])
 *   3  alpha_t = exp(log_g[b,h,t]) for all k (log_g is [B,H,T]): the
 *      data-dependent scalar gate G_t = gamma_t 1^T 1 of the Mamba-2, mLSTM
 *      and Gated Retention rows of Table 1 (GLA paper, §4.1)
 *   4  the bilinear gate G_t = alpha_t^T beta_t of Table 1's DFW row: the state
 *      update is S_t[i][j] = alpha_t[i] beta_t[j] S_{t-1}[i][j] + k_t[i] v_t[j]
 *      with alpha_t = exp(log_g[b,h,t,:]) ([B,H,T,dk]) and
 *      beta_t = exp(log_b[b,h,t,:]) ([B,H,T,dv])
 *
 * Layouts (row-major, contiguous): q [B,H,T,dk], k [B,H,T,dk], v [B,H,T,dv],
 * O [B,H,T,dv], S0 and ST [B,H,dk,dv]. S0 may be NULL (zero state); ST may be
 * NULL (not written).
 *
 * Parallelism: the columns j of S evolve independently (the gate scales the
 * rows i of S only), so work is split over (b, h, column block) with POSIX
 * threads. The arithmetic per column is unchanged by the split.
 *
 * "mutant" plants one deliberate mistake so that the tests can show the
 * pins catch it. It is 0 everywhere except in those tests:
 *   1  decay applied after the update:  S_t = Diag(a_t)(S_{t-1} + k^T v)
 *   2  output read before the update:    o_t = q_t S_{t-1}
 *   3  gate applied to the columns j instead of the rows i (needs dk == dv)
 *   4  gate taken one step late:          alpha_{t-1} used at step t
 *   5  S_0 ignored
 *   6  q and k exchanged
 *   7  diagonal (current-token) term dropped from the output
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *log_g, *log_b, *S0;
    double *O, *ST;
    long B, H, T, dk, dv;
    int gate, mutant;
    long j0, j1; /* column block [j0, j1) */
    long bh;     /* flattened (b, h) */
    int status;
} job_t;

static double gate_alpha(const job_t* J, long t, long i)
{
    if (J->gate == 0) return 1.0;
    if (J->gate == 1) return exp(J->log_g[J->bh % J->H]);
    if (J->gate == 3) return exp(J->log_g[J->bh * J->T + t]);
    return exp(J->log_g[(J->bh * J->T + t) * J->dk + i]);
}

static void run_job(job_t* J)
{
    const long dk = J->dk, dv = J->dv, T = J->T, w = J->j1 - J->j0;
    double* S = (double*)calloc((size_t)(dk * w), sizeof(double));
    double* Sprev = (J->mutant == 2 || J->mutant == 7) ? (double*)calloc((size_t)(dk * w), sizeof(double)) : NULL;
    double* alpha = (double*)malloc((size_t)dk * sizeof(double));
    double* beta = (double*)malloc((size_t)w * sizeof(double));
    if (!S || !alpha || !beta || ((J->mutant == 2 || J->mutant == 7) && !Sprev)) {
        J->status = 1;
        free(S); free(Sprev); free(alpha); free(beta);
        return;
    }
    const double* q = J->q + J->bh * T * dk;
    const double* k = J->k + J->bh * T * dk;
    const double* v = J->v + J->bh * T * dv;
    double* O = J->O + J->bh * T * dv;
    if (J->mutant == 6) { const double* tmp = q; q = k; k = tmp; }

    /* S <- S_0 (or zero) */
    if (J->S0 && J->mutant != 5) {
        const double* s0 = J->S0 + J->bh * dk * dv;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < w; ++j) S[i * w + j] = s0[i * dv + J->j0 + j];
    }

    for (long t = 0; t < T; ++t) {
        /* alpha_t (one value per row i of S) */
        long tg = (J->mutant == 4) ? (t > 0 ? t - 1 : 0) : t;
        for (long i = 0; i < dk; ++i) alpha[i] = gate_alpha(J, tg, i);
        if (J->mutant == 4 && t == 0)
            for (long i = 0; i < dk; ++i) alpha[i] = 1.0;
        /* beta_t (one value per column j of S; 1 unless the gate is bilinear) */
        for (long j = 0; j < w; ++j)
            beta[j] = (J->gate == 4) ? exp(J->log_b[(J->bh * T + t) * dv + J->j0 + j]) : 1.0;
        if (Sprev) memcpy(Sprev, S, (size_t)(dk * w) * sizeof(double));

        const double* kt = k + t * dk;
        const double* vt = v + t * dv + J->j0;
        const double* qt = q + t * dk;
        double* ot = O + t * dv + J->j0;
        for (long j = 0; j < w; ++j) ot[j] = 0.0;

        for (long i = 0; i < dk; ++i) {
            double* Si = S + i * w;
            const double a = alpha[i], ki = kt[i], qi = qt[i];
            if (J->mutant == 1) {
                for (long j = 0; j < w; ++j) Si[j] = a * (Si[j] + ki * vt[j]);
            } else if (J->mutant == 3) {
                /* gate indexed by the column instead of the row */
                for (long j = 0; j < w; ++j) Si[j] = alpha[J->j0 + j] * Si[j] + ki * vt[j];
            } else if (J->gate == 4) {
                /* S_t[i][j] = alpha_t[i] beta_t[j] S_{t-1}[i][j] + k_t[i] v_t[j] */
                for (long j = 0; j < w; ++j) Si[j] = a * beta[j] * Si[j] + ki * vt[j];
            } else {
                /* Eq. 3: S_t[i][j] = alpha_t[i] * S_{t-1}[i][j] + k_t[i] * v_t[j] */
                for (long j = 0; j < w; ++j) Si[j] = a * Si[j] + ki * vt[j];
            }
            if (J->mutant == 2) {
                const double* Pi = Sprev + i * w;
                for (long j = 0; j < w; ++j) ot[j] += qi * Pi[j];
            } else if (J->mutant == 7) {
                /* q_t (Diag(alpha_t) S_{t-1}): the k_t^T v_t term left out */
                const double* Pi = Sprev + i * w;
                for (long j = 0; j < w; ++j) ot[j] += qi * a * beta[j] * Pi[j];
            } else {
                /* o_t[j] = sum_i q_t[i] * S_t[i][j] */
                for (long j = 0; j < w; ++j) ot[j] += qi * Si[j];
            }
        }
    }

    if (J->ST) {
        double* st = J->ST + J->bh * dk * dv;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < w; ++j) st[i * dv + J->j0 + j] = S[i * w + j];
    }
    free(S); free(Sprev); free(alpha); free(beta);
}

typedef struct {
    job_t* jobs;
    long njobs;
    long next;
    pthread_mutex_t mu;
} pool_t;

static void* worker(void* arg)
{
    pool_t* P = (pool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&P->mu);
        long idx = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (idx >= P->njobs) break;
        run_job(&P->jobs[idx]);
    }
    return NULL;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure. */
int gla_oracle_fwd(const double* q, const double* k, const double* v,
                   const double* log_g, const double* log_b, int gate, const double* S0,
                   double* O, double* ST,
                   long B, long H, long T, long dk, long dv,
                   int nthreads, int mutant)
{
    if (!q || !k || !v || !O || B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return 1;
    if (gate < 0 || gate > 4 || (gate != 0 && !log_g) || (gate == 4 && !log_b)) return 1;
    if (mutant == 3 && dk != dv) return 1;
    if (T == 0) {
        if (ST) {
            for (long i = 0; i < B * H * dk * dv; ++i) ST[i] = (S0 && mutant != 5) ? S0[i] : 0.0;
        }
        return 0;
    }
    /* Column blocks: small enough to spread over threads, large enough to
       keep the inner loops long. Mutant 3 reads alpha by absolute column, so
       it uses one block. */
    long jb = (mutant == 3) ? dv : (dv >= 64 ? 64 : dv);
    long nblk = (dv + jb - 1) / jb;
    long njobs = B * H * nblk;
    job_t* jobs = (job_t*)calloc((size_t)njobs, sizeof(job_t));
    if (!jobs) return 2;
    for (long bh = 0; bh < B * H; ++bh)
        for (long c = 0; c < nblk; ++c) {
            job_t* J = &jobs[bh * nblk + c];
            J->q = q; J->k = k; J->v = v; J->log_g = log_g; J->log_b = log_b; J->S0 = S0;
            J->O = O; J->ST = ST;
            J->B = B; J->H = H; J->T = T; J->dk = dk; J->dv = dv;
            J->gate = gate; J->mutant = mutant;
            J->bh = bh; J->j0 = c * jb; J->j1 = (c + 1) * jb < dv ? (c + 1) * jb : dv;
        }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > njobs) nthreads = (int)njobs;
    pool_t P;
    P.jobs = jobs; P.njobs = njobs; P.next = 0;
    pthread_mutex_init(&P.mu, NULL);
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    int started = 0;
    if (th) {
        for (int i = 0; i + 1 < nthreads; ++i)
            if (pthread_create(&th[started], NULL, worker, &P) == 0) ++started;
    }
    worker(&P); /* the calling thread works too */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&P.mu);
    int st = 0;
    for (long i = 0; i < njobs; ++i) if (jobs[i].status) st = 2;
    free(jobs);
    return st;
}

/* ---------------------------------------------------------------- backward
 *
 * Gradients of a scalar loss L through the recurrence, given dO = dL/dO and
 * dST = dL/dS_T (NULL: zero). This is reverse-mode differentiation of Eq. 3
 * written out as the adjoint recurrence, with D_t = dL/dS_t counting every
 * later use of S_t:
 *   D_{T-1} = dST + q_{T-1}^T do_{T-1},
 *   D_t     = Diag(alpha_{t+1}) D_{t+1} + q_t^T do_t,
 *   dq_t = S_t do_t^T,   dk_t = D_t v_t^T,   dv_t = k_t D_t,
 *   dlog alpha_t[i] = alpha_t[i] sum_j D_t[i][j] S_{t-1}[i][j],
 *   dS0 = Diag(alpha_0) D_0.
 * Per gate mode, the gradient of log_g is dlog alpha itself (per key), its
 * sum over keys (per token) or its sum over keys, tokens and batch rows (per
 * head). S_{t-1} is needed in reverse order: the states at every CK-th step
 * are kept and the ones between recomputed from them by the same forward
 * steps, so every value is the one a run storing all states would use.
 *
 * The bilinear gate (mode 4, S_t = Diag(alpha_t) S_{t-1} Diag(beta_t) + k_t^T v_t)
 * decays D by both factors, D_t = Diag(alpha_{t+1}) D_{t+1} Diag(beta_{t+1}) + q_t^T do_t,
 * dS0 = Diag(alpha_0) D_0 Diag(beta_0), and adds
 *   dlog alpha_t[i] = alpha_t[i] sum_j D_t[i][j] beta_t[j] S_{t-1}[i][j],
 *   dlog beta_t[j]  = beta_t[j]  sum_i D_t[i][j] alpha_t[i] S_{t-1}[i][j].
 *
 * Backward mutants (tests only): 11 dlog alpha without the factor alpha_t;
 * 12 D decayed before q_t^T do_t is added; 13 dq_t read from S_{t-1};
 * 14 the decay of D skipped at t = 0 (dS0 = D_0); 15 dlog beta without the
 * factor beta_t; 16 D decayed by alpha only (beta left out).
 */
typedef struct {
    const double *q, *k, *v, *log_g, *log_b, *S0, *dO, *dST;
    double *gq, *gk, *gv, *dlg, *dlb, *dS0; /* dlg: [T][dk] dlog alpha, dlb: [T][dv] dlog beta of this (b, h) */
    long H, T, dk, dv, bh;
    int gate, mutant, status;
} bjob_t;

static double bgate(const bjob_t* J, long t, long i)
{
    if (J->gate == 0) return 1.0;
    if (J->gate == 1) return exp(J->log_g[J->bh % J->H]);
    if (J->gate == 3) return exp(J->log_g[J->bh * J->T + t]);
    return exp(J->log_g[(J->bh * J->T + t) * J->dk + i]);
}

/* beta_t[j] of the bilinear gate, 1 in every other mode */
static double bbeta(const bjob_t* J, long t, long j)
{
    return J->gate == 4 ? exp(J->log_b[(J->bh * J->T + t) * J->dv + j]) : 1.0;
}

/* S_out = Diag(alpha_t) S_in Diag(beta_t) + k_t^T v_t (Eq. 3), full width dv */
static void bstep(const bjob_t* J, long t, const double* Sin, double* Sout)
{
    const long dk = J->dk, dv = J->dv;
    const double* kt = J->k + (J->bh * J->T + t) * dk;
    const double* vt = J->v + (J->bh * J->T + t) * dv;
    for (long i = 0; i < dk; ++i) {
        const double a = bgate(J, t, i), ki = kt[i];
        for (long j = 0; j < dv; ++j) Sout[i * dv + j] = a * bbeta(J, t, j) * Sin[i * dv + j] + ki * vt[j];
    }
}

/* D <- Diag(alpha_t) D Diag(beta_t) (mutant 16: alpha only) */
static void bdecay(const bjob_t* J, long t, double* D)
{
    const long dk = J->dk, dv = J->dv;
    for (long i = 0; i < dk; ++i) {
        const double a = bgate(J, t, i);
        for (long j = 0; j < dv; ++j) D[i * dv + j] *= a * (J->mutant == 16 ? 1.0 : bbeta(J, t, j));
    }
}

static void bwd_job(bjob_t* J)
{
    const long dk = J->dk, dv = J->dv, T = J->T, n = dk * dv;
    long CK = 64;
    while (CK * CK < T) CK *= 2;
    const long nck = (T + CK - 1) / CK;
    double* ck = (double*)malloc((size_t)(nck > 0 ? nck : 1) * n * sizeof(double));
    double* blk = (double*)malloc((size_t)(CK + 1) * n * sizeof(double));
    double* D = (double*)malloc((size_t)n * sizeof(double));
    double* S = (double*)malloc((size_t)n * sizeof(double));
    double* S2 = (double*)malloc((size_t)n * sizeof(double));
    if (!ck || !blk || !D || !S || !S2) {
        J->status = 1;
        free(ck); free(blk); free(D); free(S); free(S2);
        return;
    }
    /* forward, keeping the state entering every CK-th step */
    for (long e = 0; e < n; ++e) S[e] = J->S0 ? J->S0[J->bh * n + e] : 0.0;
    for (long t = 0; t < T; ++t) {
        if (t % CK == 0) memcpy(ck + (t / CK) * n, S, (size_t)n * sizeof(double));
        bstep(J, t, S, S2);
        double* tmp = S; S = S2; S2 = tmp;
    }
    /* reverse */
    for (long e = 0; e < n; ++e) D[e] = J->dST ? J->dST[J->bh * n + e] : 0.0;
    for (long c = nck - 1; c >= 0; --c) {
        const long t0 = c * CK, t1 = (t0 + CK < T) ? t0 + CK : T;
        memcpy(blk, ck + c * n, (size_t)n * sizeof(double));
        for (long t = t0; t < t1; ++t) bstep(J, t, blk + (t - t0) * n, blk + (t - t0 + 1) * n);
        for (long t = t1 - 1; t >= t0; --t) {
            const double* Sprev = blk + (t - t0) * n;
            const double* Scur = blk + (t - t0 + 1) * n;
            const double* qt = J->q + (J->bh * T + t) * dk;
            const double* kt = J->k + (J->bh * T + t) * dk;
            const double* vt = J->v + (J->bh * T + t) * dv;
            const double* dot = J->dO + (J->bh * T + t) * dv;
            double* dqt = J->gq + (J->bh * T + t) * dk;
            double* dkt = J->gk + (J->bh * T + t) * dk;
            double* dvt = J->gv + (J->bh * T + t) * dv;
            if (J->mutant == 12) bdecay(J, t, D);
            /* D_t = (decayed later adjoint) + q_t^T do_t */
            for (long i = 0; i < dk; ++i)
                for (long j = 0; j < dv; ++j) D[i * dv + j] += qt[i] * dot[j];
            const double* Sq = (J->mutant == 13) ? Sprev : Scur;
            for (long i = 0; i < dk; ++i) {
                double aq = 0.0, ak = 0.0, ag = 0.0;
                for (long j = 0; j < dv; ++j) {
                    aq += Sq[i * dv + j] * dot[j];
                    ak += D[i * dv + j] * vt[j];
                    ag += D[i * dv + j] * bbeta(J, t, j) * Sprev[i * dv + j];
                }
                dqt[i] = aq;
                dkt[i] = ak;
                J->dlg[t * dk + i] = (J->mutant == 11) ? ag : bgate(J, t, i) * ag;
            }
            for (long j = 0; j < dv; ++j) {
                double a = 0.0, ab = 0.0;
                for (long i = 0; i < dk; ++i) {
                    a += kt[i] * D[i * dv + j];
                    ab += D[i * dv + j] * bgate(J, t, i) * Sprev[i * dv + j];
                }
                dvt[j] = a;
                if (J->gate == 4 && J->dlb) J->dlb[t * dv + j] = (J->mutant == 15) ? ab : bbeta(J, t, j) * ab;
            }
            /* the part of dL/dS_{t-1} that flows through S_t */
            if (J->mutant != 12 && !(J->mutant == 14 && t == 0)) bdecay(J, t, D);
        }
    }
    if (J->dS0) memcpy(J->dS0 + J->bh * n, D, (size_t)n * sizeof(double));
    free(ck); free(blk); free(D); free(S); free(S2);
}

typedef struct {
    bjob_t* jobs;
    long njobs, next;
    pthread_mutex_t mu;
} bpool_t;

static void* bworker(void* arg)
{
    bpool_t* P = (bpool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&P->mu);
        long idx = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (idx >= P->njobs) break;
        bwd_job(&P->jobs[idx]);
    }
    return NULL;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 * dq, dk [B,H,T,dk]; dv [B,H,T,dv]; dlog_g shaped like log_g (NULL or
 * gate 0: not written); dS0 [B,H,dk,dv] or NULL. One job per (b, h). */
int gla_oracle_bwd(const double* q, const double* k, const double* v,
                   const double* log_g, int gate, const double* S0,
                   const double* dO, const double* dST,
                   double* dq, double* dk_out, double* dv_out, double* dlog_g, double* dS0,
                   long B, long H, long T, long dk, long dv, int nthreads, int mutant,
                   const double* log_b, double* dlog_b)
{
    if (!dO || !dq || !dk_out || !dv_out || B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return 1;
    if (T > 0 && (!q || !k || !v)) return 1;
    if (gate < 0 || gate > 4 || (gate != 0 && !log_g)) return 1;
    if (gate == 4 && T > 0 && !log_b) return 1;
    const long BH = B * H;
    double* dlg = (double*)calloc((size_t)(BH * T * dk > 0 ? BH * T * dk : 1), sizeof(double));
    bjob_t* jobs = (bjob_t*)calloc((size_t)BH, sizeof(bjob_t));
    if (!dlg || !jobs) { free(dlg); free(jobs); return 2; }
    for (long bh = 0; bh < BH; ++bh) {
        bjob_t* J = &jobs[bh];
        J->q = q; J->k = k; J->v = v; J->log_g = log_g; J->log_b = log_b; J->S0 = S0; J->dO = dO; J->dST = dST;
        J->gq = dq; J->gk = dk_out; J->gv = dv_out; J->dlg = dlg + bh * T * dk; J->dS0 = dS0;
        J->dlb = (gate == 4 && dlog_b) ? dlog_b + bh * T * dv : NULL;
        J->H = H; J->T = T; J->dk = dk; J->dv = dv; J->bh = bh; J->gate = gate; J->mutant = mutant;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = (int)BH;
    bpool_t P;
    P.jobs = jobs; P.njobs = BH; P.next = 0;
    pthread_mutex_init(&P.mu, NULL);
    pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
    int started = 0;
    if (th)
        for (int i = 0; i + 1 < nthreads; ++i)
            if (pthread_create(&th[started], NULL, bworker, &P) == 0) ++started;
    bworker(&P);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&P.mu);
    int st = 0;
    for (long i = 0; i < BH; ++i) if (jobs[i].status) st = 2;
    if (st == 0 && dlog_g && gate != 0) {
        if (gate == 2 || gate == 4) {
            memcpy(dlog_g, dlg, (size_t)(BH * T * dk) * sizeof(double));
        } else if (gate == 3) {
            for (long bt = 0; bt < BH * T; ++bt) {
                double s = 0.0;
                for (long i = 0; i < dk; ++i) s += dlg[bt * dk + i];
                dlog_g[bt] = s;
            }
        } else {
            for (long h = 0; h < H; ++h) {
                double s = 0.0;
                for (long b = 0; b < B; ++b)
                    for (long e = 0; e < T * dk; ++e) s += dlg[(b * H + h) * T * dk + e];
                dlog_g[h] = s;
            }
        }
    }
    free(dlg); free(jobs);
    return st;
}
