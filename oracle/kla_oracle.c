/*
 * kla_oracle.c -- fp64 CPU oracle of the Kaczmarz (KLA) gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct definition
 * that the CUDA path is checked against. Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it. It shares no code, header, table
 * or helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes, for every (b, h) independently, starting from S = S0
 * (d_k x d_v, rows = key channels, columns = value channels), for t = 0..T-1:
 *
 *   1. forget:   S~ = alpha_t * S            (scalar gate), or
 *                S~[i,:] = alpha_t[i] * S[i,:] (per-key-channel gate: rows)
 *   2. predict:  p = S~^T k_t
 *   3. residual: e = v_t - p
 *   4. step:     beta = eta_t / (||k_t||^2 + eps)     (beta := 0 if the
 *                denominator is exactly 0)  -- the KLA step (beta_mode 0), or
 *                beta = eta_t                         -- the raw write strength of
 *                DeltaNet / Gated DeltaNet (beta_mode 1)
 *   5. write:    S = S~ + beta k_t e^T
 *   6. read:     o_t = S^T (s q_t)           (after the write; s = q_scale, 1 by
 *                default, d_k^{-1/2} in Kimi Delta Attention)
 *
 * Sources (page titles and sections):
 *  - Gist.science "Riepilogo Tecnico: Attenzione Lineare Kaczmarz (KLA)",
 *    section "La Regola di Aggiornamento KLA": the coefficient
 *    beta = eta / (||k||^2 + eps), the update S_t = S~ + beta k e^T with the
 *    residual taken against the decayed state, and the d_k x d_v state whose
 *    constraint is S^T k = v (section "Derivazione Teorica").
 *  - GeekNews "Revisando las variantes de atencion lineal de la familia DeltaNet",
 *    section "Gated DeltaNet: primero olvidar todo el estado": the mandated order
 *    forget -> predict -> correct -> write; section "Kimi Delta Attention":
 *    the per-key-channel gate and the read after the write, which reads with the
 *    scaled query d_k^{-1/2} q (and the in-chunk coefficients carry the same s,
 *    section "KDA por chunks"); section "Gated DeltaNet": beta_t in (0,1) is the
 *    write strength itself, the plain delta-rule step without the KLA normaliser.
 *  - Paithon "Scrivere meglio nella memoria: gate e delta rule": the key-channel
 *    side of the diagonal gate.
 *
 * The transposed d_v x d_k convention of the last two pages gives the same
 * numbers; this file uses the d_k x d_v orientation of the KLA page.
 *
 * Layouts (row-major, contiguous):
 *   q, k      [B, T, H, d_k]      v, o     [B, T, H, d_v]
 *   alpha     [B, T, H] or [B, T, H, d_k]
 *   eta       [B, T, H]           S0, S_T  [B, H, d_k, d_v]  (S0 may be NULL)
 *
 * Mutation switch (tests only): compiling with -DKLA_ORACLE_MUTANT=n plants one
 * deliberate mistake so that the test suite can show its pins catch it. The
 * default build (no macro) is the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#ifndef KLA_ORACLE_MUTANT
#define KLA_ORACLE_MUTANT 0
#endif

typedef struct {
    const double *q, *k, *v, *alpha, *eta, *S0;
    double *o, *S_T;
    long B, T, H, dk, dv;
    int alpha_per_channel;
    double eps;
    int beta_mode;        /* 0: beta = eta / (||k||^2 + eps);  1: beta = eta */
    double q_scale;       /* read with s * q */
    long chain_begin, chain_end;
    int status;
} job_t;

/* One (b, h) chain, token by token. */
static int run_chain(const job_t *J, long b, long h, double *S, double *St, double *p)
{
    const long T = J->T, H = J->H, dk = J->dk, dv = J->dv;
    if (J->S0) memcpy(S, J->S0 + ((b * H + h) * dk) * dv, sizeof(double) * dk * dv);
    else memset(S, 0, sizeof(double) * dk * dv);

    for (long t = 0; t < T; ++t) {
        const long tok = (b * T + t) * H + h;
        const double *kt = J->k + tok * dk;
        const double *vt = J->v + tok * dv;
        const double *qt = J->q + tok * dk;
        const double eta = J->eta[tok];

        /* 1. forget (a per-channel gate scales rows: the key channels) */
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) {
#if KLA_ORACLE_MUTANT == 6
                /* mutant: per-channel gate applied to the value channels (columns) */
                const long ch = j % dk;
#else
                const long ch = i;
#endif
                const double a = J->alpha_per_channel ? J->alpha[tok * dk + ch] : J->alpha[tok];
                St[i * dv + j] = a * S[i * dv + j];
            }

        /* 2. predict: p = S~^T k */
        for (long j = 0; j < dv; ++j) p[j] = 0.0;
        for (long i = 0; i < dk; ++i)
#if KLA_ORACLE_MUTANT == 1
            /* mutant: predict from the state before the forget gate */
            for (long j = 0; j < dv; ++j) p[j] += S[i * dv + j] * kt[i];
#else
            for (long j = 0; j < dv; ++j) p[j] += St[i * dv + j] * kt[i];
#endif

        /* 3. residual (stored in p): e = v - p */
        for (long j = 0; j < dv; ++j)
#if KLA_ORACLE_MUTANT == 3
            p[j] = p[j] - vt[j];          /* mutant: sign of the residual */
#else
            p[j] = vt[j] - p[j];
#endif

        /* 4. KLA step size */
        double n2 = 0.0;
        for (long i = 0; i < dk; ++i) n2 += kt[i] * kt[i];
        double den = n2 + J->eps;
#if KLA_ORACLE_MUTANT == 2
        double beta = (n2 == 0.0) ? 0.0 : eta / n2 + J->eps;   /* mutant: eps outside */
#elif KLA_ORACLE_MUTANT == 4
        double beta = (den == 0.0) ? 0.0 : 1.0 / den;          /* mutant: eta dropped */
#else
        double beta = (den == 0.0) ? 0.0 : eta / den;
#endif
#if KLA_ORACLE_MUTANT != 8   /* mutant 8: the raw mode still takes the KLA step */
        if (J->beta_mode == 1) beta = eta;
#endif

        /* 5. write: S = S~ + beta k e^T */
        for (long i = 0; i < dk; ++i) {
            const double bk = beta * kt[i];
            for (long j = 0; j < dv; ++j) S[i * dv + j] = St[i * dv + j] + bk * p[j];
        }

        /* 6. read after the write: o = S^T (s q) */
        double *ot = J->o + tok * dv;
#if KLA_ORACLE_MUTANT == 9
        const double s = 1.0;           /* mutant: the query scale is dropped */
#else
        const double s = J->q_scale;
#endif
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
#if KLA_ORACLE_MUTANT == 5
        /* mutant: read before the write */
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) ot[j] += St[i * dv + j] * qt[i];
#elif KLA_ORACLE_MUTANT == 7
        /* mutant: transposed read o = S q (only meaningful when d_k == d_v) */
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) ot[i % dv] += S[i * dv + j] * qt[j % dk];
#else
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * (s * qt[i]);
#endif
    }
    if (J->S_T) memcpy(J->S_T + ((b * H + h) * dk) * dv, S, sizeof(double) * dk * dv);
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * J->dk * J->dv);
    double *St = (double *)malloc(sizeof(double) * J->dk * J->dv);
    double *p = (double *)malloc(sizeof(double) * J->dv);
    if (!S || !St || !p) { J->status = -2; free(S); free(St); free(p); return NULL; }
    for (long c = J->chain_begin; c < J->chain_end; ++c) run_chain(J, c / J->H, c % J->H, S, St, p);
    free(S); free(St); free(p);
    J->status = 0;
    return NULL;
}

/*
 * Runs the recurrence for all B*H chains; chains are split over `nthreads`
 * POSIX threads (each chain is independent, so the split changes no result).
 * beta_mode 0 takes the KLA step, 1 the raw write strength beta = eta; the read
 * uses q_scale * q. Returns 0 on success, -1 on bad arguments, -2 on allocation
 * failure.
 */
int kla_oracle_recurrent_ex(const double *q, const double *k, const double *v,
                            const double *alpha, int alpha_per_channel,
                            const double *eta, double eps, const double *S0,
                            double *o, double *S_T,
                            long B, long T, long H, long dk, long dv,
                            int beta_mode, double q_scale, int nthreads)
{
    if (!q || !k || !v || !alpha || !eta || !o || B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 ||
        (beta_mode != 0 && beta_mode != 1))
        return -1;
    long chains = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > chains) nthreads = (int)(chains > 0 ? chains : 1);
    job_t base = {q, k, v, alpha, eta, S0, o, S_T, B, T, H, dk, dv, alpha_per_channel, eps,
                  beta_mode, q_scale, 0, 0, 0};
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -2; }
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = base;
        jobs[w].chain_begin = chains * w / nthreads;
        jobs[w].chain_end = chains * (w + 1) / nthreads;
    }
    int status = 0;
    if (nthreads == 1) {
        worker(&jobs[0]);
        status = jobs[0].status;
    } else {
        for (int w = 0; w < nthreads; ++w) pthread_create(&tid[w], NULL, worker, &jobs[w]);
        for (int w = 0; w < nthreads; ++w) {
            pthread_join(tid[w], NULL);
            if (jobs[w].status) status = jobs[w].status;
        }
    }
    free(jobs); free(tid);
    return status;
}

int kla_oracle_mutant_id(void) { return KLA_ORACLE_MUTANT; }

/* The KLA recurrence with the default read (beta_mode 0, q_scale 1). */
int kla_oracle_recurrent(const double *q, const double *k, const double *v,
                         const double *alpha, int alpha_per_channel,
                         const double *eta, double eps, const double *S0,
                         double *o, double *S_T,
                         long B, long T, long H, long dk, long dv, int nthreads)
{
    return kla_oracle_recurrent_ex(q, k, v, alpha, alpha_per_channel, eta, eps, S0, o, S_T,
                                   B, T, H, dk, dv, 0, 1.0, nthreads);
}
