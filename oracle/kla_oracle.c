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

/*
 * ---------------------------------------------------------------- backward pass
 *
 * Reverse-mode derivative of the recurrence above for one scalar loss L that
 * depends on the outputs o_t and the final state S_T, given dO = dL/do_t
 * [B, T, H, d_v] and dS_T = dL/dS_T [B, H, d_k, d_v] (NULL: zero). The pages give
 * no backward algebra; this is the chain rule applied to steps 1-6 in reverse
 * order, with G = dL/dS_t carried from t = T-1 down to 0:
 *
 *   6. read      o = S_t^T (s q):      dq_t = s S_t do_t ;  G += s q do_t^T
 *   5. write     S_t = S~ + beta k e^T: dS~ = G ;  dbeta = k^T G e ;
 *                                       dk += beta G e ;  de = beta G^T k
 *   3. residual  e = v - S~^T k:        dv_t = de ;  dS~ -= k de^T ;  dk -= S~ de
 *   4. step      KLA: beta = eta / (n + eps), n = ||k||^2:
 *                    deta = dbeta / (n + eps) ;  dk -= 2 beta dbeta / (n + eps) k
 *                    (beta := 0 when n + eps == 0: no derivative flows)
 *                raw: beta = eta:  deta = dbeta
 *   1. forget    S~ = alpha (.) S_{t-1}: dalpha = sum_j S_{t-1}[i,j] dS~[i,j] (summed
 *                over i too for a scalar gate) ;  G = alpha (.) dS~
 *
 * and dS0 = G at the end. The states S_0 .. S_{T-1} entering each token are kept
 * from a forward run (T d_k d_v doubles per chain: small cases only).
 *
 * Outputs (all written): dq, dk [B,T,H,d_k]; dv [B,T,H,d_v]; dalpha like alpha;
 * deta [B,T,H]; dS0 [B,H,d_k,d_v]. Returns 0, -1 on bad arguments, -2 on
 * allocation failure.
 */
typedef struct {
    job_t f;                      /* forward arguments (o, S_T unused) */
    const double *dO, *dST;
    double *dq, *dk, *dv, *dalpha, *deta, *dS0;
} bjob_t;

static int backward_chain(const bjob_t *J, long b, long h, double *Sall, double *G, double *St,
                          double *e, double *de, double *tmp)
{
    const job_t *F = &J->f;
    const long T = F->T, H = F->H, dk = F->dk, dv = F->dv, dd = dk * dv;
    const double s = F->q_scale;
    double *beta = tmp, *nrm = tmp + T;
    /* forward, keeping the state entering every token */
    if (F->S0) memcpy(Sall, F->S0 + ((b * H + h) * dk) * dv, sizeof(double) * dd);
    else memset(Sall, 0, sizeof(double) * dd);
    for (long t = 0; t < T; ++t) {
        const long tok = (b * T + t) * H + h;
        const double *kt = F->k + tok * dk, *vt = F->v + tok * dv;
        const double *S = Sall + t * dd;
        double *Sn = Sall + (t + 1) * dd;
        for (long i = 0; i < dk; ++i) {
            const double a = F->alpha_per_channel ? F->alpha[tok * dk + i] : F->alpha[tok];
            for (long j = 0; j < dv; ++j) St[i * dv + j] = a * S[i * dv + j];
        }
        double n2 = 0.0;
        for (long i = 0; i < dk; ++i) n2 += kt[i] * kt[i];
        const double den = n2 + F->eps;
        double bt = (den == 0.0) ? 0.0 : F->eta[tok] / den;
        if (F->beta_mode == 1) bt = F->eta[tok];
        beta[t] = bt;
        nrm[t] = den;
        for (long j = 0; j < dv; ++j) {
            double p = 0.0;
            for (long i = 0; i < dk; ++i) p += St[i * dv + j] * kt[i];
            e[t * dv + j] = vt[j] - p;
        }
        if (t + 1 < T)
            for (long i = 0; i < dk; ++i)
                for (long j = 0; j < dv; ++j) Sn[i * dv + j] = St[i * dv + j] + bt * kt[i] * e[t * dv + j];
    }
    /* reverse */
    if (J->dST) memcpy(G, J->dST + ((b * H + h) * dk) * dv, sizeof(double) * dd);
    else memset(G, 0, sizeof(double) * dd);
    for (long t = T - 1; t >= 0; --t) {
        const long tok = (b * T + t) * H + h;
        const double *kt = F->k + tok * dk, *qt = F->q + tok * dk;
        const double *dot = J->dO + tok * dv;
        const double *S = Sall + t * dd;            /* S_{t-1}: the state entering token t */
        const double *et = e + t * dv;
        const double bt = beta[t];
        double *dqt = J->dq + tok * dk, *dkt = J->dk + tok * dk, *dvt = J->dv + tok * dv;
        /* S~ and S_t */
        for (long i = 0; i < dk; ++i) {
            const double a = F->alpha_per_channel ? F->alpha[tok * dk + i] : F->alpha[tok];
            for (long j = 0; j < dv; ++j) St[i * dv + j] = a * S[i * dv + j];
        }
        /* 6. read */
        for (long i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j) acc += (St[i * dv + j] + bt * kt[i] * et[j]) * dot[j];
            dqt[i] = s * acc;
        }
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) G[i * dv + j] += s * qt[i] * dot[j];
        /* 5. write */
        double dbeta = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) dbeta += kt[i] * G[i * dv + j] * et[j];
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk; ++i) acc += G[i * dv + j] * kt[i];
            de[j] = bt * acc;
        }
        for (long i = 0; i < dk; ++i) {
            double ge = 0.0, sde = 0.0;
            for (long j = 0; j < dv; ++j) {
                ge += G[i * dv + j] * et[j];
                sde += St[i * dv + j] * de[j];
            }
            dkt[i] = bt * ge - sde;                  /* write and residual terms */
        }
        /* 3. residual */
        for (long j = 0; j < dv; ++j) dvt[j] = de[j];
#if KLA_ORACLE_MUTANT != 11   /* mutant 11: the residual's path back into the state is dropped */
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) G[i * dv + j] -= kt[i] * de[j];   /* G now holds dS~ */
#endif
        /* 4. step size */
        if (F->beta_mode == 1) {
            J->deta[tok] = dbeta;
        } else if (nrm[t] == 0.0) {
            J->deta[tok] = 0.0;
        } else {
            J->deta[tok] = dbeta / nrm[t];
#if KLA_ORACLE_MUTANT != 10   /* mutant 10: the step's dependence on ||k|| is dropped */
            for (long i = 0; i < dk; ++i) dkt[i] -= 2.0 * bt * dbeta / nrm[t] * kt[i];
#endif
        }
        /* 1. forget */
        if (F->alpha_per_channel) {
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += S[i * dv + j] * G[i * dv + j];
                J->dalpha[tok * dk + i] = acc;
            }
        } else {
            double acc = 0.0;
            for (long i = 0; i < dd; ++i) acc += S[i] * G[i];
            J->dalpha[tok] = acc;
        }
        for (long i = 0; i < dk; ++i) {
            const double a = F->alpha_per_channel ? F->alpha[tok * dk + i] : F->alpha[tok];
            for (long j = 0; j < dv; ++j) G[i * dv + j] *= a;
        }
    }
    memcpy(J->dS0 + ((b * H + h) * dk) * dv, G, sizeof(double) * dd);
    return 0;
}

static void *bworker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    const job_t *F = &J->f;
    const long dd = F->dk * F->dv;
    double *Sall = (double *)malloc(sizeof(double) * (F->T + 1) * dd);
    double *G = (double *)malloc(sizeof(double) * dd);
    double *St = (double *)malloc(sizeof(double) * dd);
    double *e = (double *)malloc(sizeof(double) * (F->T + 1) * F->dv);
    double *de = (double *)malloc(sizeof(double) * F->dv);
    double *tmp = (double *)malloc(sizeof(double) * (2 * F->T + 2));
    if (!Sall || !G || !St || !e || !de || !tmp) {
        J->f.status = -2;
    } else {
        for (long c = F->chain_begin; c < F->chain_end; ++c) backward_chain(J, c / F->H, c % F->H, Sall, G, St, e, de, tmp);
        J->f.status = 0;
    }
    free(Sall); free(G); free(St); free(e); free(de); free(tmp);
    return NULL;
}

int kla_oracle_backward(const double *q, const double *k, const double *v,
                        const double *alpha, int alpha_per_channel,
                        const double *eta, double eps, const double *S0,
                        const double *dO, const double *dS_T,
                        double *dq, double *dk_out, double *dv_out, double *dalpha, double *deta, double *dS0,
                        long B, long T, long H, long dk, long dv,
                        int beta_mode, double q_scale, int nthreads)
{
    if (!q || !k || !v || !alpha || !eta || !dO || !dq || !dk_out || !dv_out || !dalpha || !deta || !dS0 ||
        B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 || (beta_mode != 0 && beta_mode != 1))
        return -1;
    long chains = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > chains) nthreads = (int)(chains > 0 ? chains : 1);
    bjob_t base;
    memset(&base, 0, sizeof(base));
    job_t f = {q, k, v, alpha, eta, S0, NULL, NULL, B, T, H, dk, dv, alpha_per_channel, eps,
               beta_mode, q_scale, 0, 0, 0};
    base.f = f;
    base.dO = dO; base.dST = dS_T;
    base.dq = dq; base.dk = dk_out; base.dv = dv_out; base.dalpha = dalpha; base.deta = deta; base.dS0 = dS0;
    bjob_t *jobs = (bjob_t *)calloc((size_t)nthreads, sizeof(bjob_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -2; }
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = base;
        jobs[w].f.chain_begin = chains * w / nthreads;
        jobs[w].f.chain_end = chains * (w + 1) / nthreads;
    }
    int status = 0;
    if (nthreads == 1) {
        bworker(&jobs[0]);
        status = jobs[0].f.status;
    } else {
        for (int w = 0; w < nthreads; ++w) pthread_create(&tid[w], NULL, bworker, &jobs[w]);
        for (int w = 0; w < nthreads; ++w) {
            pthread_join(tid[w], NULL);
            if (jobs[w].f.status) status = jobs[w].f.status;
        }
    }
    free(jobs); free(tid);
    return status;
}
