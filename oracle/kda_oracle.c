/*
 * KDA token-by-token recurrence in fp64 — the ORACLE.
 *
 * This file is test infrastructure. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes is the plain definition of Kimi Delta Attention (a gated
 * delta rule with a per-channel decay), one token at a time:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * Source: "在 TPU 上加速 Kimi K3 KDA" (junyi.dev, tpu-kda report) §1–§2 (the
 * fixed-size recurrent state carried per sequence and head, the decay
 * bounded below) and §13 (the fp32 naive recurrence used there as the
 * reference, expanded token by token). The chunked method of §4 and §6.2
 * reaches exactly this result in exact arithmetic, so this definition is
 * the oracle for it.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes):
 *   - state layout: S[i][j], i = key channel, j = value channel, so that
 *     k_t v_t^T is the write term; stored row-major as [N, H, K, V];
 *   - g is the natural-log decay per key channel, already activated;
 *   - o_t reads the state AFTER token t's update (the chunk form's Aqk
 *     includes its diagonal, §6.2);
 *   - scale multiplies o only, never the state;
 *   - the state restarts at every sequence of the varlen packing, from
 *     initial_state[n] (or zeros when it is NULL); an empty sequence passes
 *     initial_state straight to final_state (§6.5).
 *
 * Layouts (all fp64, row-major, caller-owned host memory):
 *   q, k : [T, H, Dk]     v : [T, H, Dv]     g : [T, H, Dk]   beta : [T, H]
 *   cu_seqlens : [N + 1], cu[0] = 0, nondecreasing, cu[N] = T
 *   initial_state : [N, H, Dk, Dv] or NULL     final_state : [N, H, Dk, Dv] or NULL
 *   o : [T, H, Dv]
 *
 * The work is split over (sequence, head) chains, which are independent, on
 * num_threads POSIX threads (<= 0 means one per online core). Each chain is
 * computed by exactly one thread in the same order, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int64_t *cu;
    int64_t num_seqs, num_heads, dk, dv;
    const double *s0;
    double scale;
    double *o, *sT;
    int nthreads;
    int tid;
    int status;
} job_t;

/* One (sequence n, head h) chain, token by token. */
static int run_chain(const job_t *J, int64_t n, int64_t h, double *S, double *kS)
{
    const int64_t H = J->num_heads, K = J->dk, V = J->dv;
    const int64_t bos = J->cu[n], eos = J->cu[n + 1];
    const size_t state_elems = (size_t)K * (size_t)V;

    if (J->s0)
        memcpy(S, J->s0 + ((size_t)n * H + h) * state_elems, state_elems * sizeof(double));
    else
        memset(S, 0, state_elems * sizeof(double));

    for (int64_t t = bos; t < eos; ++t) {
        const double *qt = J->q + ((size_t)t * H + h) * K;
        const double *kt = J->k + ((size_t)t * H + h) * K;
        const double *vt = J->v + ((size_t)t * H + h) * V;
        const double *gt = J->g + ((size_t)t * H + h) * K;
        const double bt = J->beta[(size_t)t * H + h];
        double *ot = J->o + ((size_t)t * H + h) * V;

        /* S <- Diag(exp g_t) S : row i (key channel i) decays by exp(g_t[i]) */
        for (int64_t i = 0; i < K; ++i) {
            const double a = exp(gt[i]);
            double *row = S + (size_t)i * V;
            for (int64_t j = 0; j < V; ++j) row[j] *= a;
        }
        /* kS = k_t^T S  (the value the delta rule erases) */
        for (int64_t j = 0; j < V; ++j) kS[j] = 0.0;
        for (int64_t i = 0; i < K; ++i) {
            const double ki = kt[i];
            const double *row = S + (size_t)i * V;
            for (int64_t j = 0; j < V; ++j) kS[j] += ki * row[j];
        }
        /* S <- S + beta_t k_t (v_t - S^T k_t)^T
         *    = (I - beta_t k_t k_t^T) S + beta_t k_t v_t^T */
        for (int64_t i = 0; i < K; ++i) {
            const double bk = bt * kt[i];
            double *row = S + (size_t)i * V;
            for (int64_t j = 0; j < V; ++j) row[j] += bk * (vt[j] - kS[j]);
        }
        /* o_t = scale * S^T q_t */
        for (int64_t j = 0; j < V; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < K; ++i) {
            const double qi = qt[i];
            const double *row = S + (size_t)i * V;
            for (int64_t j = 0; j < V; ++j) ot[j] += qi * row[j];
        }
        for (int64_t j = 0; j < V; ++j) ot[j] *= J->scale;
    }
    if (J->sT)
        memcpy(J->sT + ((size_t)n * H + h) * state_elems, S, state_elems * sizeof(double));
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int64_t chains = J->num_seqs * J->num_heads;
    double *S = (double *)malloc((size_t)J->dk * (size_t)J->dv * sizeof(double));
    double *kS = (double *)malloc((size_t)J->dv * sizeof(double));
    if (!S || !kS) {
        J->status = 2;
        free(S);
        free(kS);
        return NULL;
    }
    for (int64_t c = J->tid; c < chains; c += J->nthreads)
        run_chain(J, c / J->num_heads, c % J->num_heads, S, kS);
    free(S);
    free(kS);
    return NULL;
}

/* Returns 0 on success, 1 on invalid arguments, 2 on allocation or thread failure.
 * Returns the thread count actually used through *threads_used when non-NULL. */
int kda_oracle_fwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int64_t *cu_seqlens, int64_t num_seqs,
                   int64_t num_heads, int64_t dk, int64_t dv, const double *initial_state,
                   double scale, double *o, double *final_state, int num_threads,
                   int *threads_used)
{
    if (num_seqs < 0 || num_heads < 1 || dk < 1 || dv < 1 || !cu_seqlens) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int64_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    if (cu_seqlens[num_seqs] > 0 && (!q || !k || !v || !g || !beta || !o)) return 1;

    int nt = num_threads;
    if (nt <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nt = c > 0 ? (int)c : 1;
    }
    const int64_t chains = num_seqs * num_heads;
    if (chains < nt) nt = chains > 0 ? (int)chains : 1;
    if (threads_used) *threads_used = nt;

    job_t *jobs = (job_t *)calloc((size_t)nt, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return 2;
    }
    int rc = 0;
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        job_t J = {q, k, v, g, beta, cu_seqlens, num_seqs, num_heads, dk, dv,
                   initial_state, scale, o, final_state, nt, i, 0};
        jobs[i] = J;
    }
    for (int i = 1; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) {
            rc = 2;
            break;
        }
        started = i;
    }
    if (rc == 0) worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < nt && rc == 0; ++i)
        if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    free(th);
    return rc;
}
