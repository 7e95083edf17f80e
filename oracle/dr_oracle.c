/*
 * dr_oracle.c -- fp64 CPU oracle of the gated delta rule.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg load this
 * file's shared library.  The CUDA library never links or calls it and shares no code
 * with it.
 *
 * What it computes is the plain token-by-token definition of the recurrence, in the
 * order given by the teaching loop `gated_delta_rule` on the page "linear-attention
 * gated-deltanet guide" (section 4, "Gated DeltaNet: three gates"): decay the state,
 * predict the value with the decayed state, write the residual scaled by beta, then read
 * with the query.  With a per-channel gate this is the KDA update of the page
 * "NLP: linear attention summary" (section "Kimi Delta Attention"):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 *
 * and with a scalar gate it is the Gated DeltaNet update alpha_t (I - beta_t k_t k_t^T)
 * S_{t-1} + beta_t k_t v_t^T of the same page (section "Gated DeltaNet"), which is the
 * same thing because a scalar commutes with the erase matrix.  With no gate (alpha = 1)
 * it is the DeltaNet rule (same page, section "DeltaNet", the gradient-step equation).
 *
 * Arithmetic: IEEE fp64, no fused multiply-add contraction (built with
 * -ffp-contract=off), alpha_t = exp(log_alpha_t) taken in fp64.  No chunking, no
 * division, no reordering: each column j of S only ever meets v_t[j], so the work is
 * split into independent tasks over (batch, head, block of state columns), and inside a
 * task every column follows exactly the loop below.
 *
 * Layouts (all contiguous, row-major, fp64):
 *   q, k        [B, T, H, dk]
 *   v, out      [B, T, H, dv]
 *   beta        [B, T, H]
 *   log_alpha   NULL (gate 0), [B, T, H] (gate 1, scalar), [B, T, H, dk] (gate 2, channel)
 *   init_state  NULL (zeros) or [B, H, dk, dv]
 *   final_state NULL (not returned) or [B, H, dk, dv]; may alias init_state
 * Returns 0 on success, -1 on a bad argument, -2 if a thread could not be started.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, T, H, dk, dv;
    int gate;
    const double *q, *k, *v, *log_alpha, *beta, *init_state;
    double *out, *final_state;
    int64_t col_block;   /* columns of S per task */
    int64_t n_tasks;
    int64_t next_task;   /* protected by mu */
    pthread_mutex_t mu;
} job_t;

/* One task: chain (b, h), state columns [j0, j1). */
static void run_task(const job_t *J, int64_t b, int64_t h, int64_t j0, int64_t j1,
                     double *S, double *a, double *p) {
    const int64_t dk = J->dk, dv = J->dv, T = J->T, H = J->H;
    const int64_t nb = j1 - j0;
    /* S holds rows i = 0..dk-1 of the column block, S[i*nb + jj] = S_{i, j0+jj}. */
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t jj = 0; jj < nb; ++jj)
            S[i * nb + jj] = J->init_state
                ? J->init_state[((b * H + h) * dk + i) * dv + j0 + jj] : 0.0;

    for (int64_t t = 0; t < T; ++t) {
        const int64_t tok = (b * T + t) * H + h;          /* index of (b, t, h) */
        const double *qt = J->q + tok * dk;
        const double *kt = J->k + tok * dk;
        const double *vt = J->v + tok * dv;
        const double bt = J->beta[tok];

        /* alpha_t: per channel, scalar broadcast, or 1 */
        for (int64_t i = 0; i < dk; ++i) {
            if (J->gate == 2)      a[i] = exp(J->log_alpha[tok * dk + i]);
            else if (J->gate == 1) a[i] = exp(J->log_alpha[tok]);
            else                   a[i] = 1.0;
        }
        /* (1) decay: S <- Diag(alpha_t) S */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t jj = 0; jj < nb; ++jj)
                S[i * nb + jj] *= a[i];
        /* (2) predict with the decayed state: p = S^T k_t */
        for (int64_t jj = 0; jj < nb; ++jj) p[jj] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t jj = 0; jj < nb; ++jj)
                p[jj] += S[i * nb + jj] * kt[i];
        /* (3) write the residual: S <- S + beta_t k_t (v_t - p)^T */
        for (int64_t jj = 0; jj < nb; ++jj) p[jj] = bt * (vt[j0 + jj] - p[jj]);
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t jj = 0; jj < nb; ++jj)
                S[i * nb + jj] += kt[i] * p[jj];
        /* (4) read after the write: o_t = S_t^T q_t */
        double *ot = J->out + tok * dv;
        for (int64_t jj = 0; jj < nb; ++jj) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * nb + jj] * qt[i];
            ot[j0 + jj] = acc;
        }
    }
    if (J->final_state)
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t jj = 0; jj < nb; ++jj)
                J->final_state[((b * H + h) * dk + i) * dv + j0 + jj] = S[i * nb + jj];
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int64_t nblk = (J->dv + J->col_block - 1) / J->col_block;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->dk * J->col_block));
    double *a = (double *)malloc(sizeof(double) * (size_t)J->dk);
    double *p = (double *)malloc(sizeof(double) * (size_t)J->col_block);
    if (!S || !a || !p) { free(S); free(a); free(p); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int64_t task = J->next_task++;
        pthread_mutex_unlock(&J->mu);
        if (task >= J->n_tasks) break;
        const int64_t blk = task % nblk, bh = task / nblk;
        const int64_t j0 = blk * J->col_block;
        const int64_t j1 = (j0 + J->col_block < J->dv) ? j0 + J->col_block : J->dv;
        run_task(J, bh / J->H, bh % J->H, j0, j1, S, a, p);
    }
    free(S); free(a); free(p);
    return NULL;
}

int oracle_forward(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv, int gate,
                   const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta, const double *init_state,
                   double *out, double *final_state, int nthreads, int64_t col_block) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    if (gate < 0 || gate > 2) return -1;
    if (gate != 0 && !log_alpha) return -1;
    if ((T > 0 && (!q || !k || !v || !beta || !out))) return -1;
    if (nthreads < 1) nthreads = 1;
    if (col_block < 1 || col_block > dv) col_block = dv;

    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.T = T; J.H = H; J.dk = dk; J.dv = dv; J.gate = gate;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta;
    J.init_state = init_state; J.out = out; J.final_state = final_state;
    J.col_block = col_block;
    J.n_tasks = B * H * ((dv + col_block - 1) / col_block);
    J.next_task = 0;
    if (J.n_tasks == 0) return 0;

    /* final_state may alias init_state: every task reads its slice of init_state before
       it writes the same slice of final_state, and slices do not overlap. */
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads > J.n_tasks) nthreads = (int)J.n_tasks;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) { pthread_mutex_destroy(&J.mu); return -2; }
    int started = 0, rc = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) { rc = -2; break; }
        ++started;
    }
    if (worker(&J) != NULL) rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&J.mu);
    return rc;
}

/* One decode step = the loop body once, state updated in place.
 * q, k [B, H, dk]; v, out [B, H, dv]; beta [B, H]; log_alpha NULL, [B, H] or [B, H, dk];
 * state [B, H, dk, dv] (read and overwritten). */
int oracle_step(int64_t B, int64_t H, int64_t dk, int64_t dv, int gate,
                const double *q, const double *k, const double *v,
                const double *log_alpha, const double *beta, double *state,
                double *out, int nthreads) {
    if (!state) return -1;
    return oracle_forward(B, 1, H, dk, dv, gate, q, k, v, log_alpha, beta, state, out,
                          state, nthreads, 0);
}
