/*
 * Sequential fp64 oracle of the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it; the library's compute
 * path never links or calls it, and it shares no code, header or constant
 * with that path.
 *
 * What it computes (per sequence s and V head h, for t in order):
 *
 *     S <- exp(g_t) * S                          (gate: alpha_t = exp(g_t))
 *     u <- S^T k_t                               (what the state recalls for k_t)
 *     S <- S + k_t ((v_t - u) * beta_t)^T        (delta-rule correction)
 *     o_t <- scale * S^T q_t                     (read-out from the updated state)
 *
 * This is the per-token loop written out on the Qwen3.5-9B NPU model card
 * ("Qwen3.5-9B - every component on the Intel NPU", section "How it works",
 * the four-line Loop step), which expands to the closed recurrence
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t
 * given in "Qwen3.5-9B: Giai ma kien truc Gated DeltaNet" (section "Gated
 * DeltaNet", state update formula).  ``scale`` is 1 in every workload; the
 * pages name no query scale.
 *
 * Head sharing: V head h reads q and k from QK head h / (H_v / H_qk), i.e.
 * each QK head feeds a contiguous group of H_v / H_qk V heads (two for
 * Qwen3.5-9B's 16 QK / 32 V heads).
 *
 * Layouts (row-major, token-major, packed over sequences by cu_seqlens):
 *     q, k  [T_total][H_qk][d_k]      v, o [T_total][H_v][d_v]
 *     g, beta [T_total][H_v]          state [n_seqs][H_v][d_k][d_v]  (in: S0, out: S_T)
 * Every array is double; callers widen the exact fp32/bf16 values.
 *
 * Parity pins: see tests/test_oracle_pins.py (closed forms, exact rational
 * brute force, invariants).  Nothing in this file is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_seqs;
    const int64_t *cu_seqlens;
    int h_qk, h_v, d_k, d_v;
    const double *q, *k, *v, *g, *beta;
    double scale;
    double *state;
    double *o;
    /* work distribution */
    int next;
    pthread_mutex_t lock;
} oracle_job;

/* One (sequence, V head) pair: the recurrence above, token by token. */
static void run_pair(const oracle_job *J, int s, int h, double *u) {
    const int dk = J->d_k, dv = J->d_v;
    const int group = J->h_v / J->h_qk;
    const int hq = h / group;
    double *S = J->state + ((size_t)s * J->h_v + h) * (size_t)dk * dv;
    for (int64_t t = J->cu_seqlens[s]; t < J->cu_seqlens[s + 1]; ++t) {
        const double *kt = J->k + ((size_t)t * J->h_qk + hq) * dk;
        const double *qt = J->q + ((size_t)t * J->h_qk + hq) * dk;
        const double *vt = J->v + ((size_t)t * J->h_v + h) * dv;
        const double alpha = exp(J->g[(size_t)t * J->h_v + h]);
        const double b = J->beta[(size_t)t * J->h_v + h];

        /* S <- alpha S */
        for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= alpha;

        /* u <- S^T k_t */
        for (int j = 0; j < dv; ++j) u[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double ki = kt[i];
            const double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) u[j] += row[j] * ki;
        }

        /* S <- S + k_t ((v_t - u) beta_t)^T */
        for (int j = 0; j < dv; ++j) u[j] = (vt[j] - u[j]) * b;
        for (int i = 0; i < dk; ++i) {
            const double ki = kt[i];
            double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) row[j] += ki * u[j];
        }

        /* o_t <- scale S^T q_t */
        double *ot = J->o + ((size_t)t * J->h_v + h) * dv;
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double qi = qt[i];
            const double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) ot[j] += row[j] * qi;
        }
        for (int j = 0; j < dv; ++j) ot[j] *= J->scale;
    }
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    double *u = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    const int total = J->n_seqs * J->h_v;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int idx = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= total) break;
        run_pair(J, idx / J->h_v, idx % J->h_v, u);
    }
    free(u);
    return NULL;
}

/*
 * Returns 0 on success, -1 on invalid arguments.  n_threads <= 1 runs on the
 * calling thread; otherwise that many worker threads share the
 * (sequence, V head) pairs.
 */
int oracle_gdr_sequential(int n_seqs, const int64_t *cu_seqlens, int h_qk, int h_v, int d_k,
                          int d_v, const double *q, const double *k, const double *v,
                          const double *g, const double *beta, double scale, double *state,
                          double *o, int n_threads) {
    if (n_seqs < 0 || h_qk <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0) return -1;
    if (h_v % h_qk != 0) return -1;
    if (n_seqs == 0) return 0;
    if (!cu_seqlens || !state) return -1;
    for (int s = 0; s < n_seqs; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    if (cu_seqlens[n_seqs] > cu_seqlens[0] && (!q || !k || !v || !g || !beta || !o)) return -1;

    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs;
    J.cu_seqlens = cu_seqlens;
    J.h_qk = h_qk;
    J.h_v = h_v;
    J.d_k = d_k;
    J.d_v = d_v;
    J.q = q;
    J.k = k;
    J.v = v;
    J.g = g;
    J.beta = beta;
    J.scale = scale;
    J.state = state;
    J.o = o;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);

    if (n_threads <= 1) {
        worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
        int started = 0;
        for (int i = 0; i < n_threads; ++i)
            if (pthread_create(&th[i], NULL, worker, &J) == 0) ++started;
        if (started == 0) worker(&J);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}
