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
 * The steps on either side of the rule (the fused pre- and post-processing
 * of the library's GDR_FLAG_* options) are here too, each a plain loop:
 *   oracle_l2norm_rows      x / sqrt(sum x^2 + eps) per row (q and k before the
 *                           rule; the pages name the normalisation, not its eps:
 *                           eps = 1e-6 inside the square root is the reading taken)
 *   oracle_sigmoid          beta = 1 / (1 + exp(-b)) (beta from its logit, as the
 *                           workloads draw it: beta = sigmoid(N(0, 1)))
 *   oracle_gated_rmsnorm    y = w * o / sqrt(mean(o^2) + eps) * silu(z) per row of
 *                           d_v, eps = 1e-6 (the RMSNorm right after the rule on
 *                           the NPU model card, "fp16 precision of the DeltaNet
 *                           output", with the 1e-6 epsilon of the Candle PR's bug
 *                           log, "Bug 7"); the gate's form silu(z) = z sigmoid(z)
 *                           is a reading: the pages do not give it.
 *
 * Parity pins: see tests/test_oracle_pins.py (closed forms, exact rational
 * brute force, invariants).  The recurrence and both norms are pinned; the
 * output gate's form (silu) is "parity unpinned" against the pages, which do
 * not state it: only its arithmetic is pinned (closed forms of silu).
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

/* ---- steps on either side of the rule ------------------------------------------- */

/* y[r] = x[r] / sqrt(sum_i x[r][i]^2 + eps) for n rows of d values (y may be x). */
int oracle_l2norm_rows(int64_t n, int d, double eps, const double *x, double *y) {
    if (n < 0 || d <= 0 || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < n; ++r) {
        const double *xr = x + (size_t)r * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
        const double inv = 1.0 / sqrt(ss + eps);
        double *yr = y + (size_t)r * d;
        for (int i = 0; i < d; ++i) yr[i] = xr[i] * inv;
    }
    return 0;
}

/* beta[i] = 1 / (1 + exp(-b[i])) for n values. */
int oracle_sigmoid(int64_t n, const double *b, double *beta) {
    if (n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) beta[i] = 1.0 / (1.0 + exp(-b[i]));
    return 0;
}

/*
 * y[r][j] = w[j] * o[r][j] / sqrt(mean_i o[r][i]^2 + eps) * silu(z[r][j]) for n rows
 * of d values, silu(z) = z / (1 + exp(-z)).  w has d entries (one weight per
 * channel, shared by every row).
 */
int oracle_gated_rmsnorm(int64_t n, int d, double eps, const double *o, const double *z, const double *w,
                         double *y) {
    if (n < 0 || d <= 0 || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < n; ++r) {
        const double *orow = o + (size_t)r * d;
        const double *zrow = z + (size_t)r * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += orow[i] * orow[i];
        const double inv = 1.0 / sqrt(ss / d + eps);
        double *yr = y + (size_t)r * d;
        for (int j = 0; j < d; ++j) {
            const double zz = zrow[j];
            const double silu = zz / (1.0 + exp(-zz));
            yr[j] = w[j] * orow[j] * inv * silu;
        }
    }
    return 0;
}
