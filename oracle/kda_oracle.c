/*
 * Oracle for the gated delta rule with a per-channel gate (Kimi Delta Attention).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, fp64 CPU statement of what
 * the chunkwise forward pass computes. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the library's own code path never does.
 * It shares no code with the CUDA path.
 *
 * What it computes (token by token, no chunking, no reordering):
 *   "TileLang 实战：KDA 从零到一–Kimi Delta Attention", §3.1 (reference A, the token
 *   recurrence) gives, in the paper layout S in R^{d_v x d_k},
 *       S_t = S_{t-1} Diag(a_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t,
 *   with Diag(a_t) between S_{t-1} and the Householder factor. The same page (§0) and
 *   "TileLang 实战：KDA 从零到一--标量衰减" (§4.0) store the transpose, S^T in R^{d_k x d_v};
 *   this file keeps that transposed layout, in which one step reads
 *       S   <- Diag(a_t) S                      (decay before the erase read)
 *       u   <- beta_t (v_t - S^T k_t)
 *       S   <- S + k_t u^T
 *       o_t <- scale * S^T q_t
 *   a_t = exp(g_t) per channel (g is the natural-log gate). The scalar-gate Gated
 *   DeltaNet ("Gated DeltaNet", section "DeltaNet 与 Gated Delta Rule") is the
 *   case where g_t is one number per head, broadcast over the d_k channels.
 *   When beta is NULL the step is the decay-only recurrence S <- Diag(a_t) S + k_t v_t^T
 *   ("TileLang 实战：KDA 从零到一--标量衰减", §1.1; "07 · linear 路线（二）：衰减机制的
 *   演进", §0), i.e. u = v.
 *
 * Readings taken where the pages leave a choice open:
 *   - scale multiplies the output only; it never touches the state;
 *   - the final state is the state after the last token of each sequence, in the
 *     transposed layout [d_k][d_v];
 *   - inputs are read as float32 (bf16 and fp32 values are exact there) and widened to
 *     fp64; every operation is done in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v, *g, *beta, *h0;
    const int64_t *seq_off; /* N + 1 token offsets */
    int N, H_k, H_v, d_k, d_v, gate_per_channel;
    double scale;
    const int32_t *units; /* unit = n * H_v + h */
    int n_units;
    const int64_t *o_row; /* first output row of each unit in o */
    double *o;            /* rows of d_v values */
    double *ht;           /* n_units blocks of d_k * d_v values */
    int next;
    int status;
    pthread_mutex_t mu;
} kda_job;

/* One (sequence, value head) unit: the recurrence over every token of the sequence. */
static void run_unit(const kda_job *J, int ui, double *S, double *a, double *u)
{
    const int unit = J->units[ui];
    const int n = unit / J->H_v, h = unit % J->H_v;
    const int hk = h / (J->H_v / J->H_k);
    const int dk = J->d_k, dv = J->d_v;
    const int64_t bos = J->seq_off[n], eos = J->seq_off[n + 1];
    double *orow = J->o + J->o_row[ui] * (int64_t)dv;
    double *ht = J->ht + (int64_t)ui * dk * dv;

    if (J->h0) {
        const float *h0 = J->h0 + ((int64_t)n * J->H_v + h) * dk * dv;
        for (int64_t i = 0; i < (int64_t)dk * dv; ++i) S[i] = (double)h0[i];
    } else {
        memset(S, 0, sizeof(double) * (size_t)dk * dv);
    }

    for (int64_t t = bos; t < eos; ++t) {
        const float *qt = J->q + (t * J->H_k + hk) * dk;
        const float *kt = J->k + (t * J->H_k + hk) * dk;
        const float *vt = J->v + (t * J->H_v + h) * dv;

        for (int i = 0; i < dk; ++i) {
            const double gi = J->gate_per_channel ? (double)J->g[(t * J->H_v + h) * dk + i]
                                                  : (double)J->g[t * J->H_v + h];
            a[i] = exp(gi);
        }
        /* S <- Diag(a) S */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= a[i];

        /* u <- beta (v - S^T k), or u <- v without the erase term */
        for (int j = 0; j < dv; ++j) u[j] = (double)vt[j];
        if (J->beta) {
            for (int i = 0; i < dk; ++i) {
                const double ki = (double)kt[i];
                for (int j = 0; j < dv; ++j) u[j] -= S[(int64_t)i * dv + j] * ki;
            }
            const double b = (double)J->beta[t * J->H_v + h];
            for (int j = 0; j < dv; ++j) u[j] *= b;
        }

        /* S <- S + k u^T */
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += ki * u[j];
        }

        /* o_t <- scale S^T q */
        double *ot = orow + (t - bos) * dv;
        for (int j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double qi = (double)qt[i];
            for (int j = 0; j < dv; ++j) ot[j] += S[(int64_t)i * dv + j] * qi;
        }
        for (int j = 0; j < dv; ++j) ot[j] *= J->scale;
    }
    memcpy(ht, S, sizeof(double) * (size_t)dk * dv);
}

static void *worker(void *arg)
{
    kda_job *J = (kda_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->d_k * J->d_v);
    double *a = (double *)malloc(sizeof(double) * (size_t)J->d_k);
    double *u = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    if (!S || !a || !u) {
        pthread_mutex_lock(&J->mu);
        J->status = -2;
        pthread_mutex_unlock(&J->mu);
        free(S); free(a); free(u);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int ui = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (ui >= J->n_units) break;
        run_unit(J, ui, S, a, u);
    }
    free(S); free(a); free(u);
    return NULL;
}

/*
 * kda_oracle_fwd: run the token recurrence for the listed (sequence, value head) units.
 *
 * q, k   [T_total, H_k, d_k] float32   (bf16 inputs passed as their exact fp32 values)
 * v      [T_total, H_v, d_v] float32
 * g      [T_total, H_v, d_k] (gate_per_channel = 1) or [T_total, H_v] (= 0), natural log
 * beta   [T_total, H_v] float32, or NULL for the decay-only recurrence
 * h0     [N, H_v, d_k, d_v] float32, or NULL for a zero initial state
 * seq_off: N + 1 non-decreasing token offsets (sequence n spans [seq_off[n], seq_off[n+1]))
 * units: n_units unit ids u = n * H_v + h; value head h reads key head h / (H_v / H_k)
 * o_row: first output row of each unit inside o (rows of d_v doubles)
 * ht:    n_units blocks of [d_k][d_v] doubles (the state after the last token)
 * n_threads <= 0 uses every online core.
 * Returns 0 on success, -1 on an invalid argument, -2 when memory runs out.
 */
int kda_oracle_fwd(const float *q, const float *k, const float *v, const float *g,
                   int gate_per_channel, const float *beta, const float *h0,
                   const int64_t *seq_off, int N, int H_k, int H_v, int d_k, int d_v,
                   double scale, const int32_t *units, int n_units, const int64_t *o_row,
                   double *o, double *ht, int n_threads)
{
    if (!q || !k || !v || !g || !seq_off || !units || !o_row || !o || !ht) return -1;
    if (N < 1 || H_k < 1 || H_v < 1 || H_v % H_k != 0 || d_k < 1 || d_v < 1 || n_units < 0)
        return -1;
    for (int i = 0; i < n_units; ++i)
        if (units[i] < 0 || units[i] >= N * H_v) return -1;

    kda_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.seq_off = seq_off; J.N = N; J.H_k = H_k; J.H_v = H_v; J.d_k = d_k; J.d_v = d_v;
    J.gate_per_channel = gate_per_channel; J.scale = scale;
    J.units = units; J.n_units = n_units; J.o_row = o_row; J.o = o; J.ht = ht;
    pthread_mutex_init(&J.mu, NULL);

    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if (n_threads > n_units) n_threads = n_units > 0 ? n_units : 1;

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) { pthread_mutex_destroy(&J.mu); return -2; }
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J); /* no thread could start: do the work here */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.status;
}

/* Number of worker threads kda_oracle_fwd uses when asked for every core. */
int kda_oracle_default_threads(void)
{
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}
