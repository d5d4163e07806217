/*
 * Oracle for the backward pass of the gated delta rule with a per-channel gate.
 *
 * TEST INFRASTRUCTURE ONLY. Plain, slow fp64 CPU code; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it. It shares no code with the CUDA path.
 *
 * What it computes: the gradients of L = sum(dO * O) + sum(dht * ht) with respect to q,
 * k, v, g, beta and h0, where O and ht are the outputs of the token recurrence that
 * kda_oracle.c states (transposed state S in R^{d_k x d_v}, a_t = exp(g_t)):
 *     S'  = Diag(a_t) S_{t-1}
 *     w   = S'^T k_t
 *     u   = beta_t (v_t - w)          (u = v_t without beta: the decay-only recurrence)
 *     S_t = S' + k_t u^T
 *     o_t = scale S_t^T q_t
 * "Gated DeltaNet", section "反向传播：状态伴随与三角变换梯度", derives the same gradients
 * for the chunk form (a state adjoint carried backwards from dht, reset per sequence, and
 * ending in dh0). This file states the plain definition instead: reverse-mode
 * differentiation of the recurrence above, token by token, in reverse order:
 *     dS  += scale q_t do_t^T                 dq_t  = scale S_t do_t
 *     dk_t = dS u                             du    = dS^T k_t
 *     dbeta_t = du . (v_t - w)                dv_t  = beta_t du       dw = -beta_t du
 *     dS' = dS + k_t dw^T                     dk_t += S' dw
 *     dg_t[i] = a_t[i] sum_j dS'[i][j] S_{t-1}[i][j]   (summed over i for a per-head gate)
 *     dS  = Diag(a_t) dS'
 * (without beta: dv_t = du and the w terms vanish). After the first token, dh0 = dS.
 *
 * The states S_0 .. S_{len-1} of a unit are kept from a forward sweep (len * d_k * d_v
 * doubles) and each reverse step recomputes S', w, u and S_t from S_{t-1}, so the reverse
 * sweep sees exactly the forward's values. Inputs are read as float32 and widened to fp64;
 * every operation is done in fp64.
 *
 * Each unit (sequence n, value head h) writes its own rows: dq and dk of the key head
 * are returned per value head, and the caller sums the value heads of a group.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v, *g, *beta, *h0, *dO, *dht;
    const int64_t *seq_off;
    int N, H_k, H_v, d_k, d_v, gate_per_channel;
    double scale;
    const int32_t *units;
    int n_units;
    const int64_t *row; /* first token row of each unit inside the per-unit outputs */
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
    int next;
    int status;
    pthread_mutex_t mu;
} kda_bwd_job;

typedef struct {
    double *S;    /* states S_0 .. S_{len-1}, then scratch */
    double *Sp;   /* S' */
    double *St;   /* S_t */
    double *dS;   /* adjoint */
    double *a, *w, *u, *du, *dw;
    int64_t cap;  /* tokens S has room for */
} bwd_ws;

static int ws_reserve(bwd_ws *W, int64_t len, int dk, int dv)
{
    const size_t m = (size_t)dk * dv;
    if (len > W->cap) {
        free(W->S);
        W->S = (double *)malloc(sizeof(double) * m * (size_t)(len > 0 ? len : 1));
        if (!W->S) { W->cap = 0; return -2; }
        W->cap = len;
    }
    return 0;
}

static void run_unit_bwd(const kda_bwd_job *J, int ui, bwd_ws *W)
{
    const int unit = J->units[ui];
    const int n = unit / J->H_v, h = unit % J->H_v;
    const int hk = h / (J->H_v / J->H_k);
    const int dk = J->d_k, dv = J->d_v;
    const int64_t m = (int64_t)dk * dv;
    const int64_t bos = J->seq_off[n], eos = J->seq_off[n + 1], len = eos - bos;
    const int gd = J->gate_per_channel ? dk : 1;
    double *dq = J->dq + J->row[ui] * dk, *dkk = J->dk + J->row[ui] * dk;
    double *dvv = J->dv + J->row[ui] * dv, *dg = J->dg + J->row[ui] * gd;
    double *dbeta = J->dbeta + J->row[ui];
    double *dh0 = J->dh0 + (int64_t)ui * m;
    double *S = W->S, *Sp = W->Sp, *St = W->St, *dS = W->dS;
    double *a = W->a, *w = W->w, *u = W->u, *du = W->du, *dw = W->dw;

    /* forward sweep: keep S_{t-1} for every token t */
    double *cur = St; /* the running state */
    if (J->h0) {
        const float *h0 = J->h0 + ((int64_t)n * J->H_v + h) * m;
        for (int64_t i = 0; i < m; ++i) cur[i] = (double)h0[i];
    } else {
        memset(cur, 0, sizeof(double) * (size_t)m);
    }
    for (int64_t t = 0; t < len; ++t) {
        const int64_t r = bos + t;
        const float *kt = J->k + (r * J->H_k + hk) * dk;
        const float *vt = J->v + (r * J->H_v + h) * dv;
        memcpy(S + t * m, cur, sizeof(double) * (size_t)m);
        for (int i = 0; i < dk; ++i)
            a[i] = exp(J->gate_per_channel ? (double)J->g[(r * J->H_v + h) * dk + i] : (double)J->g[r * J->H_v + h]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) cur[(int64_t)i * dv + j] *= a[i];
        for (int j = 0; j < dv; ++j) u[j] = (double)vt[j];
        if (J->beta) {
            for (int j = 0; j < dv; ++j) w[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) w[j] += cur[(int64_t)i * dv + j] * (double)kt[i];
            const double b = (double)J->beta[r * J->H_v + h];
            for (int j = 0; j < dv; ++j) u[j] = b * (u[j] - w[j]);
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) cur[(int64_t)i * dv + j] += (double)kt[i] * u[j];
    }

    /* reverse sweep */
    if (J->dht) {
        const float *d = J->dht + ((int64_t)n * J->H_v + h) * m;
        for (int64_t i = 0; i < m; ++i) dS[i] = (double)d[i];
    } else {
        memset(dS, 0, sizeof(double) * (size_t)m);
    }
    for (int64_t t = len - 1; t >= 0; --t) {
        const int64_t r = bos + t;
        const float *qt = J->q + (r * J->H_k + hk) * dk;
        const float *kt = J->k + (r * J->H_k + hk) * dk;
        const float *vt = J->v + (r * J->H_v + h) * dv;
        const float *dot = J->dO + (r * J->H_v + h) * dv;
        const double *Sprev = S + t * m;
        const double b = J->beta ? (double)J->beta[r * J->H_v + h] : 1.0;

        /* recompute S', w, u and S_t */
        for (int i = 0; i < dk; ++i)
            a[i] = exp(J->gate_per_channel ? (double)J->g[(r * J->H_v + h) * dk + i] : (double)J->g[r * J->H_v + h]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) Sp[(int64_t)i * dv + j] = a[i] * Sprev[(int64_t)i * dv + j];
        for (int j = 0; j < dv; ++j) w[j] = 0.0;
        if (J->beta)
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) w[j] += Sp[(int64_t)i * dv + j] * (double)kt[i];
        for (int j = 0; j < dv; ++j) u[j] = J->beta ? b * ((double)vt[j] - w[j]) : (double)vt[j];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) St[(int64_t)i * dv + j] = Sp[(int64_t)i * dv + j] + (double)kt[i] * u[j];

        /* o_t = scale S_t^T q_t */
        for (int i = 0; i < dk; ++i) {
            double s = 0.0;
            for (int j = 0; j < dv; ++j) {
                dS[(int64_t)i * dv + j] += J->scale * (double)qt[i] * (double)dot[j];
                s += St[(int64_t)i * dv + j] * (double)dot[j];
            }
            dq[t * dk + i] = J->scale * s;
        }
        /* S_t = S' + k u^T */
        for (int j = 0; j < dv; ++j) du[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            double s = 0.0;
            for (int j = 0; j < dv; ++j) {
                s += dS[(int64_t)i * dv + j] * u[j];
                du[j] += dS[(int64_t)i * dv + j] * (double)kt[i];
            }
            dkk[t * dk + i] = s;
        }
        /* u = beta (v - w), w = S'^T k */
        if (J->beta) {
            double db = 0.0;
            for (int j = 0; j < dv; ++j) {
                db += du[j] * ((double)vt[j] - w[j]);
                dvv[t * dv + j] = b * du[j];
                dw[j] = -b * du[j];
            }
            dbeta[t] = db;
            for (int i = 0; i < dk; ++i) {
                double s = 0.0;
                for (int j = 0; j < dv; ++j) {
                    dS[(int64_t)i * dv + j] += (double)kt[i] * dw[j];
                    s += Sp[(int64_t)i * dv + j] * dw[j];
                }
                dkk[t * dk + i] += s;
            }
        } else {
            for (int j = 0; j < dv; ++j) dvv[t * dv + j] = du[j];
            dbeta[t] = 0.0;
        }
        /* S' = Diag(a) S_{t-1} */
        double dgh = 0.0;
        for (int i = 0; i < dk; ++i) {
            double s = 0.0;
            for (int j = 0; j < dv; ++j) s += dS[(int64_t)i * dv + j] * Sprev[(int64_t)i * dv + j];
            if (J->gate_per_channel)
                dg[t * dk + i] = a[i] * s;
            else
                dgh += a[i] * s;
            for (int j = 0; j < dv; ++j) dS[(int64_t)i * dv + j] *= a[i];
        }
        if (!J->gate_per_channel) dg[t] = dgh;
    }
    memcpy(dh0, dS, sizeof(double) * (size_t)m);
}

static void *bwd_worker(void *arg)
{
    kda_bwd_job *J = (kda_bwd_job *)arg;
    const size_t m = (size_t)J->d_k * J->d_v;
    bwd_ws W;
    memset(&W, 0, sizeof(W));
    W.Sp = (double *)malloc(sizeof(double) * m);
    W.St = (double *)malloc(sizeof(double) * m);
    W.dS = (double *)malloc(sizeof(double) * m);
    W.a = (double *)malloc(sizeof(double) * (size_t)J->d_k);
    W.w = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    W.u = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    W.du = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    W.dw = (double *)malloc(sizeof(double) * (size_t)J->d_v);
    int ok = W.Sp && W.St && W.dS && W.a && W.w && W.u && W.du && W.dw;
    for (; ok;) {
        pthread_mutex_lock(&J->mu);
        const int ui = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (ui >= J->n_units) break;
        const int n = J->units[ui] / J->H_v;
        if (ws_reserve(&W, J->seq_off[n + 1] - J->seq_off[n], J->d_k, J->d_v) != 0) { ok = 0; break; }
        run_unit_bwd(J, ui, &W);
    }
    if (!ok) {
        pthread_mutex_lock(&J->mu);
        J->status = -2;
        pthread_mutex_unlock(&J->mu);
    }
    free(W.S); free(W.Sp); free(W.St); free(W.dS);
    free(W.a); free(W.w); free(W.u); free(W.du); free(W.dw);
    return NULL;
}

/*
 * kda_oracle_bwd: gradients for the listed (sequence, value head) units.
 *
 * Inputs as kda_oracle_fwd, plus dO [T_total, H_v, d_v] and dht [N, H_v, d_k, d_v] (or
 * NULL: no gradient reaches the final state). Per-unit outputs (fp64), unit ui's rows
 * starting at row[ui] (its sequence's tokens in order):
 *   dq, dk  [rows][d_k]  this value head's part of the key head's gradient
 *   dv      [rows][d_v]
 *   dg      [rows][d_k] (per-channel gate) or [rows] (per-head gate)
 *   dbeta   [rows]      (zero without beta)
 *   dh0     n_units blocks of [d_k][d_v]
 * Returns 0, -1 for an invalid argument, -2 when memory runs out.
 */
int kda_oracle_bwd(const float *q, const float *k, const float *v, const float *g,
                   int gate_per_channel, const float *beta, const float *h0, const float *dO,
                   const float *dht, const int64_t *seq_off, int N, int H_k, int H_v, int d_k,
                   int d_v, double scale, const int32_t *units, int n_units, const int64_t *row,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0,
                   int n_threads)
{
    if (!q || !k || !v || !g || !dO || !seq_off || !units || !row || !dq || !dk || !dv || !dg ||
        !dbeta || !dh0)
        return -1;
    if (N < 1 || H_k < 1 || H_v < 1 || H_v % H_k != 0 || d_k < 1 || d_v < 1 || n_units < 0)
        return -1;
    for (int i = 0; i < n_units; ++i)
        if (units[i] < 0 || units[i] >= N * H_v) return -1;

    kda_bwd_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.dO = dO; J.dht = dht;
    J.seq_off = seq_off; J.N = N; J.H_k = H_k; J.H_v = H_v; J.d_k = d_k; J.d_v = d_v;
    J.gate_per_channel = gate_per_channel; J.scale = scale;
    J.units = units; J.n_units = n_units; J.row = row;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
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
        if (pthread_create(&th[i], NULL, bwd_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) bwd_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.status;
}
