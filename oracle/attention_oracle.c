/*
 * attention_oracle.c — the fp64 CPU oracle for grouped-query softmax attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library: it is a plain, slow, obviously
 * correct restatement of the definition the kernels must reproduce.
 *
 * What it computes (one output row per query token i and query head h):
 *
 *   The score of key j is the scaled dot product  s_j = scale * sum_d q[d] * k_j[d],
 *   the weights are a softmax over the visible keys, and the output is the weighted
 *   sum of the value rows.  This is the row-wise formulation on the larql
 *   "Inference Engine" page, section "BLAS-Fused Attention" (per query position and
 *   head: scores from K times Q, scaling by the head scale, a two-pass softmax --
 *   max, then exp and normalise -- accumulated in double precision, then V^T times
 *   the weights).  Here every step is carried out in double precision.
 *
 *   Grouped-query attention (same page, "Supported features": any Q/KV ratio; and
 *   the lattice-inference DESIGN page, "Invariants", INV-3 and the Q-head mapping
 *   of __FA_GQA_GROUPS__): with G = n_heads / n_kv_heads, query head h reads KV
 *   head h / G (contiguous groups; the pages name the mapping but not its form, so
 *   this is the usual repeat-KV reading).
 *
 *   Masks: causal masking (larql page, "Supported features": built in) and a
 *   sliding window (hf2q "Current Inference Path" page, section 2 step 1: sliding
 *   window 1024).  Readings where the pages are silent:
 *     - the query at row i sits at absolute position p = i + (L - S) (bottom-right
 *       alignment when the key length L exceeds the query length S), so a decode
 *       step (S = 1) is the last row of a prefill over the same keys;
 *     - causal: key j is visible iff j <= p;
 *     - window W > 0: key j is visible iff p - j < W (W keys including self);
 *     - W <= 0 means no window.
 *
 *   Softcap (larql page, section "BLAS-Fused Attention", step 2 "Scale + softcap", and
 *   "Supported features": Gemma 2): when softcap > 0 the scaled score is replaced by
 *   softcap * tanh(s / softcap) before the softmax; softcap <= 0 leaves it unchanged.
 *
 *   Log-sum-exp (not on the pages; the build's reading): lse = m + ln(Z) with m the
 *   largest visible (scaled, capped) score and Z = sum_j exp(s_j - m), natural logarithm.
 *   A row with no visible key has out = 0 and lse = -inf.
 *
 * Layouts (all row-major, contiguous, double):
 *   q   [batch, seq_len, n_heads,    head_dim]
 *   k,v [batch, kv_len,  n_kv_heads, head_dim]
 *   out [n_out_rows, n_heads, head_dim]   (n_out_rows = batch*seq_len, or n_rows)
 *   lse [n_out_rows, n_heads]
 * The optional `rows` list names flattened query rows r = b*seq_len + i to compute;
 * output row t corresponds to rows[t].  Rows are independent, so a subset is exact.
 *
 * Work is spread over POSIX threads by (row, head) unit; each unit's arithmetic is
 * the plain sequential loop below, so threading changes no result bit.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v;
    double *out, *lse;
    int batch, seq_len, kv_len, n_heads, n_kv_heads, head_dim;
    int causal, window;
    double scale, softcap;
    const int64_t *rows;
    int64_t n_rows;
    int64_t unit_begin, unit_end; /* units are (output row t, head h) pairs */
} oracle_job;

/* Is key j visible from the query at absolute position p? */
static int key_visible(int j, int p, int causal, int window) {
    if (causal && j > p) return 0;
    if (window > 0 && p - j >= window) return 0;
    return 1;
}

/* One output row for query row r (= b*S + i) and query head h. */
static void attend_one(const oracle_job *jb, int64_t t, int h, double *scores) {
    const int S = jb->seq_len, L = jb->kv_len, D = jb->head_dim;
    const int64_t r = jb->rows ? jb->rows[t] : t;
    const int b = (int)(r / S), i = (int)(r % S);
    const int G = jb->n_heads / jb->n_kv_heads;
    const int hk = h / G;
    const int p = i + (L - S);

    const double *qrow = jb->q + ((int64_t)r * jb->n_heads + h) * D;
    double *orow = jb->out + (t * jb->n_heads + h) * D;
    double *lrow = jb->lse + t * jb->n_heads + h;

    /* pass 1: scores of the visible keys and their maximum */
    double m = -INFINITY;
    int n_vis = 0;
    for (int j = 0; j < L; ++j) {
        if (!key_visible(j, p, jb->causal, jb->window)) {
            scores[j] = -INFINITY;
            continue;
        }
        const double *krow = jb->k + (((int64_t)b * L + j) * jb->n_kv_heads + hk) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * krow[d];
        scores[j] = jb->scale * dot;
        if (jb->softcap > 0.0) scores[j] = jb->softcap * tanh(scores[j] / jb->softcap);
        if (scores[j] > m) m = scores[j];
        ++n_vis;
    }
    for (int d = 0; d < D; ++d) orow[d] = 0.0;
    if (n_vis == 0) {
        *lrow = -INFINITY;
        return;
    }

    /* pass 2: normaliser Z and the weighted sum of values */
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        if (!key_visible(j, p, jb->causal, jb->window)) continue;
        const double w = exp(scores[j] - m);
        Z += w;
        const double *vrow = jb->v + (((int64_t)b * L + j) * jb->n_kv_heads + hk) * D;
        for (int d = 0; d < D; ++d) orow[d] += w * vrow[d];
    }
    for (int d = 0; d < D; ++d) orow[d] /= Z;
    *lrow = m + log(Z);
}

static void *run_units(void *arg) {
    oracle_job *jb = (oracle_job *)arg;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(jb->kv_len > 0 ? jb->kv_len : 1));
    if (!scores) return (void *)1;
    for (int64_t u = jb->unit_begin; u < jb->unit_end; ++u) {
        attend_one(jb, u / jb->n_heads, (int)(u % jb->n_heads), scores);
    }
    free(scores);
    return NULL;
}

/*
 * Returns 0 on success, -1 on a bad argument, -2 on an allocation or thread failure.
 * n_threads <= 0 uses one thread.
 */
int oracle_attention_rows(const double *q, const double *k, const double *v, double *out,
                          double *lse, int batch, int seq_len, int kv_len, int n_heads,
                          int n_kv_heads, int head_dim, int causal, int window, double scale,
                          double softcap, const int64_t *rows, int64_t n_rows, int n_threads) {
    if (batch < 0 || seq_len < 0 || kv_len < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        head_dim <= 0 || n_heads % n_kv_heads != 0)
        return -1;
    if (rows) {
        for (int64_t t = 0; t < n_rows; ++t)
            if (rows[t] < 0 || rows[t] >= (int64_t)batch * seq_len) return -1;
    } else {
        n_rows = (int64_t)batch * seq_len;
    }
    const int64_t n_units = n_rows * n_heads;
    if (n_units == 0) return 0;
    if (n_threads <= 0) n_threads = 1;
    if (n_threads > n_units) n_threads = (int)n_units;

    oracle_job *jobs = (oracle_job *)calloc((size_t)n_threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0, started = 0;
    for (int t = 0; t < n_threads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->out = out; jb->lse = lse;
        jb->batch = batch; jb->seq_len = seq_len; jb->kv_len = kv_len;
        jb->n_heads = n_heads; jb->n_kv_heads = n_kv_heads; jb->head_dim = head_dim;
        jb->causal = causal; jb->window = window; jb->scale = scale; jb->softcap = softcap;
        jb->rows = rows; jb->n_rows = n_rows;
        jb->unit_begin = n_units * t / n_threads;
        jb->unit_end = n_units * (t + 1) / n_threads;
        if (t == 0) continue; /* thread 0's share runs on the calling thread */
        if (pthread_create(&tids[t], NULL, run_units, jb) != 0) {
            rc = -2;
            break;
        }
        started = t;
    }
    if (rc == 0 && run_units(&jobs[0]) != NULL) rc = -2;
    for (int t = 1; t <= started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret != NULL) rc = -2;
    }
    free(jobs);
    free(tids);
    return rc;
}
