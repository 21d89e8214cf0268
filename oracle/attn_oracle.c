/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of exact softmax attention,
 * computed in fp64. It exists so the CUDA path can be checked against it; no
 * product code may link or call it (only tests, the smoke check and the
 * benchmark's CPU-baseline leg do).
 *
 * What it computes (the definition, written out):
 *   "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *    IO-Awareness", abstract: the method is *exact* attention, so its result
 *   is softmax(Q K^T * scale) V, with nothing approximated.
 *   "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
 *    Low-precision", abstract and core claim: the same exact layer, sped up.
 *
 * For one query row i of sequence s and query head h (kv head hk = h / (H/Hkv),
 * i.e. H/Hkv consecutive query heads share one K/V head):
 *   allowed(j) = j < n_s and (not causal or j <= i)
 *   s_j  = scale * sum_c q[i,h,c] * k[j,hk,c]
 *   m    = max over allowed j of s_j
 *   w_j  = exp(s_j - m),  L = sum_j w_j
 *   o[c] = sum_j (w_j / L) * v[j,hk,c]
 *   lse  = m + ln(L)                       (natural log, scale included)
 * Two plain passes per row over a materialised score row; no tiling, no
 * online rescaling, no reordering beyond what the definition states.
 *
 * Inputs are fp32 arrays holding the exact values the GPU sees (bf16/fp16
 * widen to fp32 without rounding); all arithmetic is fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const float *q, *k, *v;
    int64_t q_tok_stride, kv_tok_stride; /* elements between consecutive tokens */
    int H, Hkv, d;
    const int64_t *seq_start, *seq_len;  /* per sequence: first token, length */
    int64_t nrows;
    const int64_t *row_seq, *row_head, *row_i;
    int causal;
    double scale;
    double *o, *lse;
    int64_t next;           /* shared work counter (rows handed out in chunks) */
    pthread_mutex_t lock;
} job_t;

static void one_row(const job_t *J, int64_t r, double *srow)
{
    const int64_t s = J->row_seq[r], h = J->row_head[r], i = J->row_i[r];
    const int d = J->d;
    const int64_t group = J->H / J->Hkv;
    const int64_t hk = h / group;
    const int64_t start = J->seq_start[s], n = J->seq_len[s];
    const int64_t nkeys = J->causal ? (i + 1 < n ? i + 1 : n) : n;
    const float *qi = J->q + (start + i) * J->q_tok_stride + h * d;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const float *kj = J->k + (start + j) * J->kv_tok_stride + hk * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += (double)qi[c] * (double)kj[c];
        srow[j] = J->scale * acc;
        if (srow[j] > m) m = srow[j];
    }
    /* pass 2: normaliser, then the weighted sum of V rows */
    double L = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        srow[j] = exp(srow[j] - m);
        L += srow[j];
    }
    double *oi = J->o + r * d;
    for (int c = 0; c < d; ++c) oi[c] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const float *vj = J->v + (start + j) * J->kv_tok_stride + hk * d;
        const double w = srow[j] / L;
        for (int c = 0; c < d; ++c) oi[c] += w * (double)vj[c];
    }
    J->lse[r] = m + log(L);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int64_t maxlen = 0;
    for (int64_t r = 0; r < J->nrows; ++r) {
        const int64_t n = J->seq_len[J->row_seq[r]];
        if (n > maxlen) maxlen = n;
    }
    double *srow = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!srow) return (void *)1;
    for (;;) {
        int64_t a;
        pthread_mutex_lock(&J->lock);
        a = J->next;
        J->next += 16;
        pthread_mutex_unlock(&J->lock);
        if (a >= J->nrows) break;
        const int64_t b = a + 16 < J->nrows ? a + 16 : J->nrows;
        for (int64_t r = a; r < b; ++r) one_row(J, r, srow);
    }
    free(srow);
    return NULL;
}

/*
 * Attention for an explicit list of query rows.
 *   q: token-major, q[(tok)*q_tok_stride + h*d + c]; k, v likewise with
 *   kv_tok_stride and kv head hk. Sequence s occupies tokens
 *   [seq_start[s], seq_start[s] + seq_len[s]) of q, k and v alike.
 *   Row r asks for (row_seq[r], row_head[r], row_i[r]) with row_i local to
 *   its sequence. Outputs: o[r*d + c] and lse[r].
 * Returns 0 on success, 1 on bad arguments or allocation failure.
 */
int oracle_attn_rows(const float *q, const float *k, const float *v,
                     int64_t q_tok_stride, int64_t kv_tok_stride,
                     int H, int Hkv, int d,
                     const int64_t *seq_start, const int64_t *seq_len,
                     int64_t nrows, const int64_t *row_seq, const int64_t *row_head,
                     const int64_t *row_i, int causal, double scale,
                     double *o, double *lse, int nthreads)
{
    if (H <= 0 || Hkv <= 0 || H % Hkv != 0 || d <= 0 || nrows < 0) return 1;
    job_t J;
    J.q = q; J.k = k; J.v = v;
    J.q_tok_stride = q_tok_stride; J.kv_tok_stride = kv_tok_stride;
    J.H = H; J.Hkv = Hkv; J.d = d;
    J.seq_start = seq_start; J.seq_len = seq_len;
    J.nrows = nrows; J.row_seq = row_seq; J.row_head = row_head; J.row_i = row_i;
    J.causal = causal; J.scale = scale; J.o = o; J.lse = lse;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0, rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, worker, &J) == 0) ++started;
    }
    if (worker(&J) != NULL) rc = 1;
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        if (ret != NULL) rc = 1;
    }
    pthread_mutex_destroy(&J.lock);
    return rc;
}
