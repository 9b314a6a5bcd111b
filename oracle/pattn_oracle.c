/*
 * pattn_oracle.c -- float64 CPU oracle for paged-KV varlen attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the timed CPU
 * baseline of the benchmark may load this file's library. The CUDA library
 * shares no code, header, table or helper with it.
 *
 * What it computes (plain definition, no blocking, no online softmax):
 *
 *   for every query token t of sequence b (local index i = t - cu_q[b],
 *   ql = cu_q[b+1] - cu_q[b], L = seq_lens[b]) and every query head h:
 *     kv head   hk = h / (Hq / Hkv)          (contiguous head groups: the
 *               GQA-packed Q tensor map of the trtllm-gen paged decode
 *               manifest, decode.json "tensormaps" field at byte 0, puts the
 *               group of a KV head innermost, and its fast-divmod constant
 *               0xAAAAAAAB >> 34 divides the q head by the group size 6)
 *     position  p = L - ql + i               (queries are the last ql keys)
 *     keys      J = { j : 0 <= j < L and (not causal or j <= p) }
 *     key row   page = block_table[b][j / P], row j % P of that page
 *               (decode.json buffers "kv" / "table": fixed-size pages named
 *               by a per-sequence table)
 *     s_j       = scale * sum_d q[d] * k_j[d]
 *     out       = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m),  m = max_j s_j
 *     lse       = m + log(sum_j exp(s_j - m))
 *   and out = 0, lse = -inf when J is empty.
 *
 * This is scaled dot-product attention with a causal mask aligned to the end
 * of the KV (the reading taken for the FlashAttention-4 SM100MHA2Q kernel doc,
 * "MaskType: causal or unmasked", and for the decode manifest's "Causal ...
 * VarSeq" kernel). The exp2 and log2(e) scale folding of the kernels
 * (decode.json pack scalar at byte 1220 = scale * log2 e) is the same
 * function; the oracle uses exp in double.
 *
 * Every bf16 input is widened to double exactly. Work is split over
 * (query token, query head) pairs and pthreads; each pair is summed in
 * logical key order, so the result does not depend on the thread count or
 * on which physical page holds a logical row.
 *
 * K/V addressing is stride-parameterised so that the two pool layouts seen
 * on the pages can both be checked:
 *   element (kind, page, row, head, d) = kv[page*s_page + kind*s_kv + row*s_row
 *                                           + head*s_head + d]
 * with kind 0 = K, 1 = V. With block_table == NULL the cache is contiguous:
 * sequence b's key j is row cu_kv[b] + j of page 0, cu_kv = prefix sum of L.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double widen_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q;
    const uint16_t *kv;
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    int num_seqs;
    int hq, hkv, d, page_size;
    int64_t s_page, s_kv, s_row, s_head;
    double scale;
    int causal;
    int64_t key_begin, key_end; /* logical key window [key_begin, key_end), key_end < 0: no bound */
    const int64_t *rows;        /* query tokens to compute, NULL: all */
    int64_t n_rows;
    double *out;                /* [n_rows][hq][d] */
    double *lse;                /* [n_rows][hq] or NULL */
    int64_t *cu_kv;             /* contiguous mode only */
    int64_t max_kv;
    int64_t next;
    pthread_mutex_t mu;
    int status;
} job_t;

/* Sequence owning query token t (cu_q is non-decreasing). */
static int seq_of_token(const job_t *jb, int64_t t) {
    int lo = 0, hi = jb->num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if ((int64_t)jb->cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    /* skip empty sequences that share the same start */
    while (lo + 1 < jb->num_seqs && (int64_t)jb->cu_q[lo + 1] <= t) lo++;
    return lo;
}

static const uint16_t *kv_row(const job_t *jb, int b, int64_t j, int kind, int hk) {
    if (jb->block_table) {
        int64_t slot = j / jb->page_size;
        int64_t r = j % jb->page_size;
        int64_t pg = jb->block_table[(int64_t)b * jb->bt_stride + slot];
        return jb->kv + pg * jb->s_page + kind * jb->s_kv + r * jb->s_row + hk * jb->s_head;
    }
    int64_t r = jb->cu_kv[b] + j;
    return jb->kv + kind * jb->s_kv + r * jb->s_row + hk * jb->s_head;
}

static void one_row_head(const job_t *jb, int64_t ri, int h, double *s) {
    int64_t t = jb->rows ? jb->rows[ri] : ri;
    int b = seq_of_token(jb, t);
    int64_t ql = (int64_t)jb->cu_q[b + 1] - jb->cu_q[b];
    int64_t L = jb->seq_lens[b];
    int64_t i = t - jb->cu_q[b];
    int64_t p = L - ql + i;
    int g = jb->hq / jb->hkv;
    int hk = h / g;
    int d = jb->d;
    double *o = jb->out + (ri * jb->hq + h) * (int64_t)d;
    const uint16_t *qv = jb->q + (t * jb->hq + h) * (int64_t)d;

    int64_t j0 = jb->key_begin > 0 ? jb->key_begin : 0;
    int64_t j1 = L;
    if (jb->key_end >= 0 && jb->key_end < j1) j1 = jb->key_end;
    if (jb->causal && p + 1 < j1) j1 = p + 1;

    for (int e = 0; e < d; ++e) o[e] = 0.0;
    if (j1 <= j0) {
        if (jb->lse) jb->lse[ri * jb->hq + h] = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        const uint16_t *kr = kv_row(jb, b, j, 0, hk);
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += widen_bf16(qv[e]) * widen_bf16(kr[e]);
        s[j - j0] = jb->scale * acc;
        if (s[j - j0] > m) m = s[j - j0];
    }
    double den = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double w = exp(s[j - j0] - m);
        den += w;
        const uint16_t *vr = kv_row(jb, b, j, 1, hk);
        for (int e = 0; e < d; ++e) o[e] += w * widen_bf16(vr[e]);
    }
    for (int e = 0; e < d; ++e) o[e] /= den;
    if (jb->lse) jb->lse[ri * jb->hq + h] = m + log(den);
}

static void *worker(void *arg) {
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->max_kv > 0 ? jb->max_kv : 1));
    if (!s) {
        pthread_mutex_lock(&jb->mu);
        jb->status = -2;
        pthread_mutex_unlock(&jb->mu);
        return NULL;
    }
    const int64_t total = jb->n_rows * jb->hq;
    const int64_t chunk = 8;
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t w0 = jb->next;
        jb->next += chunk;
        pthread_mutex_unlock(&jb->mu);
        if (w0 >= total) break;
        int64_t w1 = w0 + chunk < total ? w0 + chunk : total;
        for (int64_t w = w0; w < w1; ++w) one_row_head(jb, w / jb->hq, (int)(w % jb->hq), s);
    }
    free(s);
    return NULL;
}

int pattn_oracle_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Returns 0 on success, -1 on an argument error, -2 on allocation failure.
 * rows == NULL computes every query token (n_rows must then equal total_q).
 * key_end < 0 means no upper bound on the key window.
 */
int pattn_oracle_forward(double *out, double *lse, const uint16_t *q, const uint16_t *kv,
                         const int32_t *block_table, int64_t bt_stride,
                         const int32_t *seq_lens, const int32_t *cu_q, int num_seqs,
                         int n_heads_q, int n_heads_kv, int head_dim, int page_size,
                         int64_t s_page, int64_t s_kv, int64_t s_row, int64_t s_head,
                         double scale, int causal, const int64_t *rows, int64_t n_rows,
                         int64_t key_begin, int64_t key_end, int n_threads) {
    if (!out || !q || !kv || !seq_lens || !cu_q || num_seqs <= 0) return -1;
    if (n_heads_kv <= 0 || n_heads_q % n_heads_kv != 0 || head_dim <= 0) return -1;
    if (block_table && page_size <= 0) return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.kv = kv; jb.block_table = block_table; jb.bt_stride = bt_stride;
    jb.seq_lens = seq_lens; jb.cu_q = cu_q; jb.num_seqs = num_seqs;
    jb.hq = n_heads_q; jb.hkv = n_heads_kv; jb.d = head_dim; jb.page_size = page_size;
    jb.s_page = s_page; jb.s_kv = s_kv; jb.s_row = s_row; jb.s_head = s_head;
    jb.scale = scale; jb.causal = causal; jb.rows = rows; jb.n_rows = n_rows;
    jb.key_begin = key_begin; jb.key_end = key_end; jb.out = out; jb.lse = lse;
    for (int b = 0; b < num_seqs; ++b)
        if (seq_lens[b] > jb.max_kv) jb.max_kv = seq_lens[b];
    if (!block_table) {
        jb.cu_kv = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
        if (!jb.cu_kv) return -2;
        jb.cu_kv[0] = 0;
        for (int b = 0; b < num_seqs; ++b) jb.cu_kv[b + 1] = jb.cu_kv[b] + seq_lens[b];
    }
    pthread_mutex_init(&jb.mu, NULL);
    if (n_threads <= 0) n_threads = pattn_oracle_threads();
    if (n_threads > 512) n_threads = 512;
    pthread_t th[512];
    int started = 0;
    for (int k = 0; k < n_threads; ++k) {
        if (pthread_create(&th[k], NULL, worker, &jb) != 0) break;
        started++;
    }
    if (started == 0) worker(&jb);
    for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
    pthread_mutex_destroy(&jb.mu);
    free(jb.cu_kv);
    return jb.status;
}

/*
 * Log-sum-exp merge of attention results over disjoint key sets, in natural
 * logs: LSE = log sum_s exp(lse_s), out = sum_s exp(lse_s - LSE) * out_s.
 * Parts with lse_s = -inf (no visible key) carry no weight; if every part is
 * empty the result is 0 with LSE = -inf. This is the split-KV reduction the
 * decode manifest's "stats" and "partial" scratch buffers exist for.
 * out_parts: [n_parts][n][d], lse_parts: [n_parts][n]; out: [n][d]; lse: [n].
 */
void pattn_oracle_combine(double *out, double *lse, const double *out_parts,
                          const double *lse_parts, int n_parts, int64_t n, int d) {
    for (int64_t r = 0; r < n; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < n_parts; ++s)
            if (lse_parts[s * n + r] > M) M = lse_parts[s * n + r];
        for (int e = 0; e < d; ++e) out[r * d + e] = 0.0;
        if (M == -INFINITY) {
            if (lse) lse[r] = -INFINITY;
            continue;
        }
        double den = 0.0;
        for (int s = 0; s < n_parts; ++s) den += exp(lse_parts[s * n + r] - M);
        double LSE = M + log(den);
        for (int s = 0; s < n_parts; ++s) {
            double w = exp(lse_parts[s * n + r] - LSE);
            if (w == 0.0) continue;
            const double *o = out_parts + ((int64_t)s * n + r) * d;
            for (int e = 0; e < d; ++e) out[r * d + e] += w * o[e];
        }
        if (lse) lse[r] = LSE;
    }
}
