/*
 * Paged-attention forward: plain, slow, fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or table with
 * the CUDA library.
 *
 * What it computes, and where that is stated:
 *
 *  - Decode step ("Perhatian berhalaman", HF transformers docs, section
 *    "Jalur decode": Perilaku cache / Mekanisme pengindeksan / Contoh):
 *    one query per sequence; the cache is reached through
 *    block_table[batch, max_blocks_per_seq]; cache_seqlens[b] is the cached
 *    key length; the new token's K/V is written in place, into the block
 *    that holds logical position cache_seqlens[b] (the worked example:
 *    30+1 fits block 2, 32+1 needs the second block, 70 lands in the third).
 *
 *  - Attention itself ("39 · PagedAttention", inference-notes, sections
 *    "1. Attention cần gì" and "2. Phiên bản phân trang"): walk the logical
 *    blocks in order, logical block i -> physical block table[i], score every
 *    key (dot product, one score per token), apply ONE softmax over all the
 *    scores, then walk the blocks again and sum the weighted values.  The
 *    same page states that this is exact attention, not an approximation, so
 *    the oracle is that definition written out, in the page's three passes.
 *
 *  - Varlen path ("Perhatian berhalaman", section "Jalur Varlen": Mekanisme
 *    pengindeksan / Contoh): requests are packed along the token axis and
 *    located with the cumulative lengths cu_seq_lens_q / cu_seq_lens_k.
 *    The cache is read and written by a separate update step (section
 *    "Perilaku cache"), which pa_oracle_cache_update restates.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes): cache layout [num_blocks, block_size, num_kv_heads, head_dim];
 * the new token is attended (attended length cache_seqlens[b] + 1);
 * cache_seqlens is not updated by the call; softmax scale 1/sqrt(head_dim)
 * unless given; q head h reads kv head h / (num_heads / num_kv_heads);
 * causal masking is bottom-right aligned (query i of a request with q
 * length ql and k length kl sees key j iff j <= i + kl - ql); a query with
 * no visible key returns a zero row.
 *
 * Element types: dtype 0 = IEEE fp32, dtype 1 = bfloat16 (upper 16 bits of
 * an fp32).  Both upcast exactly to fp64.  Writes into the pool are bitwise
 * copies of the stored element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARGS (-1)
#define OR_ERR_BAD_BLOCK (-2) /* a needed block_table entry is <0 or >= num_blocks */
#define OR_ERR_OVERFLOW (-3)  /* position beyond max_blocks_per_seq * block_size */
#define OR_ERR_BAD_CU (-4)    /* cumulative lengths inconsistent */

static size_t elt_size(int dtype) { return dtype == 1 ? 2u : 4u; }

/* exact upcast of element i of a dtype array to fp64 */
static double load_elt(const void *base, int64_t i, int dtype)
{
    if (dtype == 1) {
        uint16_t h = ((const uint16_t *)base)[i];
        uint32_t bits = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
    return (double)((const float *)base)[i];
}

static void copy_elts(void *dst, int64_t di, const void *src, int64_t si, int64_t n, int dtype)
{
    size_t e = elt_size(dtype);
    memcpy((char *)dst + (size_t)di * e, (const char *)src + (size_t)si * e, (size_t)n * e);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int pa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Offset, in elements, of (physical block p, slot s, kv head h, dim 0) in a
 * pool laid out [num_blocks, block_size, num_kv_heads, head_dim]. */
static int64_t pool_row(int64_t p, int64_t s, int64_t h, int block_size, int hkv, int d)
{
    return ((p * block_size + s) * hkv + h) * (int64_t)d;
}

/*
 * Physical location of logical position `pos` of sequence b: the block is
 * table[b][pos / block_size], the slot pos % block_size ("Jalur decode",
 * Contoh; "2. Phiên bản phân trang": logical block i -> physical table[i]).
 * Returns 0, or an OR_ERR_* code for an entry that is not a valid block.
 */
static int locate(const int32_t *block_table, int b, int pos, int block_size,
                  int max_blocks_per_seq, int num_blocks, int64_t *phys, int *slot)
{
    int lb = pos / block_size;
    if (pos < 0 || lb >= max_blocks_per_seq) return OR_ERR_OVERFLOW;
    int32_t p = block_table[(int64_t)b * max_blocks_per_seq + lb];
    if (p < 0 || p >= num_blocks) return OR_ERR_BAD_BLOCK;
    *phys = p;
    *slot = pos % block_size;
    return OR_OK;
}

/*
 * Softmax-weighted sum for ONE query row over n keys that the caller has
 * already scored: w = softmax(scores), out = sum_j w_j * V_j.  Pass 2 and 3
 * of the page's description ("áp một softmax trên tất cả", then the weighted
 * sum of values).  vrow(j) gives the element offset of key j's value row.
 * n == 0 gives a zero row.
 */
static void softmax_weighted_sum(const double *scores, int n, const void *v, const int64_t *vrow,
                                 int d, int dtype, double *out)
{
    for (int k = 0; k < d; ++k) out[k] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (scores[j] > m) m = scores[j];
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += exp(scores[j] - m);
    for (int j = 0; j < n; ++j) {
        double w = exp(scores[j] - m) / l;
        for (int k = 0; k < d; ++k) out[k] += w * load_elt(v, vrow[j] + k, dtype);
    }
}

/*
 * Decode step.
 *   q       [batch, num_heads, head_dim]
 *   k_cache [num_blocks, block_size, num_kv_heads, head_dim]   (modified: append)
 *   v_cache same layout                                         (modified: append)
 *   block_table [batch, max_blocks_per_seq] int32, -1 = not allocated
 *   cache_seqlens [batch] int32: keys already cached (read only)
 *   k_new, v_new [batch, num_kv_heads, head_dim]
 *   out     [batch, num_heads, head_dim] fp64
 * softmax_scale <= 0 selects 1/sqrt(head_dim).
 * Step 1 writes every sequence's new K/V first; step 2 attends over
 * positions 0..cache_seqlens[b] inclusive in logical order.
 */
int pa_oracle_decode(const void *q, void *k_cache, void *v_cache, const int32_t *block_table,
                     const int32_t *cache_seqlens, const void *k_new, const void *v_new,
                     double *out, int batch, int num_heads, int num_kv_heads, int head_dim,
                     int num_blocks, int block_size, int max_blocks_per_seq, int dtype,
                     double softmax_scale, int nthreads)
{
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_heads % num_kv_heads != 0 || (dtype != 0 && dtype != 1))
        return OR_ERR_ARGS;
    const int g = num_heads / num_kv_heads;
    const double scale = softmax_scale > 0 ? softmax_scale : 1.0 / sqrt((double)head_dim);
    const int rowlen = num_kv_heads * head_dim;

    /* step 1: in-place append at logical position cache_seqlens[b] */
    for (int b = 0; b < batch; ++b) {
        int64_t p;
        int s;
        int rc = locate(block_table, b, cache_seqlens[b], block_size, max_blocks_per_seq,
                        num_blocks, &p, &s);
        if (rc != OR_OK) return rc;
        copy_elts(k_cache, pool_row(p, s, 0, block_size, num_kv_heads, head_dim), k_new,
                  (int64_t)b * rowlen, rowlen, dtype);
        copy_elts(v_cache, pool_row(p, s, 0, block_size, num_kv_heads, head_dim), v_new,
                  (int64_t)b * rowlen, rowlen, dtype);
    }
    /* every position that will be read must resolve to a valid block */
    for (int b = 0; b < batch; ++b) {
        int t = cache_seqlens[b] + 1;
        for (int pos = 0; pos < t; pos += block_size) {
            int64_t p;
            int s;
            int rc = locate(block_table, b, pos, block_size, max_blocks_per_seq, num_blocks, &p, &s);
            if (rc != OR_OK) return rc;
        }
    }

    set_threads(nthreads);
    int64_t work = (int64_t)batch * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < work; ++bh) {
        int b = (int)(bh / num_heads), h = (int)(bh % num_heads);
        int hk = h / g;
        int t = cache_seqlens[b] + 1;
        double *scores = (double *)malloc(sizeof(double) * (size_t)t);
        int64_t *krow = (int64_t *)malloc(sizeof(int64_t) * (size_t)t);
        /* pass 1: walk logical blocks in order, one score per token */
        for (int j = 0; j < t; ++j) {
            int64_t p;
            int s;
            locate(block_table, b, j, block_size, max_blocks_per_seq, num_blocks, &p, &s);
            krow[j] = pool_row(p, s, hk, block_size, num_kv_heads, head_dim);
            double dot = 0.0;
            for (int k = 0; k < head_dim; ++k)
                dot += load_elt(q, ((int64_t)b * num_heads + h) * head_dim + k, dtype) *
                       load_elt(k_cache, krow[j] + k, dtype);
            scores[j] = scale * dot;
        }
        /* passes 2 and 3: one softmax, then the weighted sum of V (same rows) */
        softmax_weighted_sum(scores, t, v_cache, krow, head_dim, dtype,
                             out + ((int64_t)b * num_heads + h) * head_dim);
        free(scores);
        free(krow);
    }
    return OR_OK;
}

/*
 * Plain attention of one query row over contiguous K/V rows: the
 * non-paged ("kernel liền mạch") computation the pages compare against.
 *   q [head_dim], k/v [n, row_stride] with the head's row at offset
 *   head_off, out [head_dim] fp64.
 */
int pa_oracle_attend_contiguous(const void *q, const void *k, const void *v, int n, int head_dim,
                                int64_t row_stride, int64_t head_off, int dtype,
                                double softmax_scale, double *out)
{
    if (n < 0 || head_dim <= 0) return OR_ERR_ARGS;
    const double scale = softmax_scale > 0 ? softmax_scale : 1.0 / sqrt((double)head_dim);
    double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) {
        rows[j] = (int64_t)j * row_stride + head_off;
        double dot = 0.0;
        for (int kk = 0; kk < head_dim; ++kk)
            dot += load_elt(q, kk, dtype) * load_elt(k, rows[j] + kk, dtype);
        scores[j] = scale * dot;
    }
    softmax_weighted_sum(scores, n, v, rows, head_dim, dtype, out);
    free(scores);
    free(rows);
    return OR_OK;
}

/*
 * Varlen cache update ("Jalur Varlen", Perilaku cache: the varlen kernel
 * cannot reach the paged cache, so the cache is written and read by a
 * separate update step).
 *   k_chunk/v_chunk [total_q, num_kv_heads, head_dim]: the new tokens of all
 *       requests, packed by cu_seq_lens_q.
 *   prefix_lens [batch]: tokens of request b already in the cache; chunk row
 *       i of request b goes to logical position prefix_lens[b] + i.
 *   k_full/v_full (optional, both or neither) [total_k, num_kv_heads,
 *       head_dim]: request b's rows [cu_seq_lens_k[b], cu_seq_lens_k[b+1])
 *       receive positions 0 .. prefix_lens[b] + q_len - 1, the prefix read
 *       back from the pool and then the chunk.
 * All writes are bitwise copies.
 */
int pa_oracle_cache_update(const void *k_chunk, const void *v_chunk, const int32_t *cu_seq_lens_q,
                           const int32_t *prefix_lens, const int32_t *block_table, void *k_cache,
                           void *v_cache, void *k_full, void *v_full,
                           const int32_t *cu_seq_lens_k, int batch, int num_kv_heads,
                           int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                           int dtype)
{
    if (batch < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return OR_ERR_ARGS;
    if ((k_full == NULL) != (v_full == NULL) || (k_full != NULL && cu_seq_lens_k == NULL))
        return OR_ERR_ARGS;
    const int rowlen = num_kv_heads * head_dim;
    for (int b = 0; b < batch; ++b) {
        int ql = cu_seq_lens_q[b + 1] - cu_seq_lens_q[b];
        if (ql < 0 || prefix_lens[b] < 0) return OR_ERR_BAD_CU;
        if (k_full != NULL && cu_seq_lens_k[b + 1] - cu_seq_lens_k[b] != prefix_lens[b] + ql)
            return OR_ERR_BAD_CU;
        /* scatter: chunk row i -> logical position prefix + i */
        for (int i = 0; i < ql; ++i) {
            int64_t p;
            int s;
            int rc = locate(block_table, b, prefix_lens[b] + i, block_size, max_blocks_per_seq,
                            num_blocks, &p, &s);
            if (rc != OR_OK) return rc;
            int64_t src = (int64_t)(cu_seq_lens_q[b] + i) * rowlen;
            int64_t dst = pool_row(p, s, 0, block_size, num_kv_heads, head_dim);
            copy_elts(k_cache, dst, k_chunk, src, rowlen, dtype);
            copy_elts(v_cache, dst, v_chunk, src, rowlen, dtype);
        }
    }
    if (k_full == NULL) return OR_OK;
    /* gather: the whole key sequence of each request, in logical order */
    for (int b = 0; b < batch; ++b) {
        int kl = cu_seq_lens_k[b + 1] - cu_seq_lens_k[b];
        for (int pos = 0; pos < kl; ++pos) {
            int64_t p;
            int s;
            int rc = locate(block_table, b, pos, block_size, max_blocks_per_seq, num_blocks, &p, &s);
            if (rc != OR_OK) return rc;
            int64_t src = pool_row(p, s, 0, block_size, num_kv_heads, head_dim);
            int64_t dst = (int64_t)(cu_seq_lens_k[b] + pos) * rowlen;
            copy_elts(k_full, dst, k_cache, src, rowlen, dtype);
            copy_elts(v_full, dst, v_cache, src, rowlen, dtype);
        }
    }
    return OR_OK;
}

/*
 * Varlen attention ("Jalur Varlen", Mekanisme pengindeksan / Contoh).
 *   q [total_q, num_heads, head_dim], k/v [total_k, num_kv_heads, head_dim]
 *   request r owns q rows [cu_q[r], cu_q[r+1]) and k rows [cu_k[r], cu_k[r+1])
 *   out [total_q, num_heads, head_dim] fp64
 * causal != 0: query i sees key j iff j <= i + kl - ql (bottom-right).
 * A query with no visible key (kl == 0, or masked out) gets a zero row.
 */
int pa_oracle_varlen(const void *q, const void *k, const void *v, const int32_t *cu_seq_lens_q,
                     const int32_t *cu_seq_lens_k, int batch, int num_heads, int num_kv_heads,
                     int head_dim, int causal, int dtype, double softmax_scale, double *out,
                     int nthreads)
{
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_heads % num_kv_heads != 0 || (dtype != 0 && dtype != 1))
        return OR_ERR_ARGS;
    for (int r = 0; r < batch; ++r)
        if (cu_seq_lens_q[r + 1] < cu_seq_lens_q[r] || cu_seq_lens_k[r + 1] < cu_seq_lens_k[r])
            return OR_ERR_BAD_CU;
    const int g = num_heads / num_kv_heads;
    const double scale = softmax_scale > 0 ? softmax_scale : 1.0 / sqrt((double)head_dim);
    const int64_t total_q = cu_seq_lens_q[batch];
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t qh = 0; qh < total_q * num_heads; ++qh) {
        int64_t row = qh / num_heads;
        int h = (int)(qh % num_heads), hk = h / g;
        int r = 0;
        while (cu_seq_lens_q[r + 1] <= row) ++r; /* request that owns this row */
        int ql = cu_seq_lens_q[r + 1] - cu_seq_lens_q[r];
        int kl = cu_seq_lens_k[r + 1] - cu_seq_lens_k[r];
        int i = (int)(row - cu_seq_lens_q[r]);
        int n = kl;
        if (causal) {
            n = i + kl - ql + 1;
            if (n < 0) n = 0;
            if (n > kl) n = kl;
        }
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
        for (int j = 0; j < n; ++j) {
            rows[j] = ((int64_t)(cu_seq_lens_k[r] + j) * num_kv_heads + hk) * head_dim;
            double dot = 0.0;
            for (int kk = 0; kk < head_dim; ++kk)
                dot += load_elt(q, (row * num_heads + h) * head_dim + kk, dtype) *
                       load_elt(k, rows[j] + kk, dtype);
            scores[j] = scale * dot;
        }
        softmax_weighted_sum(scores, n, v, rows, head_dim, dtype,
                             out + (row * num_heads + h) * head_dim);
        free(scores);
        free(rows);
    }
    return OR_OK;
}
