/*
 * oracle.c -- plain, slow, fp64 CPU oracle for paged KV append, single-token
 * decode attention, ragged end-aligned causal prefill and the mixed step
 * (chunked prefill and multi-token decode rows in one batch).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (sources, by page title and section):
 *  - "mini-infer ... True PagedAttention" (smarter.xin), sections 1 and 3:
 *    one call writes the new token's K/V in place at index cache_seqlens[b]
 *    of the request's logical sequence, found through block_table, then
 *    attends over the paged cache with no dense copy.  Cache tensors are
 *    [num_blocks, block_size, num_kv_heads, head_dim].
 *  - same page, section 1: the replaced "gather -> dense -> attention" path;
 *    this oracle is that formulation written out: it gathers each key and
 *    value in logical order by walking block_table, then applies textbook
 *    softmax attention in fp64.
 *  - "[flashinfer] ... causal work based admission" (blog.secrett2633.cloud),
 *    code analysis part 1: with q queries and kv keys (q <= kv, end aligned)
 *    query i (0-based) sees kv - q + i + 1 keys; summing gives the pair count
 *    q(2kv - q + 1)/2 per head.  Pages there are in the HND layout
 *    [num_pages, num_kv_heads, page_size, head_dim].
 *  - "flex_attention + paged KV + CUDA graphs vs vLLM", "What broke
 *    correctness": physical page 0 is a reserved null slot and a row that
 *    sees no key must not produce NaN.  Here such a row gives out = 0 and
 *    lse = -inf.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - cache_seqlens is the length BEFORE the append; the decode attends
 *    L_b + 1 keys when new K/V are given, L_b keys otherwise.
 *  - query head h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 *  - cache_seqlens[b] < 0 marks an inactive (padding) row: no append,
 *    out = 0, lse = -inf, no error.
 *  - a needed block_table entry outside [1, num_pages), or a row whose
 *    tokens do not fit max_blocks * page_size, is a data error: the row's
 *    appends are dropped, out = 0, lse = -inf and an error bit is raised.
 *    "Needed" means touched: attention needs every page of the row, a
 *    standalone append only the pages it writes.
 *  - lse is the natural-log log-sum-exp of the scaled scores.
 *
 * All values are bf16 bit patterns (uint16).  bf16 -> double is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NHD 0
#define ORACLE_HND 1

#define ORACLE_ERR_PAGE 1     /* a needed page id outside [1, num_pages) */
#define ORACLE_ERR_OVERFLOW 2 /* tokens do not fit max_blocks * page_size */
#define ORACLE_ERR_QLEN 8     /* a malformed query range or length */

typedef struct {
    int32_t num_pages;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t layout; /* ORACLE_NHD or ORACLE_HND */
} oracle_cache;

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element offset of (physical page, slot in page, kv head, dim 0). */
static int64_t element_offset(const oracle_cache *c, int64_t page, int64_t slot, int64_t h)
{
    int64_t P = c->page_size, H = c->num_kv_heads, D = c->head_dim;
    if (c->layout == ORACLE_NHD)
        return ((page * P + slot) * H + h) * D;
    return ((page * H + h) * P + slot) * D;
}

/* Physical page holding logical token t of row b, or -1 if the table entry
 * is not a usable page. */
static int64_t page_of(const oracle_cache *c, const int32_t *block_table, int max_blocks,
                       int b, int64_t t)
{
    int64_t blk = t / c->page_size;
    if (blk >= max_blocks)
        return -1;
    int32_t page = block_table[(int64_t)b * max_blocks + blk];
    if (page < 1 || page >= c->num_pages)
        return -1;
    return page;
}

/* Error bits for a row whose tokens first .. len-1 are touched (pages of
 * all of them must be usable) and which must hold `len` tokens. */
static int range_check(const oracle_cache *c, const int32_t *block_table, int max_blocks, int b,
                       int64_t first, int64_t len)
{
    if (len > (int64_t)max_blocks * c->page_size)
        return ORACLE_ERR_OVERFLOW;
    for (int64_t t = first; t < len; t++)
        if (page_of(c, block_table, max_blocks, b, t) < 0)
            return ORACLE_ERR_PAGE;
    return 0;
}

/* Error bits for a row that reads all of its `len` tokens. */
static int row_check(const oracle_cache *c, const int32_t *block_table, int max_blocks, int b,
                     int64_t len)
{
    return range_check(c, block_table, max_blocks, b, 0, len);
}

/* Writes n_new tokens of row b at logical positions L, L+1, ... (bit copy). */
static void write_tokens(const oracle_cache *c, uint16_t *k_cache, uint16_t *v_cache,
                         const uint16_t *k_src, const uint16_t *v_src, int64_t n_new,
                         const int32_t *block_table, int max_blocks, int b, int64_t L)
{
    int64_t H = c->num_kv_heads, D = c->head_dim;
    for (int64_t i = 0; i < n_new; i++) {
        int64_t t = L + i;
        int64_t page = page_of(c, block_table, max_blocks, b, t);
        int64_t slot = t % c->page_size;
        for (int64_t h = 0; h < H; h++) {
            int64_t dst = element_offset(c, page, slot, h);
            int64_t src = (i * H + h) * D;
            memcpy(k_cache + dst, k_src + src, (size_t)D * sizeof(uint16_t));
            memcpy(v_cache + dst, v_src + src, (size_t)D * sizeof(uint16_t));
        }
    }
}

/*
 * Standalone append.  Row b receives n_b new tokens at positions
 * cache_seqlens[b] ... cache_seqlens[b] + n_b - 1, where n_b =
 * append_indptr[b+1] - append_indptr[b] (or 1 when append_indptr is NULL);
 * its K/V rows are k_new[append_indptr[b] + i] ([T, Hkv, D] bf16).
 * Only the pages receiving a token are checked (the append reads no other
 * page); a failing row appends nothing.
 * Returns the OR of the error bits; err_rows[b] (optional) gets each row's.
 */
int oracle_append(const oracle_cache *c, uint16_t *k_cache, uint16_t *v_cache,
                  const uint16_t *k_new, const uint16_t *v_new, const int32_t *append_indptr,
                  const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                  int batch, int32_t *err_rows)
{
    int64_t H = c->num_kv_heads, D = c->head_dim;
    int err_all = 0;
    for (int b = 0; b < batch; b++) {
        int64_t first = append_indptr ? append_indptr[b] : b;
        int64_t n_new = append_indptr ? append_indptr[b + 1] - append_indptr[b] : 1;
        int64_t L = cache_seqlens[b];
        int err = 0;
        if (L >= 0 && n_new > 0) {
            err = range_check(c, block_table, max_blocks, b, L, L + n_new);
            if (!err)
                write_tokens(c, k_cache, v_cache, k_new + first * H * D, v_new + first * H * D,
                             n_new, block_table, max_blocks, b, L);
        }
        if (err_rows)
            err_rows[b] = err;
        err_all |= err;
    }
    return err_all;
}

/*
 * Softmax attention of one query row over keys 0 .. n_keys-1 of row b,
 * kv head kvh, in logical order.  q points at D bf16 values.  Writes D
 * doubles to out and the natural-log log-sum-exp to *lse.  `scores` is
 * scratch of n_keys doubles.
 */
static void attend_row(const oracle_cache *c, const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_table, int max_blocks, int b, int kvh,
                       int64_t n_keys, const uint16_t *q, double scale, double *out,
                       double *lse, double *scores)
{
    int64_t D = c->head_dim;
    for (int64_t d = 0; d < D; d++)
        out[d] = 0.0;
    if (n_keys <= 0) {
        *lse = -INFINITY;
        return;
    }
    /* scores s_j = scale * <q, k_j> */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; j++) {
        int64_t page = page_of(c, block_table, max_blocks, b, j);
        const uint16_t *k = k_cache + element_offset(c, page, j % c->page_size, kvh);
        double dot = 0.0;
        for (int64_t d = 0; d < D; d++)
            dot += bf16_value(q[d]) * bf16_value(k[d]);
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }
    /* w_j = exp(s_j - m);  out = sum_j w_j v_j / sum_j w_j */
    double denom = 0.0;
    for (int64_t j = 0; j < n_keys; j++) {
        double w = exp(scores[j] - m);
        int64_t page = page_of(c, block_table, max_blocks, b, j);
        const uint16_t *v = v_cache + element_offset(c, page, j % c->page_size, kvh);
        for (int64_t d = 0; d < D; d++)
            out[d] += w * bf16_value(v[d]);
        denom += w;
    }
    for (int64_t d = 0; d < D; d++)
        out[d] /= denom;
    *lse = m + log(denom);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * Decode with fused append.  For every active row b (L_b = cache_seqlens[b]
 * >= 0): when k_new/v_new are given, token L_b's K/V (k_new[b], [B, Hkv, D])
 * are written into the cache first and the row attends L_b + 1 keys,
 * otherwise it attends L_b keys.  q is [B, Hq, D]; out [B, Hq, D] and lse
 * [B, Hq] are doubles.  If `sel` is given, only the nsel (b, h) pairs
 * sel[2i], sel[2i+1] are computed (all appends still happen); otherwise all.
 * k_cache / v_cache are modified in place (pass copies).  Returns the OR of
 * error bits; err_rows[b] (optional) gets each row's bits.
 */
int oracle_decode(const oracle_cache *c, uint16_t *k_cache, uint16_t *v_cache,
                  const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                  const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens,
                  int batch, int num_q_heads, double scale, const int32_t *sel, int nsel,
                  double *out, double *lse, int32_t *err_rows, int nthreads)
{
    int64_t D = c->head_dim;
    int group = num_q_heads / c->num_kv_heads;
    int with_new = (k_new != NULL && v_new != NULL);
    int32_t *row_err = (int32_t *)calloc((size_t)batch, sizeof(int32_t));
    int err_all = 0;

    for (int b = 0; b < batch; b++) {
        int64_t L = cache_seqlens[b];
        if (L < 0)
            continue;
        row_err[b] = row_check(c, block_table, max_blocks, b, L + with_new);
        if (!row_err[b] && with_new)
            write_tokens(c, k_cache, v_cache, k_new + (int64_t)b * c->num_kv_heads * D,
                         v_new + (int64_t)b * c->num_kv_heads * D, 1, block_table, max_blocks,
                         b, L);
        err_all |= row_err[b];
    }

    int64_t n_items = sel ? nsel : (int64_t)batch * num_q_heads;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_items; i++) {
        int b = sel ? sel[2 * i] : (int)(i / num_q_heads);
        int h = sel ? sel[2 * i + 1] : (int)(i % num_q_heads);
        int64_t L = cache_seqlens[b];
        int64_t n_keys = L < 0 || row_err[b] ? 0 : L + with_new;
        double *scores = (double *)malloc((size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
        int64_t o = (int64_t)b * num_q_heads + h;
        attend_row(c, k_cache, v_cache, block_table, max_blocks, b, h / group, n_keys,
                   q + o * D, scale, out + o * D, lse + o, scores);
        free(scores);
    }
    if (err_rows)
        memcpy(err_rows, row_err, (size_t)batch * sizeof(int32_t));
    free(row_err);
    return err_all;
}

/*
 * Ragged end-aligned causal prefill over a paged cache (no append).
 * Request b owns query tokens qo_indptr[b] .. qo_indptr[b+1]-1 (q_b of them)
 * and kv_b = kv_lens[b] cached keys; its query i sees keys 0 .. kv_b - q_b + i.
 * q and out are [total_q, Hq, D]; lse is [total_q, Hq].  If `sel` is given,
 * only the nsel (token, head) pairs sel[2i], sel[2i+1] are computed.
 * Returns the number of (query, key, head) pairs visited, or -1 on a
 * malformed request (q_b < 0 or q_b > kv_b) and -2 on a data error (then
 * err_rows flags the row, whose outputs are 0 with lse = -inf).
 */
int64_t oracle_prefill(const oracle_cache *c, const uint16_t *k_cache, const uint16_t *v_cache,
                       const uint16_t *q, const int32_t *qo_indptr, const int32_t *kv_lens,
                       const int32_t *block_table, int max_blocks, int batch, int num_q_heads,
                       double scale, const int32_t *sel, int nsel, double *out, double *lse,
                       int32_t *err_rows, int nthreads)
{
    int64_t D = c->head_dim;
    int group = num_q_heads / c->num_kv_heads;
    int64_t total_q = qo_indptr[batch];
    int32_t *row_err = (int32_t *)calloc((size_t)batch, sizeof(int32_t));
    int32_t *row_of = (int32_t *)malloc((size_t)(total_q > 0 ? total_q : 1) * sizeof(int32_t));
    int any_err = 0;
    for (int b = 0; b < batch; b++) {
        int64_t qn = qo_indptr[b + 1] - qo_indptr[b];
        if (qn < 0 || qn > kv_lens[b]) {
            free(row_err);
            free(row_of);
            return -1;
        }
        row_err[b] = row_check(c, block_table, max_blocks, b, kv_lens[b]);
        any_err |= row_err[b];
        for (int64_t t = qo_indptr[b]; t < qo_indptr[b + 1]; t++)
            row_of[t] = b;
    }

    int64_t n_items = sel ? nsel : total_q * num_q_heads;
    int64_t pairs = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : pairs)
    for (int64_t i = 0; i < n_items; i++) {
        int64_t t = sel ? sel[2 * i] : i / num_q_heads;
        int h = sel ? sel[2 * i + 1] : (int)(i % num_q_heads);
        int b = row_of[t];
        int64_t qi = t - qo_indptr[b];
        int64_t qn = qo_indptr[b + 1] - qo_indptr[b];
        int64_t n_keys = row_err[b] ? 0 : kv_lens[b] - qn + qi + 1;
        double *scores = (double *)malloc((size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
        int64_t o = t * num_q_heads + h;
        attend_row(c, k_cache, v_cache, block_table, max_blocks, b, h / group, n_keys,
                   q + o * D, scale, out + o * D, lse + o, scores);
        free(scores);
        pairs += n_keys;
    }
    if (err_rows)
        memcpy(err_rows, row_err, (size_t)batch * sizeof(int32_t));
    free(row_err);
    free(row_of);
    return any_err ? -2 : pairs;
}

/*
 * One step of a mixed batch: chunked prefill, multi-token and single-token
 * decode rows together.  Row b brings q_b = qo_indptr[b+1] - qo_indptr[b]
 * new tokens (query rows qo_indptr[b] .. qo_indptr[b+1]-1 of q, [total_q,
 * Hq, D]) on top of L_b = cache_seqlens[b] cached tokens.
 *  - With k_new / v_new ([total_q, Hkv, D]) the new tokens' K/V are written
 *    at positions L_b .. L_b + q_b - 1 first (as oracle_append: only the
 *    pages written are checked for the append) and the row holds
 *    kv_b = L_b + q_b keys; without them the caller appended already and
 *    kv_b = L_b.
 *  - Query i of the row sees keys 0 .. kv_b - q_b + i (the end-aligned
 *    causal rule of the FlashInfer page, code analysis part 1).
 * Row fates, checked in this order:
 *  - a query range outside [0, total_q] or reversed: ORACLE_ERR_QLEN, no
 *    append, no output row is written;
 *  - q_b == 0: nothing;
 *  - q_b > max_qlen: ORACLE_ERR_QLEN, no append, out = 0, lse = -inf;
 *  - L_b < 0 (inactive): no append, out = 0, lse = -inf, no error;
 *  - kv_b < q_b (attend only): ORACLE_ERR_QLEN, out = 0, lse = -inf;
 *  - overflow or a bad page among keys 0 .. kv_b - 1: the bit, out = 0,
 *    lse = -inf (the append is dropped when its own pages fail).
 * sel (optional) lists nsel (query row, head) pairs to compute; the appends
 * of every row still happen.  Returns the OR of the error bits; err_rows[b]
 * (optional) gets each row's.
 */
int oracle_mixed(const oracle_cache *c, uint16_t *k_cache, uint16_t *v_cache, const uint16_t *q,
                 const uint16_t *k_new, const uint16_t *v_new, const int32_t *qo_indptr, int64_t total_q,
                 const int32_t *block_table, int max_blocks, const int32_t *cache_seqlens, int batch,
                 int num_q_heads, int64_t max_qlen, double scale, const int32_t *sel, int nsel,
                 double *out, double *lse, int32_t *err_rows, int nthreads)
{
    int64_t H = c->num_kv_heads, D = c->head_dim;
    int group = num_q_heads / c->num_kv_heads;
    int with_new = (k_new != NULL && v_new != NULL);
    int32_t *row_err = (int32_t *)calloc((size_t)(batch > 0 ? batch : 1), sizeof(int32_t));
    int64_t *row_keys = (int64_t *)calloc((size_t)(batch > 0 ? batch : 1), sizeof(int64_t));
    int32_t *row_of = (int32_t *)malloc((size_t)(total_q > 0 ? total_q : 1) * sizeof(int32_t));
    int err_all = 0;
    for (int64_t t = 0; t < total_q; t++)
        row_of[t] = -1;

    for (int b = 0; b < batch; b++) {
        int64_t s = qo_indptr[b], e = qo_indptr[b + 1], qn = e - s;
        int64_t L = cache_seqlens[b];
        int err = 0;
        row_keys[b] = 0;
        if (s < 0 || e > total_q || qn < 0) {
            row_err[b] = ORACLE_ERR_QLEN;
            err_all |= ORACLE_ERR_QLEN;
            continue; /* no valid query rows: nothing is written */
        }
        if (qn == 0)
            continue;
        for (int64_t t = s; t < e; t++)
            row_of[t] = b;
        if (qn > max_qlen) {
            err = ORACLE_ERR_QLEN;
        } else if (L >= 0) {
            int64_t kv = with_new ? L + qn : L;
            if (with_new && !range_check(c, block_table, max_blocks, b, L, L + qn))
                write_tokens(c, k_cache, v_cache, k_new + s * H * D, v_new + s * H * D, qn,
                             block_table, max_blocks, b, L);
            if (kv < qn)
                err = ORACLE_ERR_QLEN;
            else
                err = row_check(c, block_table, max_blocks, b, kv);
            if (!err)
                row_keys[b] = kv;
        }
        row_err[b] = err;
        err_all |= err;
    }

    int64_t n_items = sel ? nsel : total_q * num_q_heads;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_items; i++) {
        int64_t t = sel ? sel[2 * i] : i / num_q_heads;
        int h = sel ? sel[2 * i + 1] : (int)(i % num_q_heads);
        int b = row_of[t];
        if (b < 0)
            continue; /* no row owns this query row */
        int64_t qn = qo_indptr[b + 1] - qo_indptr[b];
        int64_t qi = t - qo_indptr[b];
        int64_t n_keys = row_keys[b] > 0 ? row_keys[b] - qn + qi + 1 : 0;
        double *scores = (double *)malloc((size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
        int64_t o = t * num_q_heads + h;
        attend_row(c, k_cache, v_cache, block_table, max_blocks, b, h / group, n_keys,
                   q + o * D, scale, out + o * D, lse + o, scores);
        free(scores);
    }
    if (err_rows)
        memcpy(err_rows, row_err, (size_t)batch * sizeof(int32_t));
    free(row_err);
    free(row_keys);
    free(row_of);
    return err_all;
}

/* Threads an OpenMP region would use (1 when compiled without OpenMP). */
int oracle_max_threads(int nthreads)
{
#ifdef _OPENMP
    set_threads(nthreads);
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    (void)nthreads;
    return 1;
#endif
}
