/*
 * Reference oracle for paged GQA attention — TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct CPU statement of what the
 * attention hot path computes.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Precision: every bf16 input is widened exactly to double, and everything
 * after that (scores, softmax, weighted sum) is double with no intermediate
 * rounding.  Outputs are double.  (The encoder layer at the end of the file
 * chains several operators and rounds each one's result to bf16 before the
 * next reads it; see its section.)
 *
 * What is computed (the definition, not a fast algorithm):
 *
 *   attention of one query row q over keys K[0..n) and values V[0..n):
 *       s_j = scale * sum_d q[d] * K[j][d]
 *       p_j = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i)
 *       out = sum_j p_j * V[j]
 *   (qwenasr.cpp ARCHITECTURE.md, "Attention and RoPE" and "Qwen3 Thinker
 *   decoder": the manual F32 chain mul_mat -> soft_max_ext -> mul_mat; the
 *   OneSpeech Qwen3 page, "Front end and graph numerics": score and softmax
 *   intermediates stay in higher precision than the attended output.)
 *   A row with no visible key (n == 0) returns zeros.
 *
 *   GQA head mapping: query head h reads KV head h / (Hq / Hkv), contiguous
 *   grouping (qwenasr.cpp ARCHITECTURE.md, "GGUF layout": head_count 16,
 *   head_count_kv 8, GQA 2:1; Glossary "GQA").
 *
 *   Decode: request b attends over positions [0, seq_lens[b]); position j
 *   lives in physical page page_table[b][j / page_size], slot j % page_size
 *   (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder": decode attends
 *   over [0, cur_len + 1); M* "Speech recognition: Whisper and Qwen3-ASR",
 *   "Graph" and "Serving notes": decode runs on paged KV, requests hold pages).
 *   Pool layout [num_pages][page_size][Hkv][D].
 *
 *   Prefill: packed requests, request r owns rows [cu[r], cu[r+1]); row i of
 *   a request attends over rows j <= i of the same request, using K/V from
 *   the packed input (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder":
 *   prefill rewinds the cache, writes the prompt span and attends over
 *   [0, n_past + T) with n_past = 0; causal).
 *
 *   Page write: row i of request r is copied bit for bit to page
 *   page_table[r][i / page_size], slot i % page_size ("write fresh K/V into
 *   the cache at [n_past, n_past + T)", same section).
 *
 *   Chunked prefill (same section: the fresh span sits at [n_past,
 *   n_past + T) and attends over [0, n_past + T)): request r already holds
 *   n_past[r] positions in its pages; its new row i (absolute position
 *   n_past + i) attends over the cached positions [0, n_past) read through
 *   the page table and the new rows j <= i from the packed input, and the
 *   new rows are written at positions n_past + i.  With n_past = 0 this is
 *   the prefill above.
 *
 *   Window: packed windows, window w owns rows [cu_w[w], cu_w[w+1]); every
 *   row attends over every row of its own window, no mask inside, no GQA
 *   (qwenasr.cpp ARCHITECTURE.md, "Windowed audio tower": block-diagonal
 *   mask over windows, plain bidirectional MHA scaled by 1/sqrt(head_dim);
 *   M* page, "Qwen3-ASR / Graph": one packed forward, one segment per window).
 *
 *   QK-norm and RoPE (qwenasr.cpp ARCHITECTURE.md, "Qwen3 Thinker decoder":
 *   per-head RMSNorm on q and k, RMS over head_dim then a [head_dim] gain,
 *   before a 1D NEOX RoPE with freq_base 1e6; "Attention and RoPE": rotate
 *   half).  For one head vector x at position pos:
 *       y[d] = x[d] / sqrt(mean_d x[d]^2 + eps) * gain[d]
 *       a_i  = pos * theta^(-2 i / D),  i in [0, D/2)
 *       z[i]       = y[i] cos a_i - y[i + D/2] sin a_i
 *       z[i + D/2] = y[i] sin a_i + y[i + D/2] cos a_i
 *
 *   Decode append: the new token of request b sits at cur_len =
 *   seq_lens[b] - 1 ("appends one position at cur_len and attends over
 *   [0, cur_len + 1)"); q and k are normalised and rotated at that position,
 *   rounded to bf16 at the operator boundary, and k with the untouched v go
 *   to slot cur_len % page_size of page page_table[b][cur_len / page_size].
 *
 *   Encoder layer (qwenasr.cpp ARCHITECTURE.md, "Windowed audio tower"): the
 *   pre-norm Whisper-style layer around the window attention -- LayerNorm,
 *   q/k/v projections with bias, window attention, output projection with
 *   bias and residual, LayerNorm, gelu MLP with biases and residual.  Written
 *   out at its section below.
 *
 * Threads: rows are independent; n_threads worker threads take contiguous
 * slices of the row list.  This is the only concession to speed.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The definition of attention for one query row (see the file header).
 * p_out, when not NULL, receives the n softmax probabilities. */
ORACLE_EXPORT void oracle_attend_row(const double *q, const double *K, const double *V,
                                     int n, int D, double scale, double *out, double *p_out)
{
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;

    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += q[d] * K[(size_t)j * D + d];
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (int j = 0; j < n; ++j) {
        double p = s[j] / z;
        if (p_out)
            p_out[j] = p;
        for (int d = 0; d < D; ++d)
            out[d] += p * V[(size_t)j * D + d];
    }
    free(s);
}

/* ------------------------------------------------------------------------- */
/* Row-parallel driver.                                                       */

typedef void (*row_fn)(const void *ctx, int row, double *out);

typedef struct {
    const void *ctx;
    row_fn fn;
    const int32_t *rows; /* NULL: row i is i */
    int first, last;     /* slice of the row list */
    int D;
    double *out;
} slice_t;

static void *run_slice(void *arg)
{
    slice_t *sl = (slice_t *)arg;
    for (int i = sl->first; i < sl->last; ++i) {
        int row = sl->rows ? sl->rows[i] : i;
        sl->fn(sl->ctx, row, sl->out + (size_t)i * sl->D);
    }
    return NULL;
}

static void run_rows(const void *ctx, row_fn fn, const int32_t *rows, int n_rows, int D,
                     double *out, int n_threads)
{
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > n_rows)
        n_threads = n_rows > 0 ? n_rows : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    slice_t *sl = (slice_t *)malloc(sizeof(slice_t) * (size_t)n_threads);
    for (int t = 0; t < n_threads; ++t) {
        sl[t].ctx = ctx;
        sl[t].fn = fn;
        sl[t].rows = rows;
        sl[t].first = (int)((long long)n_rows * t / n_threads);
        sl[t].last = (int)((long long)n_rows * (t + 1) / n_threads);
        sl[t].D = D;
        sl[t].out = out;
    }
    for (int t = 1; t < n_threads; ++t)
        pthread_create(&th[t], NULL, run_slice, &sl[t]);
    run_slice(&sl[0]);
    for (int t = 1; t < n_threads; ++t)
        pthread_join(th[t], NULL);
    free(sl);
    free(th);
}

/* ------------------------------------------------------------------------- */
/* Decode over a paged pool.                                                  */

typedef struct {
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *page_table, *seq_lens;
    int batch, Hq, Hkv, D, page_size, max_pages, num_pages;
    double scale;
} decode_ctx;

static void decode_row(const void *vctx, int row, double *out)
{
    const decode_ctx *c = (const decode_ctx *)vctx;
    int b = row / c->Hq, h = row % c->Hq;
    int g = h / (c->Hq / c->Hkv);
    int n = c->seq_lens[b];
    double *q = (double *)malloc(sizeof(double) * (size_t)c->D);
    double *K = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)(n > 0 ? n : 1));
    double *V = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)(n > 0 ? n : 1));
    for (int d = 0; d < c->D; ++d)
        q[d] = bf16_to_double(c->q[((size_t)b * c->Hq + h) * c->D + d]);
    for (int j = 0; j < n; ++j) {
        int page = c->page_table[(size_t)b * c->max_pages + j / c->page_size];
        int slot = j % c->page_size;
        size_t base = (((size_t)page * c->page_size + slot) * c->Hkv + g) * c->D;
        for (int d = 0; d < c->D; ++d) {
            K[(size_t)j * c->D + d] = bf16_to_double(c->k_pages[base + d]);
            V[(size_t)j * c->D + d] = bf16_to_double(c->v_pages[base + d]);
        }
    }
    oracle_attend_row(q, K, V, n, c->D, c->scale, out, NULL);
    free(V);
    free(K);
    free(q);
}

/* out[i] = attention of row rows[i] = b * Hq + h (all B*Hq rows when rows is
 * NULL).  Returns 0, or -1 on inconsistent arguments (nothing computed). */
ORACLE_EXPORT int oracle_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                                const int32_t *page_table, const int32_t *seq_lens, int batch,
                                int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                                double scale, const int32_t *rows, int n_rows, double *out,
                                int n_threads)
{
    if (batch < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0)
        return -1;
    for (int b = 0; b < batch; ++b) {
        int n = seq_lens[b];
        if (n < 0 || n > max_pages * page_size)
            return -1;
        for (int p = 0; p < (n + page_size - 1) / page_size; ++p) {
            int page = page_table[(size_t)b * max_pages + p];
            if (page < 0 || page >= num_pages)
                return -1;
        }
    }
    if (!rows)
        n_rows = batch * Hq;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= batch * Hq)
            return -1;
    decode_ctx c = {q, k_pages, v_pages, page_table, seq_lens, batch, Hq, Hkv, D,
                    page_size, max_pages, num_pages, scale};
    run_rows(&c, decode_row, rows, n_rows, D, out, n_threads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Causal prefill over packed requests.                                       */

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *cu;
    int batch, Hq, Hkv, D;
    double scale;
} prefill_ctx;

static void prefill_row(const void *vctx, int row, double *out)
{
    const prefill_ctx *c = (const prefill_ctx *)vctx;
    int t = row / c->Hq, h = row % c->Hq;
    int g = h / (c->Hq / c->Hkv);
    int r = 0;
    while (!(c->cu[r] <= t && t < c->cu[r + 1]))
        ++r;
    int first = c->cu[r];
    int n = t - first + 1; /* keys j <= i within the request */
    double *q = (double *)malloc(sizeof(double) * (size_t)c->D);
    double *K = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    double *V = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    for (int d = 0; d < c->D; ++d)
        q[d] = bf16_to_double(c->q[((size_t)t * c->Hq + h) * c->D + d]);
    for (int j = 0; j < n; ++j) {
        size_t base = ((size_t)(first + j) * c->Hkv + g) * c->D;
        for (int d = 0; d < c->D; ++d) {
            K[(size_t)j * c->D + d] = bf16_to_double(c->k[base + d]);
            V[(size_t)j * c->D + d] = bf16_to_double(c->v[base + d]);
        }
    }
    oracle_attend_row(q, K, V, n, c->D, c->scale, out, NULL);
    free(V);
    free(K);
    free(q);
}

/* out[i] = attention of row rows[i] = t * Hq + h over its request's keys
 * j <= t (all total_tokens*Hq rows when rows is NULL). */
ORACLE_EXPORT int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const int32_t *cu_seqlens, int batch, int total_tokens,
                                 int Hq, int Hkv, int D, double scale, const int32_t *rows,
                                 int n_rows, double *out, int n_threads)
{
    if (batch <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0)
        return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[batch] != total_tokens)
        return -1;
    for (int r = 0; r < batch; ++r)
        if (cu_seqlens[r + 1] < cu_seqlens[r])
            return -1;
    if (!rows)
        n_rows = total_tokens * Hq;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_tokens * Hq)
            return -1;
    prefill_ctx c = {q, k, v, cu_seqlens, batch, Hq, Hkv, D, scale};
    run_rows(&c, prefill_row, rows, n_rows, D, out, n_threads);
    return 0;
}

/* Bit copy of the packed K/V rows of every request into its pages.  Slots
 * that no row maps to are left as they were.  Returns -1 (and writes
 * nothing) if a needed page id is outside [0, num_pages). */
ORACLE_EXPORT int oracle_page_write(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                                    int batch, const int32_t *page_table, int max_pages,
                                    int page_size, int num_pages, int Hkv, int D,
                                    uint16_t *k_pages, uint16_t *v_pages)
{
    for (int r = 0; r < batch; ++r) {
        int n = cu_seqlens[r + 1] - cu_seqlens[r];
        if (n < 0 || n > max_pages * page_size)
            return -1;
        for (int i = 0; i < n; ++i) {
            int page = page_table[(size_t)r * max_pages + i / page_size];
            if (page < 0 || page >= num_pages)
                return -1;
        }
    }
    size_t row_elems = (size_t)Hkv * D;
    for (int r = 0; r < batch; ++r) {
        int n = cu_seqlens[r + 1] - cu_seqlens[r];
        for (int i = 0; i < n; ++i) {
            int page = page_table[(size_t)r * max_pages + i / page_size];
            size_t dst = ((size_t)page * page_size + i % page_size) * row_elems;
            size_t src = (size_t)(cu_seqlens[r] + i) * row_elems;
            memcpy(k_pages + dst, k + src, row_elems * sizeof(uint16_t));
            memcpy(v_pages + dst, v + src, row_elems * sizeof(uint16_t));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Chunked prefill: new rows after n_past cached positions.                   */

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *cu, *n_past;
    const uint16_t *k_pages, *v_pages;
    const int32_t *page_table;
    int batch, Hq, Hkv, D, max_pages, page_size;
    double scale;
} chunk_ctx;

static void chunk_row(const void *vctx, int row, double *out)
{
    const chunk_ctx *c = (const chunk_ctx *)vctx;
    int t = row / c->Hq, h = row % c->Hq;
    int g = h / (c->Hq / c->Hkv);
    int r = 0;
    while (!(c->cu[r] <= t && t < c->cu[r + 1]))
        ++r;
    int first = c->cu[r];
    int i = t - first;          /* local index of the new row */
    int past = c->n_past[r];    /* cached positions before it */
    int n = past + i + 1;       /* keys: every cached position and new rows j <= i */
    double *q = (double *)malloc(sizeof(double) * (size_t)c->D);
    double *K = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    double *V = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    for (int d = 0; d < c->D; ++d)
        q[d] = bf16_to_double(c->q[((size_t)t * c->Hq + h) * c->D + d]);
    for (int j = 0; j < n; ++j) {
        const uint16_t *ks, *vs;
        if (j < past) { /* cached: through the page table */
            int page = c->page_table[(size_t)r * c->max_pages + j / c->page_size];
            size_t base = (((size_t)page * c->page_size + j % c->page_size) * c->Hkv + g) * c->D;
            ks = c->k_pages + base;
            vs = c->v_pages + base;
        } else { /* new: the packed rows */
            size_t base = ((size_t)(first + (j - past)) * c->Hkv + g) * c->D;
            ks = c->k + base;
            vs = c->v + base;
        }
        for (int d = 0; d < c->D; ++d) {
            K[(size_t)j * c->D + d] = bf16_to_double(ks[d]);
            V[(size_t)j * c->D + d] = bf16_to_double(vs[d]);
        }
    }
    oracle_attend_row(q, K, V, n, c->D, c->scale, out, NULL);
    free(V);
    free(K);
    free(q);
}

/* Checks of a chunked request list: n_past >= 0, cached and new positions
 * within the page-table row, every page id they use in [0, num_pages). */
static int chunk_args_ok(const int32_t *cu, const int32_t *n_past, int batch, const int32_t *page_table,
                         int max_pages, int page_size, int num_pages)
{
    for (int r = 0; r < batch; ++r) {
        int n = cu[r + 1] - cu[r];
        if (n < 0 || n_past[r] < 0 || (long long)n_past[r] + n > (long long)max_pages * page_size)
            return 0;
        for (int p = 0; p < (n_past[r] + n + page_size - 1) / page_size; ++p) {
            int page = page_table[(size_t)r * max_pages + p];
            if (page < 0 || page >= num_pages)
                return 0;
        }
    }
    return 1;
}

/* out[i] = attention of row rows[i] = t * Hq + h of the chunked prefill
 * (all total_tokens*Hq rows when rows is NULL); the pools hold the cached
 * positions [0, n_past) of every request. */
ORACLE_EXPORT int oracle_prefill_chunk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                       const int32_t *cu_seqlens, const int32_t *n_past, int batch,
                                       int total_tokens, int Hq, int Hkv, int D, const uint16_t *k_pages,
                                       const uint16_t *v_pages, const int32_t *page_table, int max_pages,
                                       int page_size, int num_pages, double scale, const int32_t *rows,
                                       int n_rows, double *out, int n_threads)
{
    if (batch <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0)
        return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[batch] != total_tokens)
        return -1;
    if (!chunk_args_ok(cu_seqlens, n_past, batch, page_table, max_pages, page_size, num_pages))
        return -1;
    if (!rows)
        n_rows = total_tokens * Hq;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_tokens * Hq)
            return -1;
    chunk_ctx c = {q, k, v, cu_seqlens, n_past, k_pages, v_pages, page_table, batch, Hq, Hkv, D,
                   max_pages, page_size, scale};
    run_rows(&c, chunk_row, rows, n_rows, D, out, n_threads);
    return 0;
}

/* Bit copy of the new rows of every request to positions n_past[r] + i of
 * its pages.  Slots that no row maps to are left as they were.  Returns -1
 * (and writes nothing) on inconsistent arguments. */
ORACLE_EXPORT int oracle_page_write_at(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens,
                                       const int32_t *n_past, int batch, const int32_t *page_table,
                                       int max_pages, int page_size, int num_pages, int Hkv, int D,
                                       uint16_t *k_pages, uint16_t *v_pages)
{
    if (!chunk_args_ok(cu_seqlens, n_past, batch, page_table, max_pages, page_size, num_pages))
        return -1;
    size_t row_elems = (size_t)Hkv * D;
    for (int r = 0; r < batch; ++r) {
        int n = cu_seqlens[r + 1] - cu_seqlens[r];
        for (int i = 0; i < n; ++i) {
            int pos = n_past[r] + i; /* the new row's position */
            int page = page_table[(size_t)r * max_pages + pos / page_size];
            size_t dst = ((size_t)page * page_size + pos % page_size) * row_elems;
            size_t src = (size_t)(cu_seqlens[r] + i) * row_elems;
            memcpy(k_pages + dst, k + src, row_elems * sizeof(uint16_t));
            memcpy(v_pages + dst, v + src, row_elems * sizeof(uint16_t));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Windowed bidirectional attention over packed windows.                      */

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *cu;
    int n_windows, H, D;
    double scale;
} window_ctx;

static void window_row(const void *vctx, int row, double *out)
{
    const window_ctx *c = (const window_ctx *)vctx;
    int t = row / c->H, h = row % c->H;
    int w = 0;
    while (!(c->cu[w] <= t && t < c->cu[w + 1]))
        ++w;
    int first = c->cu[w];
    int n = c->cu[w + 1] - first; /* every row of the window */
    double *q = (double *)malloc(sizeof(double) * (size_t)c->D);
    double *K = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    double *V = (double *)malloc(sizeof(double) * (size_t)c->D * (size_t)n);
    for (int d = 0; d < c->D; ++d)
        q[d] = bf16_to_double(c->q[((size_t)t * c->H + h) * c->D + d]);
    for (int j = 0; j < n; ++j) {
        size_t base = ((size_t)(first + j) * c->H + h) * c->D;
        for (int d = 0; d < c->D; ++d) {
            K[(size_t)j * c->D + d] = bf16_to_double(c->k[base + d]);
            V[(size_t)j * c->D + d] = bf16_to_double(c->v[base + d]);
        }
    }
    oracle_attend_row(q, K, V, n, c->D, c->scale, out, NULL);
    free(V);
    free(K);
    free(q);
}

/* out[i] = attention of row rows[i] = t * H + h over its own window (all
 * total_tokens*H rows when rows is NULL). */
ORACLE_EXPORT int oracle_window(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                const int32_t *cu_windows, int n_windows, int total_tokens, int H,
                                int D, double scale, const int32_t *rows, int n_rows, double *out,
                                int n_threads)
{
    if (n_windows <= 0 || H <= 0 || D <= 0)
        return -1;
    if (cu_windows[0] != 0 || cu_windows[n_windows] != total_tokens)
        return -1;
    for (int w = 0; w < n_windows; ++w)
        if (cu_windows[w + 1] < cu_windows[w])
            return -1;
    if (!rows)
        n_rows = total_tokens * H;
    for (int i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_tokens * H)
            return -1;
    window_ctx c = {q, k, v, cu_windows, n_windows, H, D, scale};
    run_rows(&c, window_row, rows, n_rows, D, out, n_threads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Per-head QK-norm, NEOX RoPE and the decode KV append.                      */

/* z[0..D) = RoPE_pos(RMSNorm(x) * gain) for one head vector (file header). */
static void norm_rope_vec(const uint16_t *x, int D, long pos, const float *gain, double eps,
                          double theta, double *z)
{
    double ms = 0.0;
    for (int d = 0; d < D; ++d) {
        double xd = bf16_to_double(x[d]);
        ms += xd * xd;
    }
    ms /= D;
    double r = 1.0 / sqrt(ms + eps);
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double y0 = bf16_to_double(x[i]) * r * (double)gain[i];
        double y1 = bf16_to_double(x[i + half]) * r * (double)gain[i + half];
        double a = (double)pos * pow(theta, -2.0 * i / D);
        double ca = cos(a), sa = sin(a);
        z[i] = y0 * ca - y1 * sa;
        z[i + half] = y0 * sa + y1 * ca;
    }
}

/* x [n_rows][H][D] bf16, row t at position pos[t]; out [n_rows][H][D]. */
ORACLE_EXPORT int oracle_qk_norm_rope(const uint16_t *x, int n_rows, int H, int D,
                                      const int32_t *pos, const float *gain, double eps,
                                      double theta, double *out)
{
    if (n_rows < 0 || H <= 0 || D <= 0 || D % 2)
        return -1;
    for (int t = 0; t < n_rows; ++t)
        for (int h = 0; h < H; ++h) {
            size_t o = ((size_t)t * H + h) * D;
            norm_rope_vec(x + o, D, pos[t], gain, eps, theta, out + o);
        }
    return 0;
}

/* bf16 at an operator boundary: the value as a binary32 (round to nearest),
 * then to bf16, round to nearest even (finite values). */
static uint16_t bf16_round(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* One new token per request (file header, "Decode append").  q [B][Hq][D],
 * k and v [B][Hkv][D] bf16; gains [D] float.  Writes q_rot [B][Hq][D] and
 * k_rot [B][Hkv][D] (double, before rounding), q_bf16 [B][Hq][D] (rounded),
 * and the token's K (rounded) and V rows into the pools.  Returns -1 and
 * writes nothing on a length outside [1, max_pages * page_size] or a page id
 * outside [0, num_pages). */
ORACLE_EXPORT int oracle_decode_append(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                       const float *q_gain, const float *k_gain, double eps,
                                       double theta, const int32_t *page_table,
                                       const int32_t *seq_lens, int batch, int Hq, int Hkv, int D,
                                       int page_size, int max_pages, int num_pages, double *q_rot,
                                       double *k_rot, uint16_t *q_bf16, uint16_t *k_pages,
                                       uint16_t *v_pages)
{
    if (batch < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D % 2 || page_size <= 0)
        return -1;
    for (int b = 0; b < batch; ++b) {
        int n = seq_lens[b];
        if (n < 1 || n > max_pages * page_size)
            return -1;
        int page = page_table[(size_t)b * max_pages + (n - 1) / page_size];
        if (page < 0 || page >= num_pages)
            return -1;
    }
    for (int b = 0; b < batch; ++b) {
        int cur = seq_lens[b] - 1; /* the new token's position */
        for (int h = 0; h < Hq; ++h) {
            size_t o = ((size_t)b * Hq + h) * D;
            norm_rope_vec(q + o, D, cur, q_gain, eps, theta, q_rot + o);
            for (int d = 0; d < D; ++d)
                q_bf16[o + d] = bf16_round(q_rot[o + d]);
        }
        int page = page_table[(size_t)b * max_pages + cur / page_size];
        int slot = cur % page_size;
        for (int g = 0; g < Hkv; ++g) {
            size_t o = ((size_t)b * Hkv + g) * D;
            size_t dst = (((size_t)page * page_size + slot) * Hkv + g) * D;
            norm_rope_vec(k + o, D, cur, k_gain, eps, theta, k_rot + o);
            for (int d = 0; d < D; ++d) {
                k_pages[dst + d] = bf16_round(k_rot[o + d]);
                v_pages[dst + d] = v[o + d];
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* AuT encoder layer around the window attention.                             */
/*
 * qwenasr.cpp ARCHITECTURE.md, "Windowed audio tower": the encoder is a
 * pre-norm Whisper-style transformer (d_model 896, 14 heads of head_dim 64,
 * FFN 3584 with gelu on the 0.6B), LayerNorm with bias, bias on q / k / v /
 * output, plain bidirectional attention under the block-diagonal window mask;
 * "GGUF layout": per layer attn_norm (weight, bias), attn_q / attn_k /
 * attn_v / attn_output (weight, bias), ffn_norm (weight, bias), ffn_up /
 * ffn_down (weight, bias); "Tensor shape and layout": a Linear weight is
 * PyTorch (out, in), y = x W^T + b.  One layer, for token row t:
 *
 *   a   = LN1(x)                       LN(v) = (v - mean) / sqrt(var + eps) * g + b,
 *                                      mean and biased variance over the row
 *   q|k|v = a Wqkv^T + bqkv            Wqkv = [Wq; Wk; Wv] stacked (3 d x d)
 *   o   = window attention of q, k, v  heads: columns [h Dh, (h + 1) Dh)
 *   h   = x + (o Wo^T + bo)
 *   f   = gelu(LN2(h) W1^T + b1)       gelu(u) = u / 2 (1 + erf(u / sqrt 2)),
 *                                      the exact form ("GGML conventions",
 *                                      "Conv2d stem": ggml_gelu_erf)
 *   y   = h + (f W2^T + b2)
 *
 * Precision: each of those lines is one operator; its result is rounded to
 * bf16 (through binary32, bf16_round) before the next line reads it -- the
 * bf16-at-operator-boundaries policy of the OneSpeech page ("Front end and
 * graph numerics") applied to this layer.  Inside a line everything is
 * double.  The layer's last line is returned unrounded (double).
 */

typedef struct {
    const uint16_t *x, *g, *b;
    int d;
    double eps;
} ln_ctx;

static void ln_row(const void *vctx, int t, double *out)
{
    const ln_ctx *c = (const ln_ctx *)vctx;
    const uint16_t *xr = c->x + (size_t)t * c->d;
    double mean = 0.0;
    for (int i = 0; i < c->d; ++i)
        mean += bf16_to_double(xr[i]);
    mean /= c->d;
    double var = 0.0;
    for (int i = 0; i < c->d; ++i) {
        double u = bf16_to_double(xr[i]) - mean;
        var += u * u;
    }
    var /= c->d;
    double inv = 1.0 / sqrt(var + c->eps);
    for (int i = 0; i < c->d; ++i)
        out[i] = (bf16_to_double(xr[i]) - mean) * inv * bf16_to_double(c->g[i]) + bf16_to_double(c->b[i]);
}

/* y [T][d] = LayerNorm over each row of x [T][d] with gain g and bias b
 * (bf16 [d]). */
ORACLE_EXPORT int oracle_layer_norm(const uint16_t *x, int T, int d, const uint16_t *g, const uint16_t *b,
                                    double eps, double *y, int n_threads)
{
    if (T < 0 || d <= 0 || !(eps >= 0.0))
        return -1;
    ln_ctx c = {x, g, b, d, eps};
    if (T > 0)
        run_rows(&c, ln_row, NULL, T, d, y, n_threads);
    return 0;
}

static double gelu_erf(double u)
{
    return 0.5 * u * (1.0 + erf(u / sqrt(2.0)));
}

typedef struct {
    const uint16_t *x, *w, *bias, *res;
    int K, N, act;
} linear_ctx;

static void linear_row(const void *vctx, int t, double *out)
{
    const linear_ctx *c = (const linear_ctx *)vctx;
    double *xr = (double *)malloc(sizeof(double) * (size_t)c->K);
    for (int k = 0; k < c->K; ++k)
        xr[k] = bf16_to_double(c->x[(size_t)t * c->K + k]);
    for (int n = 0; n < c->N; ++n) {
        const uint16_t *wr = c->w + (size_t)n * c->K;
        double acc = 0.0;
        for (int k = 0; k < c->K; ++k)
            acc += xr[k] * bf16_to_double(wr[k]);
        if (c->bias)
            acc += bf16_to_double(c->bias[n]);
        if (c->act == 1)
            acc = gelu_erf(acc);
        if (c->res)
            acc += bf16_to_double(c->res[(size_t)t * c->N + n]);
        out[n] = acc;
    }
    free(xr);
}

/* y [T][N] = act(x W^T + bias) + res: x [T][K], w [N][K] (PyTorch Linear
 * layout), bias [N] or NULL, act 0 (none) or 1 (exact gelu), res [T][N] or
 * NULL; all bf16. */
ORACLE_EXPORT int oracle_linear(const uint16_t *x, int T, int K, const uint16_t *w, int N, const uint16_t *bias,
                                int act, const uint16_t *res, double *y, int n_threads)
{
    if (T < 0 || K <= 0 || N <= 0 || (act != 0 && act != 1))
        return -1;
    linear_ctx c = {x, w, bias, res, K, N, act};
    if (T > 0)
        run_rows(&c, linear_row, NULL, T, N, y, n_threads);
    return 0;
}

/* double [n] -> bf16 [n] at an operator boundary */
static void round_all(const double *v, size_t n, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = bf16_round(v[i]);
}

/* One AuT encoder layer (see above) over T packed tokens x [T][d] cut into
 * windows cu_windows [n_windows + 1]; H heads of d / H dims, FFN width
 * d_ffn.  Weights bf16 in PyTorch Linear layout: w_qkv [3 d][d] (q, k, v
 * stacked), w_o [d][d], w_fc1 [d_ffn][d], w_fc2 [d][d_ffn]; biases and
 * LayerNorm gains / biases bf16 vectors.  blocks = 1 stops after the
 * attention block (y = the unrounded h), 2 runs the whole layer.  y [T][d]. */
ORACLE_EXPORT int oracle_encoder_layer(const uint16_t *x, const int32_t *cu_windows, int n_windows, int T, int d,
                                       int H, int d_ffn, const uint16_t *ln1_g, const uint16_t *ln1_b,
                                       const uint16_t *w_qkv, const uint16_t *b_qkv, const uint16_t *w_o,
                                       const uint16_t *b_o, const uint16_t *ln2_g, const uint16_t *ln2_b,
                                       const uint16_t *w_fc1, const uint16_t *b_fc1, const uint16_t *w_fc2,
                                       const uint16_t *b_fc2, double eps, int blocks, double *y, int n_threads)
{
    if (T <= 0 || d <= 0 || H <= 0 || d % H || d_ffn <= 0 || (blocks != 1 && blocks != 2))
        return -1;
    if (n_windows <= 0 || cu_windows[0] != 0 || cu_windows[n_windows] != T)
        return -1;
    for (int w = 0; w < n_windows; ++w)
        if (cu_windows[w + 1] < cu_windows[w])
            return -1;
    const int Dh = d / H;
    const size_t Td = (size_t)T * d;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)T * (size_t)(d_ffn > 3 * d ? d_ffn : 3 * d));
    uint16_t *a = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *qkv = (uint16_t *)malloc(sizeof(uint16_t) * Td * 3);
    uint16_t *q = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *k = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *v = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *o = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * Td);
    uint16_t *f = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * d_ffn);

    /* a = LN1(x) */
    oracle_layer_norm(x, T, d, ln1_g, ln1_b, eps, tmp, n_threads);
    round_all(tmp, Td, a);
    /* q | k | v = a Wqkv^T + bqkv, split into q, k, v [T][H][Dh] */
    oracle_linear(a, T, d, w_qkv, 3 * d, b_qkv, 0, NULL, tmp, n_threads);
    round_all(tmp, Td * 3, qkv);
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) {
            q[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + i];
            k[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + d + i];
            v[(size_t)t * d + i] = qkv[(size_t)t * 3 * d + 2 * d + i];
        }
    /* o = window attention, scale 1 / sqrt(Dh) */
    oracle_window(q, k, v, cu_windows, n_windows, T, H, Dh, 1.0 / sqrt((double)Dh), NULL, 0, tmp, n_threads);
    round_all(tmp, Td, o);
    /* h = x + (o Wo^T + bo) */
    oracle_linear(o, T, d, w_o, d, b_o, 0, x, tmp, n_threads);
    if (blocks == 1) {
        memcpy(y, tmp, sizeof(double) * Td);
    } else {
        round_all(tmp, Td, h);
        /* f = gelu(LN2(h) W1^T + b1) */
        oracle_layer_norm(h, T, d, ln2_g, ln2_b, eps, tmp, n_threads);
        round_all(tmp, Td, a);
        oracle_linear(a, T, d, w_fc1, d_ffn, b_fc1, 1, NULL, tmp, n_threads);
        round_all(tmp, (size_t)T * d_ffn, f);
        /* y = h + (f W2^T + b2) */
        oracle_linear(f, T, d_ffn, w_fc2, d, b_fc2, 0, h, y, n_threads);
    }
    free(f);
    free(h);
    free(o);
    free(v);
    free(k);
    free(q);
    free(qkv);
    free(a);
    free(tmp);
    return 0;
}
