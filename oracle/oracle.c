/*
 * CPU oracle for the heterogeneous multi-LoRA delta.  TEST INFRASTRUCTURE ONLY:
 * it is imported by the tests, by the smoke check and by the CPU-baseline leg of
 * the benchmark, never by the library.  It shares no code, header or table with
 * the CUDA path.
 *
 * What it computes (plain definitions, written out):
 *
 *   delta   y_i <- y_i + s_k * (x_i . A_k) . B_k   for every row i with k = ids[i] >= 0
 *           (Punica, "BEE-30060 Multi-LoRA serving", Background: the per-request
 *           difference y_i += x_i * A_i * B_i; S-LoRA page, Batching: compute xAB
 *           separately from the batched base model, "formula 2").
 *   shrink  v_i = x_i . A_k            (first factor of the same product)
 *   expand  y_i <- y_i + s_k * v_i . B_k
 *   merge   W <- W +/- s_k * A_k . B_k (VaLoRA blog, section 4.4.1: Delta W is computed
 *           at run time from the stored A and B and added to / subtracted from the
 *           base weight in one go; S-LoRA page, Batching, "formula 1").
 *   base    y_i = x_i . W + s_k * (x_i . A_k) . B_k, and y_i = x_i . W for a released
 *           row (S-LoRA page, Batching: the batched base model xW plus the separately
 *           computed xAB, "formula 2"; VaLoRA blog, C2: unmerged inference computes
 *           x.W and the adapter term; LoRazor page: released rows keep the backbone).
 *           The oracle supplies the adapter term in double (oracle_delta) and the
 *           rounding (oracle_round_bf16); the product x.W is a library matmul in
 *           float64 on the Python side, and the two are added before the one rounding.
 *   plan    active rows, stable grouping of active rows by adapter id
 *           (Punica: requests grouped by adapter identity; LoRazor page: rows of
 *           released adapters take no part in the LoRA operator).
 *
 * Adapter storage follows S-LoRA's unified paging (S-LoRA page, Unified Paging: a
 * rank-R weight occupies R pages of one H-vector each): column j of A_k is the
 * vector a_pool[a_pages[k*max_rank+j] * a_page_width + c], c < d_in, and row j of
 * B_k is b_pool[b_pages[k*max_rank+j] * b_page_width + o], o < d_out.
 *
 * Precision: bf16 inputs are decoded exactly, every sum is taken in double in
 * ascending index order, and each output element is rounded once to bf16
 * (round-to-nearest-even).  The shrink output v is fp32 by the interface, so
 * oracle_shrink rounds the double sum to float; oracle_fused keeps v in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 <-> double --------------------------------------------------- */

static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Nearest bf16 to a double, ties to even, written from the format's definition:
 * 8 significant bits for normal numbers, a fixed quantum of 2^-133 below 2^-126,
 * overflow to infinity once the rounded magnitude reaches 2^128. */
static uint16_t double_to_bf16(double v)
{
    if (v != v)
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    (void)frexp(a, &e);                  /* a = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;                       /* exponent of one unit in the last place */
    if (q < -133)
        q = -133;
    double units = rint(ldexp(a, -q));   /* default rounding mode: nearest, ties even */
    double r = ldexp(units, q);
    if (r >= 0x1p128)
        return sign | 0x7F80;
    float f = (float)r;                  /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

uint16_t oracle_bf16_round(double v) { return double_to_bf16(v); }
double oracle_bf16_value(uint16_t h) { return bf16_to_double(h); }

/* ---- adapter table as seen by the oracle -------------------------------- */

typedef struct {
    const uint16_t *a_pool;
    int64_t a_page_width;
    const uint16_t *b_pool;
    int64_t b_page_width;
    const int32_t *rank;
    const float *scale;
    const int32_t *a_pages;
    const int32_t *b_pages;
    int max_rank;
} table_t;

static double A_at(const table_t *t, int k, int64_t c, int j)
{
    int64_t page = t->a_pages[(int64_t)k * t->max_rank + j];
    return bf16_to_double(t->a_pool[page * t->a_page_width + c]);
}

static double B_at(const table_t *t, int k, int j, int64_t o)
{
    int64_t page = t->b_pages[(int64_t)k * t->max_rank + j];
    return bf16_to_double(t->b_pool[page * t->b_page_width + o]);
}

/* ---- row-parallel driver (rows are independent; each row's arithmetic is the
 *      same whatever the thread count, so results do not depend on it) ------- */

typedef void (*row_fn)(void *ctx, int64_t row);
typedef struct {
    row_fn fn;
    void *ctx;
    int64_t begin, end;
} slice_t;

static void *run_slice(void *p)
{
    slice_t *s = (slice_t *)p;
    for (int64_t i = s->begin; i < s->end; ++i)
        s->fn(s->ctx, i);
    return NULL;
}

static void for_rows(int64_t n, int nthreads, row_fn fn, void *ctx)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads == 1 || n < 2) {
        for (int64_t i = 0; i < n; ++i)
            fn(ctx, i);
        return;
    }
    pthread_t tid[256];
    int live[256];
    slice_t sl[256];
    for (int t = 0; t < nthreads; ++t) {
        sl[t].fn = fn;
        sl[t].ctx = ctx;
        sl[t].begin = n * t / nthreads;
        sl[t].end = n * (t + 1) / nthreads;
        live[t] = pthread_create(&tid[t], NULL, run_slice, &sl[t]) == 0;
        if (!live[t])
            run_slice(&sl[t]);           /* could not start a thread: do it here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (live[t])
            pthread_join(tid[t], NULL);
}

/* ---- shrink: v[i, j] = sum_c x[i, c] * A_k[c, j] ------------------------ */

typedef struct {
    table_t t;
    const int32_t *ids;
    const uint16_t *x;
    int64_t ldx;
    int d_in;
    float *v;
    int64_t ldv;
} shrink_ctx;

static void shrink_row(void *p, int64_t i)
{
    shrink_ctx *c = (shrink_ctx *)p;
    int k = c->ids[i];
    if (k < 0)
        return;
    for (int j = 0; j < c->t.rank[k]; ++j) {
        double acc = 0.0;
        for (int64_t col = 0; col < c->d_in; ++col)
            acc += bf16_to_double(c->x[i * c->ldx + col]) * A_at(&c->t, k, col, j);
        c->v[i * c->ldv + j] = (float)acc;
    }
}

/* ---- expand: y[i, o] = bf16(y[i, o] + s_k * sum_j v[i, j] * B_k[j, o]) -- */

typedef struct {
    table_t t;
    const int32_t *ids;
    const float *v;
    int64_t ldv;
    uint16_t *y;
    int64_t ldy;
    int d_out;
} expand_ctx;

static void expand_row(void *p, int64_t i)
{
    expand_ctx *c = (expand_ctx *)p;
    int k = c->ids[i];
    if (k < 0)
        return;
    int r = c->t.rank[k];
    double s = (double)c->t.scale[k];
    for (int64_t o = 0; o < c->d_out; ++o) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j)
            acc += (double)c->v[i * c->ldv + j] * B_at(&c->t, k, j, o);
        uint16_t *yo = &c->y[i * c->ldy + o];
        *yo = double_to_bf16(bf16_to_double(*yo) + s * acc);
    }
}

/* ---- the adapter term of one row, unscaled, in double:
 *      term[o] = sum_j v_j * B_k[j, o],  v_j = sum_c x[c] * A_k[c, j]
 *      (both sums in ascending index order).  Returns 0, or -1 if out of memory. */

static int adapter_term(const table_t *t, int k, const uint16_t *x_row, int d_in, int d_out,
                        double *term)
{
    int r = t->rank[k];
    double *v = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    if (!v)
        return -1;
    for (int j = 0; j < r; ++j) {
        double acc = 0.0;
        for (int64_t col = 0; col < d_in; ++col)
            acc += bf16_to_double(x_row[col]) * A_at(t, k, col, j);
        v[j] = acc;
    }
    for (int64_t o = 0; o < d_out; ++o) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j)
            acc += v[j] * B_at(t, k, j, o);
        term[o] = acc;
    }
    free(v);
    return 0;
}

/* ---- fused: y[i, o] = bf16(y[i, o] + s_k * term[o]) -------------------- */

typedef struct {
    table_t t;
    const int32_t *ids;
    const uint16_t *x;
    int64_t ldx;
    int d_in;
    uint16_t *y;
    int64_t ldy;
    int d_out;
} fused_ctx;

static void fused_row(void *p, int64_t i)
{
    fused_ctx *c = (fused_ctx *)p;
    int k = c->ids[i];
    if (k < 0)
        return;
    const double s_fused = (double)c->t.scale[k];
    double *term = (double *)malloc(sizeof(double) * (size_t)(c->d_out > 0 ? c->d_out : 1));
    if (!term)
        return;
    if (adapter_term(&c->t, k, &c->x[i * c->ldx], c->d_in, c->d_out, term) == 0)
        for (int64_t o = 0; o < c->d_out; ++o) {
            uint16_t *yo = &c->y[i * c->ldy + o];
            *yo = double_to_bf16(bf16_to_double(*yo) + s_fused * term[o]);
        }
    free(term);
}

/* ---- delta in double: out[i, o] = s_k * term[o], 0 for a released row (the
 *      adapter term of the base projection, unrounded) -------------------- */

typedef struct {
    table_t t;
    const int32_t *ids;
    const uint16_t *x;
    int64_t ldx;
    int d_in;
    double *out;
    int64_t ldo;
    int d_out;
} delta_ctx;

static void delta_row(void *p, int64_t i)
{
    delta_ctx *c = (delta_ctx *)p;
    double *dst = &c->out[i * c->ldo];
    int k = c->ids[i];
    if (k < 0) {
        for (int64_t o = 0; o < c->d_out; ++o)
            dst[o] = 0.0;
        return;
    }
    const double s_delta = (double)c->t.scale[k];
    if (adapter_term(&c->t, k, &c->x[i * c->ldx], c->d_in, c->d_out, dst) == 0)
        for (int64_t o = 0; o < c->d_out; ++o)
            dst[o] *= s_delta;
}

/* ---- merge: W[c, o] = bf16(W[c, o] + sign * s_k * sum_j A_k[c, j] B_k[j, o]) */

typedef struct {
    table_t t;
    int k;
    double signed_scale;
    uint16_t *W;
    int64_t ldw;
    int d_out;
} merge_ctx;

static void merge_row(void *p, int64_t c_row)
{
    merge_ctx *c = (merge_ctx *)p;
    int r = c->t.rank[c->k];
    for (int64_t o = 0; o < c->d_out; ++o) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j)
            acc += A_at(&c->t, c->k, c_row, j) * B_at(&c->t, c->k, j, o);
        uint16_t *w = &c->W[c_row * c->ldw + o];
        *w = double_to_bf16(bf16_to_double(*w) + c->signed_scale * acc);
    }
}

/* ---- public entry points (host pointers only) --------------------------- */

#define TABLE_ARGS                                                              \
    const uint16_t *a_pool, int64_t a_page_width, const uint16_t *b_pool,       \
        int64_t b_page_width, const int32_t *rank, const float *scale,          \
        const int32_t *a_pages, const int32_t *b_pages, int max_rank

#define TABLE_INIT                                                              \
    { a_pool, a_page_width, b_pool, b_page_width, rank, scale, a_pages, b_pages, \
      max_rank }

void oracle_shrink(TABLE_ARGS, const int32_t *ids, int64_t n, const uint16_t *x,
                   int64_t ldx, int d_in, float *v, int64_t ldv, int nthreads)
{
    shrink_ctx c = {TABLE_INIT, ids, x, ldx, d_in, v, ldv};
    for_rows(n, nthreads, shrink_row, &c);
}

void oracle_expand(TABLE_ARGS, const int32_t *ids, int64_t n, const float *v,
                   int64_t ldv, uint16_t *y, int64_t ldy, int d_out, int nthreads)
{
    expand_ctx c = {TABLE_INIT, ids, v, ldv, y, ldy, d_out};
    for_rows(n, nthreads, expand_row, &c);
}

void oracle_fused(TABLE_ARGS, const int32_t *ids, int64_t n, const uint16_t *x,
                  int64_t ldx, int d_in, uint16_t *y, int64_t ldy, int d_out,
                  int nthreads)
{
    fused_ctx c = {TABLE_INIT, ids, x, ldx, d_in, y, ldy, d_out};
    for_rows(n, nthreads, fused_row, &c);
}

/* out [n, ldo] doubles: the adapter term s_k (x_i A_k) B_k of each row, unrounded. */
void oracle_delta(TABLE_ARGS, const int32_t *ids, int64_t n, const uint16_t *x,
                  int64_t ldx, int d_in, double *out, int64_t ldo, int d_out, int nthreads)
{
    delta_ctx c = {TABLE_INIT, ids, x, ldx, d_in, out, ldo, d_out};
    for_rows(n, nthreads, delta_row, &c);
}

/* out[q] = nearest bf16 (ties to even) of v[q], q < count. */
void oracle_round_bf16(const double *v, uint16_t *out, int64_t count)
{
    for (int64_t q = 0; q < count; ++q)
        out[q] = double_to_bf16(v[q]);
}

/* sign = +1 merges the adapter into W, -1 takes it out again. */
void oracle_merge(TABLE_ARGS, int adapter, int sign, uint16_t *W, int64_t ldw,
                  int d_in, int d_out, int nthreads)
{
    merge_ctx c = {TABLE_INIT, adapter,
                   (sign < 0 ? -1.0 : 1.0) * (double)scale[adapter], W, ldw, d_out};
    for_rows(d_in, nthreads, merge_row, &c);
}

/* Plan: active rows in ascending order, then a stable counting sort of them by
 * adapter id (ascending); segments are the maximal runs of one id in that order.
 * Arrays are caller-sized: active_rows/perm [n], seg_offsets [n+1], seg_adapter [n].
 * Returns 0, or -1 when an id is >= n_adapters or below -1. */
int oracle_plan(const int32_t *ids, int64_t n, int n_adapters, int32_t *active_rows,
                int64_t *n_active, int32_t *perm, int32_t *seg_offsets,
                int32_t *seg_adapter, int64_t *n_seg)
{
    int64_t na = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < -1 || ids[i] >= n_adapters)
            return -1;
        if (ids[i] >= 0)
            active_rows[na++] = (int32_t)i;
    }
    *n_active = na;

    int64_t *count = (int64_t *)calloc((size_t)n_adapters + 1, sizeof(int64_t));
    int64_t *next = (int64_t *)calloc((size_t)n_adapters + 1, sizeof(int64_t));
    if (!count || !next) {
        free(count);
        free(next);
        return -1;
    }
    for (int64_t q = 0; q < na; ++q)
        count[ids[active_rows[q]]] += 1;
    int64_t run = 0, ns = 0;
    for (int k = 0; k < n_adapters; ++k) {
        next[k] = run;
        if (count[k] > 0) {
            seg_offsets[ns] = (int32_t)run;
            seg_adapter[ns] = k;
            ns += 1;
        }
        run += count[k];
    }
    seg_offsets[ns] = (int32_t)run;
    *n_seg = ns;
    for (int64_t q = 0; q < na; ++q) {
        int32_t row = active_rows[q];
        perm[next[ids[row]]++] = row;
    }
    free(count);
    free(next);
    return 0;
}
