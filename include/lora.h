/*
 * lora.h -- C ABI of the GB300 (sm_103a) heterogeneous multi-LoRA delta library.
 *
 * The operation (Punica in "BEE-30060 Multi-LoRA serving", Background; S-LoRA page,
 * Batching, formula 2): for a batch of n rows (tokens) where row i uses adapter
 * k = ids[i],
 *
 *     y_i  <-  y_i + s_k * (x_i . A_k) . B_k        (rows with ids[i] == -1 untouched)
 *
 * with x_i a row vector of d_in, A_k a d_in x r_k matrix, B_k an r_k x d_out matrix
 * and s_k the adapter's scale.  Rows are grouped into segments by adapter id
 * (Punica: requests grouped by adapter identity) and released rows (id -1) take no
 * part in the launch (LoRazor page: active-row-aware kernels).  The merge mode
 * switch applies W <- W +/- s_k A_k B_k in place (VaLoRA blog, section 4.4.1).
 *
 * Adapter storage (S-LoRA page, Unified Paging: a rank-R weight takes R pages of one
 * hidden-size vector): column j of A_k is the contiguous vector
 *     a_pool + a_pages[k * max_rank + j] * a_page_width      (d_in elements used)
 * and row j of B_k is
 *     b_pool + b_pages[k * max_rank + j] * b_page_width      (d_out elements used).
 * a_pool and b_pool may be the same unified pool.  Unpaged (contiguous) storage is
 * the special case a_pages[k][j] = offset_k + j.
 *
 * Conventions for every call:
 *  - Return value: LORA_OK (0) or a negative LORA_E_* code.  Arguments are checked
 *    on the host before anything is launched; on error nothing is launched and no
 *    caller memory is written.
 *  - Element type: bf16 (bit pattern in 16 bits) for x, y, W and the pools; fp32
 *    for v and scales; int32 for ids and page ids.  Matrices are row-major with a
 *    row stride given in elements (ld*).
 *  - Pointers named *_host (and lora_page_in's host_a / host_b) are host memory;
 *    every other data pointer is device memory of the context's device, owned by
 *    the caller (the library never frees it).  Device pointers and row strides
 *    must be 16-byte aligned (ld* and widths multiples of 8 elements).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on that stream; ids are read on the host during the call and
 *    need not outlive it (lora_fused_device_ids excepted: its ids stay on the
 *    device and must stay valid until the stream has passed the call).  A context
 *    is not thread-safe, and its scratch (partial V, dense adapter rows, the
 *    device-side plan) is shared by its calls: calls of one context that could
 *    overlap on the GPU (different streams) must be ordered by events; page-in
 *    uses no scratch.
 *  - Ranks must be multiples of 8 in [8, LORA_MAX_RANK].
 */
#ifndef LORA_H
#define LORA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_MAX_RANK 128

enum {
    LORA_OK = 0,
    LORA_E_INVAL = -1,        /* null / misaligned pointer, bad size or stride      */
    LORA_E_RANK = -2,         /* rank not a multiple of 8, or outside [8, max_rank] */
    LORA_E_ADAPTER = -3,      /* adapter id >= n_adapters, or < -1                  */
    LORA_E_NOT_RESIDENT = -4, /* a referenced adapter has a page id of -1           */
    LORA_E_PAGE = -5,         /* a page id >= the pool's page count                 */
    LORA_E_CUDA = -6,         /* CUDA runtime error; see lora_last_cuda_error()     */
    LORA_E_TIMEOUT = -7,      /* a bounded device-side wait expired                 */
    LORA_E_NOMEM = -8,        /* host or device allocation inside the library failed*/
    LORA_E_CAPACITY = -9,     /* n exceeds the context's max_rows                   */
    LORA_E_UNSUPPORTED = -10, /* shape beyond what the kernels handle, or not sm_103 */
    LORA_E_IO = -11,          /* tile-table or shape file could not be read/written */
    LORA_E_NOTUNED = -12      /* information only, never returned by a call that
                                 computes: lora_tile_status() reports it when the last
                                 call took a built-in default launch shape because the
                                 tile table had no entry for its shape             */
};

typedef struct lora_ctx lora_ctx;
typedef struct lora_table lora_table;

/* Host view of the last plan built by lora_plan_build (arrays owned by the context,
 * valid until the next call on it).  Bookkeeping of the grouping step:
 *   active_rows  ascending row indices i with ids[i] >= 0            [n_active]
 *   perm         active rows stably sorted by adapter id (ascending) [n_active]
 *   seg_offsets  segment s is perm[seg_offsets[s] .. seg_offsets[s+1])  [n_segments+1]
 *   seg_adapter  adapter id of segment s                              [n_segments]
 *   row_items    work items of the row-gather (decode) kernel, each at most
 *                rows_per_item consecutive entries of one segment of perm
 *   tile_items   tiles of at most 128 consecutive rows of one adapter for the
 *                tensor-core kernels: every maximal run of consecutive row indices
 *                inside a segment that is at least tile_min_run long (0: no tiles) */
typedef struct {
    int64_t n_active;
    const int32_t *active_rows;
    const int32_t *perm;
    int64_t n_segments;
    const int32_t *seg_offsets;
    const int32_t *seg_adapter;
    int64_t row_items;
    int64_t tile_items;
    int64_t rows_per_item;
    int64_t tile_min_run;
} lora_plan_view;

/* Create a context on `device` for batches of at most max_rows rows and adapters
 * of rank <= max_rank.  Allocates eight pinned staging buffers of 24 * max_rows
 * bytes (plus 8 KB) and their device copies (for the plans that do not travel in
 * the launch parameters), device plan buffers and a device status word, all owned
 * by the context, so that calls within max_rows allocate no staging memory.  device = -1 makes a
 * host-only context: plans, tables and tile files work, every launching call
 * returns LORA_E_UNSUPPORTED.  Fails with LORA_E_UNSUPPORTED on a device other
 * than compute capability 10.3. */
int lora_ctx_create(int device, int64_t max_rows, int max_rank, lora_ctx **out);
int lora_ctx_destroy(lora_ctx *ctx);

/* Register an adapter table.  The pools stay caller-owned device memory and must
 * outlive the table; rank_host, scale_host, a_pages_host and b_pages_host
 * ([n_adapters], [n_adapters], [n_adapters * max_rank] x2, page id -1 = not
 * resident) are copied.  Entries j >= rank[k] of the page arrays are ignored.
 * Per-adapter problems (bad rank, non-resident or out-of-range pages) are not
 * errors here: they are reported by the calls that reference that adapter. */
int lora_table_create(lora_ctx *ctx, const void *a_pool, int64_t a_n_pages,
                      int a_page_width, const void *b_pool, int64_t b_n_pages,
                      int b_page_width, int n_adapters, int max_rank,
                      const int32_t *rank_host, const float *scale_host,
                      const int32_t *a_pages_host, const int32_t *b_pages_host,
                      lora_table **out);
int lora_table_destroy(lora_table *table);

/* The tensor-core kernels read an adapter as consecutive rows.  For an adapter whose
 * pages are scattered in the pool (S-LoRA's unified paging), or whose rank is not a
 * multiple of 16, the table keeps a dense copy of its pages (full pages, rank padded
 * to 16 with zero rows, up to 1 GB per table; beyond that a call copies its adapters
 * into per-call scratch), made by the first tensor-core call that needs it and used
 * by every later one, so that a steady-state prefill call launches no copy.
 * lora_page_in marks its adapter's copy stale.  A caller that writes pool pages in
 * any other way must call this for the adapters it changed (adapter = -1: all)
 * before the next call on the table; the next tensor-core call then copies them
 * again.  Host-only; LORA_E_INVAL for a bad table or adapter. */
int lora_table_invalidate(lora_table *table, int adapter);

/* Host-only: build the plan for ids_host[n] and expose it (for inspection). */
int lora_plan_build(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
                    int64_t n, lora_plan_view *out);

/* Shrink: v[i, j] = sum_{c < d_in} x[i, c] * A_k[c, j] for j < r_k (fp32 out).
 * x [n, ldx] bf16, v [n, ldv] fp32 (ldv >= max rank referenced).  Columns j >= r_k
 * and rows with id -1 are not written. */
int lora_shrink(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
                int64_t n, const void *x, int64_t ldx, int d_in, float *v,
                int64_t ldv, void *stream);

/* Expand: y[i, o] = bf16(y[i, o] + s_k * sum_{j < r_k} v[i, j] * B_k[j, o]).
 * v [n, ldv] fp32, y [n, ldy] bf16 updated in place; rows with id -1 untouched. */
int lora_expand(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
                int64_t n, const float *v, int64_t ldv, void *y, int64_t ldy,
                int d_out, void *stream);

/* Fused: y_i <- y_i + s_k (x_i A_k) B_k, one bf16 rounding per output element.
 * x_i . A_k never leaves the chip in the row-gather kernel; the tensor-core tile
 * kernels accumulate it in fp32 tensor memory and hand it to the expand as a pair
 * of bf16 operands (hi + lo, about 16 significant bits) through a context-owned
 * scratch that stays in L2.  Rows with id -1 untouched. */
int lora_fused(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
               int64_t n, const void *x, int64_t ldx, int d_in, void *y, int64_t ldy,
               int d_out, void *stream);

/* Base projection with the adapter term fused into it (S-LoRA article, Batching: the
 * batched base model x W plus the separately computed x A B, "formula 2"; VaLoRA
 * blog, C2: the overhead of unmerged inference):
 *     y_i = bf16( x_i . W + s_k (x_i . A_k) . B_k ),   k = ids[i] >= 0
 *     y_i = bf16( x_i . W )                           ids[i] == -1 (released rows keep
 *                                                     the backbone, LoRazor article)
 * one bf16 rounding per output element.  x [n, ldx] bf16, W [d_in, ldw] bf16 (the
 * base weight, row-major d_in x d_out, as for lora_merge), y [n, ldy] bf16 written
 * (never read: every row of y is overwritten, released rows included).  The
 * shrink kernels first write v = x_i A_k (fp32) into context scratch; then one
 * tensor-core GEMM over 256 x 256 tiles (each computed by a pair of CTAs on two
 * SMs) accumulates x W and, in the same accumulator, the adapter terms of the
 * tile's rows (s_k v as a pair of bf16 operands, hi + lo, about 16 significant
 * bits, times B_k).  Errors (nothing launched): as lora_fused, and LORA_E_INVAL
 * for W. */
int lora_base_fused(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
                    int64_t n, const void *x, int64_t ldx, int d_in, const void *W, int64_t ldw,
                    void *y, int64_t ldy, int d_out, void *stream);

/* Fused delta that allocates nothing.  Same operation, arguments and results as
 * lora_fused (within the same tolerance; the two may pick different summation
 * orders), for callers that must not allocate device or pinned memory while they
 * run: code paths that forbid cudaMalloc / cudaFree, or that run inside a
 * pre-sized memory budget, such as an allocator hook or a graph-building step that
 * must not grow the device footprint.  There is no counterpart of this entry point on the
 * pages.  The context and the table are created beforehand (those calls do
 * allocate); this call then only launches kernels.  Its tensor-core scratch is
 * fixed file-scope device arrays that every GPU loading the library holds until
 * the process exits: 4 MB of partial V (64 slots of 128 x 128 fp32) and 8 MB for
 * the dense adapter rows of a call whose tile adapters do not sit in consecutive
 * pages of a rank that is a multiple of 16 (slots x rank padded to 16 x (d_in +
 * d_out) bf16).  Limits (else LORA_E_CAPACITY, nothing launched): at most 64
 * tiles of up to 128 consecutive same-adapter rows, those 8 MB, at most 256
 * row-gather work items and 512 active rows outside those tiles, n <= the
 * context's max_rows.  The arrays sit in a module of their own, which the CUDA
 * runtime loads (committing their 12 MB) the first time it is touched on a device:
 * lora_ctx_create does that and looks their device addresses up, so this call
 * itself allocates nothing, also on its first use (a context created after a
 * cudaDeviceReset looks the addresses up again).  Every call shares the arrays:
 * calls that overlap on the GPU (different streams, or one stream and a capture
 * replay) race on them; calls in order on one stream do not.  Nothing in it needs clearing: every slot a
 * call reads is written by the same call first.  Profiling (lora_profile_begin) is
 * ignored for this call. */
int lora_fused_noalloc(lora_ctx *ctx, const lora_table *table, const int32_t *ids_host,
                       int64_t n, const void *x, int64_t ldx, int d_in, void *y, int64_t ldy,
                       int d_out, void *stream);

/* lora_fused with the adapter ids in device memory (ids_dev: int32 [n], 16-byte
 * alignment not needed, 4-byte alignment required; -1 = released row), for decode
 * batches whose ids are produced on the GPU.  LoRazor article: the operator's work
 * follows the rows still active -- here the active rows are found on the device:
 * by default each row-gather cluster takes one row and reads its adapter id
 * itself (after waiting for the kernel that wrote the ids); with
 * LORA_OPT_DEVICE_PLAN = 1 a one-CTA plan kernel first counts the rows per adapter,
 * lays out work items (at most R rows of one adapter each) and the by-adapter
 * permutation in context scratch, which the row-gather kernel reads after waiting
 * for it.  Either way the grid has room for n items and the idle clusters leave at
 * once.
 * The call reads nothing on the host, copies nothing and allocates nothing, so it
 * can be captured in a CUDA graph (and replayed with new ids written in place).
 * Row-gather kernel only (no tensor-core tiles): meant for decode-sized batches.
 * Results are those of lora_fused on the same ids, element for element.  An id
 * outside [-1, n_adapters) or an adapter the table cannot serve leaves its row
 * unchanged and makes the next lora_sync_status return LORA_E_ADAPTER (the host
 * never sees the ids, so the call itself cannot).  Errors before any launch:
 * LORA_E_INVAL (arguments, n > max_rows), LORA_E_UNSUPPORTED (more than 16384
 * adapters in the table), LORA_E_ADAPTER (the table can serve no adapter). */
int lora_fused_device_ids(lora_ctx *ctx, const lora_table *table, const int32_t *ids_dev,
                          int64_t n, const void *x, int64_t ldx, int d_in, void *y,
                          int64_t ldy, int d_out, void *stream);

/* The arguments of lora_fused / lora_fused_device_ids in one block, for callers that
 * issue the same call shape many times (a decode loop): a binding fills the block
 * once per ids buffer and passes one pointer, instead of marshalling eleven
 * arguments on every call.  ids is host memory for lora_fused_args_call and device
 * memory for lora_fused_device_ids_args_call.  The block is read during the call
 * only and is never kept; every field is checked as in the call it stands for. */
typedef struct lora_fused_args {
    lora_ctx *ctx;
    const lora_table *table;
    const int32_t *ids;
    int64_t n;
    const void *x;
    int64_t ldx;
    void *y;
    int64_t ldy;
    int d_in;
    int d_out;
    void *stream;
} lora_fused_args;

/* lora_fused(a->ctx, a->table, a->ids, a->n, a->x, a->ldx, a->d_in, a->y, a->ldy,
 * a->d_out, a->stream); LORA_E_INVAL for a null block. */
int lora_fused_args_call(const lora_fused_args *a);

/* lora_fused_device_ids with the same fields (ids in device memory); LORA_E_INVAL
 * for a null block. */
int lora_fused_device_ids_args_call(const lora_fused_args *a);

/* Merge / unmerge (mode switch): W[c, o] = bf16(W[c, o] +/- s_k sum_j A_k[c, j]
 * B_k[j, o]) in place, W [d_in, ldw] bf16 row-major.  Unmerge after merge restores
 * W to within two bf16 rounding steps (not bit-exactly). */
int lora_merge(lora_ctx *ctx, const lora_table *table, int adapter, void *W,
               int64_t ldw, int d_in, int d_out, void *stream);
int lora_unmerge(lora_ctx *ctx, const lora_table *table, int adapter, void *W,
                 int64_t ldw, int d_in, int d_out, void *stream);

/* Adapter page-in (S-LoRA: adapters kept in host memory are brought into the unified
 * pool when a batch needs them, overlapped with compute; VaLoRA, section 4.4.1: only
 * A and B move): copies adapter `adapter`'s A and B from host memory into its pages
 * of the table's pools, asynchronously on `stream`.
 *   host_a  rank[adapter] rows of d_in bf16, row j = page j of A_k (column j of A_k)
 *   host_b  rank[adapter] rows of d_out bf16, row j = page j of B_k (row j of B_k)
 * Both rows-by-width blocks are contiguous, 16-byte aligned and page-locked
 * (cudaHostAlloc, or cudaHostRegister'ed): one kernel reads them directly over the
 * CPU-GPU link and writes the pool pages, so they must stay valid and unchanged
 * until the stream has passed the call.  d_in <= the A page width, d_out <= the B
 * page width, both multiples of 8; the rest of each page is left as it is.  The
 * pools are written (they are the caller's device memory, registered with the
 * table): the copy starts after every earlier kernel of the stream; a delta or
 * merge call that reads the adapter on another stream must be ordered after it
 * (an event).  With LORA_OPT_EARLY_PAGES, the next delta or merge call on the same
 * stream takes no early page copies.  Errors (nothing launched): LORA_E_INVAL (a
 * bad argument, or a buffer that is not page-locked host memory), LORA_E_ADAPTER,
 * or the adapter's own problem (LORA_E_RANK, LORA_E_NOT_RESIDENT, LORA_E_PAGE). */
int lora_page_in(lora_ctx *ctx, const lora_table *table, int adapter, const void *host_a,
                 int d_in, const void *host_b, int d_out, void *stream);

/* Shape -> tile-configuration table (VaLoRA blog, section 4.3.2: an offline
 * search stores the best tiling per input shape in a hash table that the runtime
 * looks up).  Lines of the text file are
 *     kind m_bucket s_bucket d_in d_out rank  cfg0 cfg1 cfg2 cfg3
 * kind: 0 row-gather fused, 1 shrink, 2 expand, 3 tile fused, 4 merge.
 * m_bucket: active rows (merge: d_in) rounded up to a power of two; s_bucket:
 * for kind 0 the number of distinct adapters, rounded up likewise, else 0.  A
 * line with nine fields has no s_bucket (read as 0).  Unknown shapes use a
 * built-in default; a lookup never fails. */
int lora_tiles_load(lora_ctx *ctx, const char *path);
int lora_tiles_save(const lora_ctx *ctx, const char *path);
int64_t lora_tiles_count(const lora_ctx *ctx);

/* Whether the last delta, merge or unmerge call of the context found every launch
 * shape it needed in the tile table: LORA_OK, or LORA_E_NOTUNED when at least one
 * came from the built-in default (the call itself succeeded either way).  Read it
 * after the call; the next call overwrites it.  LORA_E_INVAL for a null context. */
int lora_tile_status(const lora_ctx *ctx);

/* Offline search over a file of shapes (VaLoRA blog, section 4.3.2: every candidate
 * tiling of each input shape is profiled offline and the best kept in the table the
 * runtime looks up).  One shape per line of the text file at shapes_path:
 *     kind n d_in d_out rank adapters [run [objective]]
 * kind: rows (row-gather fused call), tiles (tensor-core fused call), merge; n rows
 * (ignored for merge); `adapters` adapters of rank `rank`; run: rows per request,
 * the ids being (i / run) % adapters (0, the default: i % adapters); objective:
 * latency (default: lora_tune_shape's cold single-call median) or throughput (rows
 * only: back-to-back calls over rotating copies of the inputs larger than L2).
 * '#' starts a comment.  The whole file is checked before anything runs (LORA_E_IO
 * if it cannot be read, LORA_E_INVAL for a malformed line or a rank above the
 * context's max_rank).  Each shape then runs on device buffers the call allocates,
 * fills with synthetic values (uniform, the variances of the workloads) on
 * `stream`, and frees; the winners go into the context's table.  If out_path is not
 * NULL the table is written there (lora_tiles_save format) followed by one comment
 * line per shape with its best time.  A host-only context (device -1) parses the
 * file and returns LORA_E_UNSUPPORTED. */
int lora_tune(lora_ctx *ctx, const char *shapes_path, const char *out_path, void *stream);

/* Offline search for one shape (VaLoRA blog, section 4.3.2): times every
 * candidate of a pruned configuration space with CUDA events (two warm-up calls,
 * then the median of `iters` calls, each timed alone after a 256 MB write that
 * leaves L2 cold; the context allocates that buffer on its first search and frees
 * it with the context), keeps the fastest in the context's table under
 * the key the runtime looks up, and returns its time in *best_us.
 *   kind 0 (row-gather fused): cluster width x rows per item;
 *   kind 3 (tile fused):       minimum run length routed to the tensor-core tiles;
 *   kind 4 (merge):            tensor-core or CUDA-core kernel; `y` is W
 *                              [d_in, ldy], ids_host[0] names the adapter, x unused.
 * Kinds 1 and 2 return LORA_E_UNSUPPORTED.  The buffers are updated by every
 * timed call (y receives the delta 2 + iters times per candidate). */
int lora_tune_shape(lora_ctx *ctx, const lora_table *table, int kind,
                    const int32_t *ids_host, int64_t n, const void *x, int64_t ldx,
                    int d_in, void *y, int64_t ldy, int d_out, int iters,
                    float *best_us, void *stream);

/* Synchronize `stream`, then read and clear the device status word: LORA_OK or
 * LORA_E_TIMEOUT if a kernel's bounded wait expired since the last check. */
int lora_sync_status(lora_ctx *ctx, void *stream);

/* Context options:
 *   LORA_OPT_TILE_PATH     1 (default) route runs of >= tile_min_run consecutive
 *                          same-adapter rows to the tensor-core tile kernels; 0 keeps
 *                          every row on the row-gather kernel
 *   LORA_OPT_MERGE_KERNEL  0 (default) tensor-core merge where supported; 1 CUDA cores
 *   LORA_OPT_TILE_MIN_RUN  > 0 fixes the minimum run length; 0 uses the tile table
 *                          (default 128)
 *   LORA_OPT_EARLY_PAGES   0 (default) / 1.  The kernels are launched as programmatic
 *                          dependents of the kernel before them in the stream and
 *                          read nothing that kernel may write before it finishes.  With
 *                          1 the row-gather kernel copies the adapter pages (A and B
 *                          pools) before that wait, overlapping the previous kernel's
 *                          tail, and so does the tensor-core path's copy of scattered
 *                          adapters into dense rows (it writes the half of its
 *                          double-buffered scratch that the previous staged call does
 *                          not read, and still waits before it ends).  The caller then
 *                          guarantees that no kernel launched immediately before a
 *                          delta, merge or unmerge call in the same stream writes the
 *                          pools or page tables (this library's own kernels never do; a
 *                          copy or a host-side wait in between is enough).
 *                          For lora_fused_device_ids in its default mode the guarantee
 *                          covers the device ids as well: with 1 the kernel reads them
 *                          (and copies the pages they select) before the wait.
 *   LORA_OPT_EARLY_INPUT   0 (default) / 1.  With 1 a delta call reads x and the
 *                          adapters before waiting for the kernels before it in the
 *                          stream: the tensor-core shrink loads x and the A rows and
 *                          runs its MMAs, the row-gather kernel also computes its
 *                          cluster's v and (when each thread has one output vector)
 *                          its term s_k v B_k; only the reads of y and the writes of
 *                          y, v and the partial sums wait.  Consecutive row-gather
 *                          calls then overlap almost whole.  The caller guarantees
 *                          that x and the pools are written neither by the kernel
 *                          launched immediately before a delta call in the same stream
 *                          nor by an earlier call of this library on that stream since
 *                          the last kernel that is not this library's (a kernel that
 *                          writes y, such as the base projection, is fine; so is a
 *                          chain of delta calls on one x; a copy or a host-side wait
 *                          in between is enough; one call's y passed as the next
 *                          call's x is not).  Not applied to a call whose own dense
 *                          copy of scattered adapters runs just before its shrink, nor
 *                          after a page-in on the same stream.
 *   LORA_OPT_DEVICE_PLAN   lora_fused_device_ids: 0 (default) one row per row-gather
 *                          cluster, its adapter read from the device ids by the kernel
 *                          itself (one launch); 1 a plan kernel first groups the rows by
 *                          adapter into items of several rows (two launches, fewer
 *                          re-reads of a shared adapter).
 *   LORA_OPT_ROWS_B_OVER_A 0 (default) a fused row-gather launch copies each CTA's
 *                          slice of B into the shared memory its slice of A used, once
 *                          the shrink has read it, when the call runs with
 *                          LORA_OPT_EARLY_INPUT, or when the launch has more CTAs than
 *                          the GPU holds at once and the smaller footprint lets more
 *                          be resident; 1 does so in every fused row-gather launch; -1
 *                          in none.  The results are the same bits either way. */
enum { LORA_OPT_TILE_PATH = 1, LORA_OPT_MERGE_KERNEL = 2, LORA_OPT_TILE_MIN_RUN = 3,
       LORA_OPT_EARLY_PAGES = 4, LORA_OPT_DEVICE_PLAN = 5, LORA_OPT_EARLY_INPUT = 6,
       LORA_OPT_ROWS_B_OVER_A = 7 };
int lora_ctx_set_option(lora_ctx *ctx, int option, int value);

/* Per-launch timing: between lora_profile_begin and lora_profile_end every
 * `every`-th kernel launch of the context (every >= 1) is bracketed by CUDA events
 * on its stream.  _end synchronizes on those events and returns, per kernel
 * family (0 row-gather, 1 tensor-core tile shrink, 2 merge, 3 tensor-core streaming
 * expand, 4 base projection GEMM of lora_base_fused), the number of launches made
 * while profiling in launches[] and their device time in ms[] (arrays of 5): the mean of the bracketed launches times that
 * number.  A call that first copies adapter pages into dense rows (dense.cu)
 * counts the copy in the family of the kernel that reads it. */
int lora_profile_begin(lora_ctx *ctx, int every);
int lora_profile_end(lora_ctx *ctx, double *ms, int64_t *launches);

/* Failure-detection self-test: launches one thread that waits, for limit_us
 * microseconds (1 .. 1e6), on a barrier nothing arrives on -- the bounded wait every
 * kernel of this library uses -- so that the wait gives up, records a timeout in
 * the status word and returns.  The next lora_sync_status on the stream then
 * returns LORA_E_TIMEOUT (and clears the word); the context stays usable.  No
 * trap, no fault: the kernel ends normally. */
int lora_selftest_timeout(lora_ctx *ctx, int64_t limit_us, void *stream);

/* Kernels launched by this context since it was created. */
int64_t lora_launch_count(const lora_ctx *ctx);

/* Which kernel the last call launched: 0 none, 1 row-gather, 2 tensor-core tile,
 * 3 both (delta calls), 4 merge / unmerge, 8 page-in, 16 base projection GEMM (with
 * the bits of the shrink kernels lora_base_fused launched before it); and how many
 * kernels it launched. */
int lora_last_path(const lora_ctx *ctx, int *n_launches);

const char *lora_strerror(int code);
const char *lora_last_cuda_error(const lora_ctx *ctx);
int lora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_H */
