// C ABI of the multi-LoRA delta library (declared in include/lora.h): argument
// checks, the host plan, staging of the plan to the device, kernel selection
// through the shape -> configuration table, and launches on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cctype>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include "../../include/lora.h"
#include "internal.h"
#include "status.h"
#include "plan.h"
#include "tiles.h"

namespace lora {
cudaError_t launch_merge_simt(const MergeParams &p, cudaStream_t stream);
cudaError_t launch_merge_tc(const MergeParams &p, int n_split, cudaStream_t stream);
bool merge_tc_supported(int d_in, int d_out, int rank);
}  // namespace lora

using namespace lora;

namespace {

constexpr int kSlots = 8;
constexpr int kSms = 152;
// Kernel families of the profiler: row-gather, tile shrink, merge, streaming
// expand, base projection.
constexpr int kFamilies = 5;

struct Slot {
    uint8_t *host = nullptr;   // pinned
    uint8_t *dev = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    bool pending = false;
};

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int round_up8(int64_t v) { return int((v + 7) / 8 * 8); }

}  // namespace

struct lora_ctx {
    int device = 0;
    int64_t max_rows = 0;
    int max_rank = 0;
    unsigned *d_status = nullptr;
    uint8_t *d_dplan = nullptr;     // device-side plan: items [max_rows], perm [max_rows], count
    Slot slots[kSlots];
    int next_slot = 0;
    Plan plan;
    TileTable tiles;
    char cuda_err[256] = {0};
    int last_path = 0;
    int last_launches = 0;
    bool untuned = false;           // the last call took a built-in default launch shape
    // Per-launch CUDA-event timing (lora_profile_begin / lora_profile_end).
    struct ProfEv {
        cudaEvent_t a = nullptr, b = nullptr;
        int family = 0;
    };
    bool prof = false;
    std::vector<ProfEv> prof_ev;
    size_t prof_used = 0;
    RowsParamsInline inline_args;   // staging of in-parameter plans
    RowsParamsInlineSmall inline_small;
    // Launches of recent row-gather-only fused calls whose plan travelled in the
    // parameters, by (table, shape, options, ids): a call repeating one of them (the
    // same ids for every layer of a decode step) patches x and y and launches.
    struct RowCacheEntry {
        bool valid = false;
        uint64_t table_sig = 0, tiles_gen = 0;
        std::vector<int32_t> adapters;   // the plan's adapters (checked against the table)
        int d_in = 0, d_out = 0;
        int64_t n = 0;
        std::vector<int32_t> ids;
        bool small = true;
        size_t smem = 0;
        RowsParamsInlineSmall small_args;
        std::unique_ptr<RowsParamsInline> big_args;
        bool untuned = false;
    };
    RowCacheEntry rcache[4];
    int rcache_next = 0;
    bool rows_last_small = true;    // what run_rows launched last (in-parameter plans)
    size_t rows_last_smem = 0;
    bool rows_last_inline = false;
    int64_t launches_total = 0;     // every kernel launched by this context
    int prof_every = 1;             // bracket one launch in this many, per kernel family
    int64_t prof_seen[kFamilies] = {0, 0, 0, 0, 0};
    int merge_path = 0;             // 0 auto (tensor cores when supported), 1 CUDA cores
    int tile_path = 1;              // 1: long same-adapter runs use the tensor-core tiles
    int tile_min_run_override = 0;  // > 0: fixed minimum run for the tile path
    int early_pages = 0;            // LORA_OPT_EARLY_PAGES
    int early_input = 0;            // LORA_OPT_EARLY_INPUT
    bool call_early_x = false;      // this call's shrink may load x before its wait
    int call_early = 0;             // early page copies for the call in progress
    int device_plan = 0;            // LORA_OPT_DEVICE_PLAN
    int b_over_a = 0;               // LORA_OPT_ROWS_B_OVER_A: 0 auto, 1 always, -1 never
    cudaStream_t pool_write_stream = nullptr;   // stream of the last page-in ...
    bool pool_write_pending = false;            // ... and no delta / merge launch after it yet
    int force_cluster = 0;          // > 0 while tuning: row-kernel cluster width
    int force_rows = 0;             // > 0 while tuning: rows per item
    float *vrows = nullptr;         // lora_base_fused: the shrink's fp32 rows
    size_t vrows_cap = 0;           //   (bytes)
    uint8_t *brows = nullptr;       // lora_base_fused: dense B rows, when needed
    size_t brows_cap = 0;
    uint16_t *aprep = nullptr;      // lora_base_fused: the prepared left operands
    size_t aprep_cap = 0;
    std::vector<int32_t> proj_mark, proj_off, proj_slots, proj_bbase;
    std::vector<ProjChunk> proj_chunks;
    uint8_t *vparts = nullptr;      // fused tile path: partial V between its two kernels
    size_t vparts_cap = 0;
    uint8_t *dense = nullptr;       // dense adapter rows of a call (dense.cu): two halves,
    size_t dense_cap = 0;           //   of dense_cap bytes each, used by turns
    int dense_turn = 0;
    std::vector<int32_t> slot_of;   // adapter -> slot while a call's slots are assigned
    std::unique_ptr<TileParams> tparams;   // launch parameters of the tile kernels
    uint8_t *flush = nullptr;       // lora_tune_shape: a buffer larger than L2, written
                                    // before each timed call so that it starts cold
};

struct lora_table {
    lora_ctx *ctx = nullptr;           // the context it was registered with (not owned)
    uint64_t serial = 0;               // unique per table created in this process
    uint64_t sig = 0;                  // hash of what a row-gather plan depends on: adapter
                                       // count, max rank, page widths, ranks, scales
    int device = -1;                   // device of the device copies (-1: host-only)
    const uint16_t *a_pool = nullptr;
    const uint16_t *b_pool = nullptr;
    int64_t a_n_pages = 0, b_n_pages = 0;
    int a_pw = 0, b_pw = 0;
    int n_adapters = 0, max_rank = 0;
    std::vector<int32_t> rank, a_pages, b_pages;
    std::vector<float> scale;
    std::vector<int8_t> status;        // per adapter: LORA_OK or the error a reference gets
    std::vector<uint8_t> a_contig, b_contig;   // per adapter: pages j < rank are p0 + j
    int32_t *d_rank = nullptr, *d_a_pages = nullptr, *d_b_pages = nullptr;
    float *d_scale = nullptr;
    uint8_t *d_ok = nullptr;           // per adapter: 1 when its status is LORA_OK
    int rank_max_ok = 0;               // largest rank among the adapters it can serve
    // Dense rows of the adapters whose pages the tensor-core kernels cannot read as
    // they are (scattered pages, or a rank not a multiple of 16): one slot of rp
    // rows per adapter, full pages (widths a_pw / b_pw), copied once and kept until
    // the adapter's pages change (lora_page_in, lora_table_invalidate).
    uint16_t *dense_a = nullptr, *dense_b = nullptr;
    int dense_cap = 0, dense_used = 0, dense_rp = 0;
    std::vector<int32_t> dense_slot;   // adapter -> slot, -1 none
    std::vector<uint8_t> dense_valid;  // adapter -> its slot holds its current pages
};

namespace {

int cuda_fail(lora_ctx *ctx, cudaError_t e)
{
    if (ctx)
        std::snprintf(ctx->cuda_err, sizeof ctx->cuda_err, "%s: %s", cudaGetErrorName(e),
                      cudaGetErrorString(e));
    return LORA_E_CUDA;
}

#define CUDA_TRY(ctx, expr)                          \
    do {                                             \
        cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess)                       \
            return cuda_fail((ctx), _e);             \
    } while (0)

int use_device(lora_ctx *ctx)
{
    if (ctx->device < 0)
        return LORA_E_UNSUPPORTED;   // host-only context
    (void)cudaGetLastError();        // drop a stale error left by an unrelated call
    int cur = -1;
    CUDA_TRY(ctx, cudaGetDevice(&cur));
    if (cur != ctx->device)
        CUDA_TRY(ctx, cudaSetDevice(ctx->device));
    return LORA_OK;
}

// Take the next staging slot with room for `bytes`; waits for the slot's previous
// upload/launches to finish before reusing its buffers.
// Early page copies for the call about to launch: the option, unless the kernel just
// before on this stream may be a page-in, which writes the pools.
void begin_call(lora_ctx *ctx, cudaStream_t stream)
{
    ctx->untuned = false;
    ctx->call_early = ctx->early_pages && !(ctx->pool_write_pending && ctx->pool_write_stream == stream);
    ctx->call_early_x = ctx->early_input && !(ctx->pool_write_pending && ctx->pool_write_stream == stream);
}

// A launch of a delta / merge call: after it, the stream's previous kernel is no
// longer a page-in.
void count_launch(lora_ctx *ctx, cudaStream_t stream)
{
    ctx->last_launches += 1;
    ctx->launches_total += 1;
    if (ctx->pool_write_pending && ctx->pool_write_stream == stream)
        ctx->pool_write_pending = false;
}

int acquire_slot(lora_ctx *ctx, size_t bytes, Slot **out)
{
    Slot &s = ctx->slots[ctx->next_slot];
    ctx->next_slot = (ctx->next_slot + 1) % kSlots;
    if (s.pending) {
        CUDA_TRY(ctx, cudaEventSynchronize(s.ev));
        s.pending = false;
    }
    if (bytes > s.cap) {
        size_t cap = std::max(bytes, s.cap * 2);
        cap = (cap + 255) & ~size_t(255);
        if (s.host)
            cudaFreeHost(s.host);
        if (s.dev)
            cudaFree(s.dev);
        s.host = nullptr;
        s.dev = nullptr;
        s.cap = 0;
        if (cudaMallocHost(reinterpret_cast<void **>(&s.host), cap) != cudaSuccess)
            return LORA_E_NOMEM;
        if (cudaMalloc(reinterpret_cast<void **>(&s.dev), cap) != cudaSuccess)
            return LORA_E_NOMEM;
        s.cap = cap;
    }
    *out = &s;
    return LORA_OK;
}

int release_slot(lora_ctx *ctx, Slot *s, cudaStream_t stream)
{
    CUDA_TRY(ctx, cudaEventRecord(s->ev, stream));
    s->pending = true;
    return LORA_OK;
}

// Bracket one kernel launch with events when profiling is on.  Returns the slot.
long prof_start(lora_ctx *ctx, int family, cudaStream_t stream)
{
    if (!ctx->prof)
        return -1;
    if ((ctx->prof_seen[family % kFamilies]++ % ctx->prof_every) != 0)
        return -1;
    if (ctx->prof_used == ctx->prof_ev.size()) {
        lora_ctx::ProfEv e;
        if (cudaEventCreate(&e.a) != cudaSuccess || cudaEventCreate(&e.b) != cudaSuccess)
            return -1;
        ctx->prof_ev.push_back(e);
    }
    lora_ctx::ProfEv &e = ctx->prof_ev[ctx->prof_used];
    e.family = family;
    if (cudaEventRecord(e.a, stream) != cudaSuccess)
        return -1;
    return long(ctx->prof_used++);
}

void prof_stop(lora_ctx *ctx, long slot, cudaStream_t stream)
{
    if (slot >= 0)
        cudaEventRecord(ctx->prof_ev[size_t(slot)].b, stream);
}

// Per-adapter status computed once when the table is registered.
int8_t adapter_status(const lora_table *t, int k)
{
    const int r = t->rank[size_t(k)];
    if (r < 8 || r > t->max_rank || r > LORA_MAX_RANK || (r % 8) != 0)
        return LORA_E_RANK;
    for (int j = 0; j < r; ++j) {
        const int32_t pa = t->a_pages[size_t(k) * t->max_rank + j];
        const int32_t pb = t->b_pages[size_t(k) * t->max_rank + j];
        if (pa == -1 || pb == -1)
            return LORA_E_NOT_RESIDENT;
        if (pa < -1 || pb < -1 || pa >= t->a_n_pages || pb >= t->b_n_pages)
            return LORA_E_PAGE;
    }
    return LORA_OK;
}

// Rows-kernel launch shape: cluster size C and rows per item R.
struct RowsCfg {
    int cluster;
    int rows;
};

size_t rows_smem_for(int mode, int cluster, int rows, int rank, int d_in, int d_out)
{
    const int si = std::max(8, round_up8(ceil_div(d_in, cluster)));
    const int so = std::max(8, round_up8(ceil_div(d_out, cluster)));
    return rows_smem_bytes(mode, si, so, rows, rank, cluster);
}

// Default launch shape when the tile table has no entry: items of at most 4 rows,
// then the smallest cluster that puts two CTAs' worth of work on every SM, grown
// further while one CTA would need more than half an SM's shared memory.
RowsCfg default_rows_cfg(int mode, int64_t n_act, int64_t n_seg, int d_in, int d_out, int rank)
{
    RowsCfg c{1, 1};
    const int64_t mean = n_seg > 0 ? ceil_div(n_act, n_seg) : 1;
    while (c.rows < 4 && c.rows < mean)
        c.rows <<= 1;
    const int64_t items = n_seg > 0 ? std::max<int64_t>(n_seg, ceil_div(n_act, c.rows)) : 0;
    const int dmin = std::min(d_in, d_out);
    const int cmax = rows_max_cluster();
    while (c.cluster < cmax && items * c.cluster < 2 * kSms && dmin / (2 * c.cluster) >= 128)
        c.cluster <<= 1;
    while (c.cluster < cmax &&
           rows_smem_for(mode, c.cluster, c.rows, rank, d_in, d_out) > size_t(110 * 1024))
        c.cluster <<= 1;
    return c;
}

// n_items: the launch's items (clusters).  A fused launch copies B's slices into A's
// space after the shrink (LORA_OPT_ROWS_B_OVER_A) by default when it reads x before
// its wait (consecutive calls overlap, and the A copies no longer share the memory
// system with B's: measured faster on every decode batch), and otherwise when it has
// more CTAs than the GPU holds at once and that layout lets more be resident (a lone
// call's chain is one B copy longer, which only pays when it saves a wave).
int rows_launch_params(const lora_ctx *ctx, int mode, RowsCfg cfg, int d_in, int d_out,
                       int rank_alloc, bool early_x, int64_t n_items, RowsParams &p,
                       size_t &smem)
{
    for (;; cfg.cluster <<= 1) {
        if (cfg.cluster > rows_max_cluster())
            return LORA_E_UNSUPPORTED;
        p.cluster = cfg.cluster;
        p.slice_in = std::max(8, round_up8(ceil_div(d_in, cfg.cluster)));
        p.slice_out = std::max(8, round_up8(ceil_div(d_out, cfg.cluster)));
        p.rows_alloc = cfg.rows;
        p.rank_alloc = rank_alloc;
        p.no_y_smem = rows_y_late(mode, early_x, p.slice_out, p.rows_alloc) ? 1 : 0;
        p.b_over_a = 0;
        smem = rows_smem_bytes(mode, p.slice_in, p.slice_out, p.rows_alloc, p.rank_alloc,
                               p.cluster, p.no_y_smem != 0);
        if (mode == kFused && ctx->b_over_a >= 0) {
            const size_t over = rows_smem_bytes(mode, p.slice_in, p.slice_out, p.rows_alloc,
                                                p.rank_alloc, p.cluster, p.no_y_smem != 0, true);
            const int64_t ctas = n_items * p.cluster;
            const int per_sm = rows_ctas_per_sm(mode, smem);
            if (ctx->b_over_a > 0 || early_x ||
                (ctas > int64_t(kSms) * per_sm && rows_ctas_per_sm(mode, over) > per_sm)) {
                p.b_over_a = 1;
                smem = over;
            }
        }
        if (smem <= size_t(rows_max_smem()))
            return LORA_OK;
    }
}

// Validate the pieces every delta call shares and build the plan.
int prepare(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n)
{
    if (!ctx || !t || t->ctx != ctx || n < 0 || (n > 0 && !ids))
        return LORA_E_INVAL;
    if (n > ctx->max_rows)
        return LORA_E_CAPACITY;
    int rc = plan_group(ctx->plan, ids, n, t->n_adapters);
    if (rc != LORA_OK)
        return rc;
    for (int32_t k : ctx->plan.seg_adapter) {
        const int8_t st = t->status[size_t(k)];
        if (st != LORA_OK)
            return st;
        if (t->rank[size_t(k)] > ctx->max_rank)
            return LORA_E_RANK;
    }
    return LORA_OK;
}

bool stride_ok(const void *p, int64_t ld, int d)
{
    return p && aligned16(p) && d > 0 && (d % 8) == 0 && ld >= d && (ld % 8) == 0;
}

// *hit: whether the shape came from the table (or a forced tuning candidate) rather
// than the built-in default.
RowsCfg choose_rows_cfg(const lora_ctx *ctx, int mode, int kind, int64_t n_act, int64_t n_seg,
                        int d_in, int d_out, int rank, bool *hit = nullptr)
{
    RowsCfg cfg = default_rows_cfg(mode, n_act, n_seg, d_in, d_out, rank);
    if (hit)
        *hit = true;
    if (ctx->force_cluster > 0 && ctx->force_rows > 0)
        return RowsCfg{ctx->force_cluster, ctx->force_rows};
    TileCfg tc;
    if (ctx->tiles.lookup(TileKey{kind, pow2_bucket(n_act), pow2_bucket(n_seg), d_in, d_out, rank}, tc) &&
        tc[0] >= 1 && tc[0] <= 16 && (tc[0] & (tc[0] - 1)) == 0 && tc[1] >= 1 && tc[1] <= 64) {
        cfg.cluster = tc[0];
        cfg.rows = tc[1];
    } else if (hit) {
        *hit = false;
    }
    return cfg;
}

// Stage items + perm and launch the row-gather kernel for the row items of the
// current plan (cut with cfg.rows rows per item).
int run_rows(lora_ctx *ctx, const lora_table *t, int mode, RowsCfg cfg, const void *x,
             int64_t ldx, int d_in, float *v, int64_t ldv, void *y, int64_t ldy, int d_out,
             cudaStream_t stream)
{
    Plan &pl = ctx->plan;
    if (pl.row_items.empty())
        return LORA_OK;
    cfg.rows = std::max(1, pl.row_max_rows);
    RowsParams p{};
    size_t smem = 0;
    int rc = rows_launch_params(ctx, mode, cfg, d_in, d_out, pl.row_max_rank, ctx->call_early_x,
                                int64_t(pl.row_items.size()), p, smem);
    if (rc != LORA_OK)
        return rc;

    const size_t items_bytes = pl.row_items.size() * sizeof(RowItem);
    const size_t perm_bytes = pl.row_perm.size() * sizeof(int32_t);
    const bool in_params = pl.row_items.size() <= size_t(kInlineItems) &&
                           pl.row_perm.size() <= size_t(kInlinePerm);
    Slot *slot = nullptr;
    if (!in_params) {
        rc = acquire_slot(ctx, items_bytes + perm_bytes + 16, &slot);
        if (rc != LORA_OK)
            return rc;
        std::memcpy(slot->host, pl.row_items.data(), items_bytes);
        std::memcpy(slot->host + items_bytes, pl.row_perm.data(), perm_bytes);
        CUDA_TRY(ctx, cudaMemcpyAsync(slot->dev, slot->host, items_bytes + perm_bytes,
                                      cudaMemcpyHostToDevice, stream));
    }

    p.x = static_cast<const uint16_t *>(x);
    p.ldx = ldx;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = ldy;
    p.v = v;
    p.ldv = ldv;
    p.a_pool = t->a_pool;
    p.a_pw = t->a_pw;
    p.b_pool = t->b_pool;
    p.b_pw = t->b_pw;
    p.a_pages = t->d_a_pages;
    p.b_pages = t->d_b_pages;
    p.rank = t->d_rank;
    p.scale = t->d_scale;
    p.items = in_params ? nullptr : reinterpret_cast<const RowItem *>(slot->dev);
    p.perm = in_params ? nullptr : reinterpret_cast<const int32_t *>(slot->dev + items_bytes);
    p.status = ctx->d_status;
    p.max_rank = t->max_rank;
    p.d_in = d_in;
    p.d_out = d_out;
    p.n_items = int(pl.row_items.size());
    p.early_pages = ctx->call_early;
    p.early_x = ctx->call_early_x;
    const long ev = prof_start(ctx, 0, stream);
    ctx->rows_last_inline = in_params;
    ctx->rows_last_smem = smem;
    ctx->rows_last_small = in_params && pl.row_items.size() <= 64 && pl.row_perm.size() <= 128;
    if (in_params && pl.row_items.size() <= 64 && pl.row_perm.size() <= 128) {
        RowsParamsInlineSmall &a = ctx->inline_small;
        a.p = p;
        std::memcpy(a.items, pl.row_items.data(), items_bytes);
        std::memcpy(a.perm, pl.row_perm.data(), perm_bytes);
        CUDA_TRY(ctx, launch_rows_inline_small(mode, a, smem, stream));
    } else if (in_params) {
        RowsParamsInline &a = ctx->inline_args;
        a.p = p;
        std::memcpy(a.items, pl.row_items.data(), items_bytes);
        std::memcpy(a.perm, pl.row_perm.data(), perm_bytes);
        CUDA_TRY(ctx, launch_rows_inline(mode, a, smem, stream));
    } else {
        CUDA_TRY(ctx, launch_rows(mode, p, smem, stream));
    }
    prof_stop(ctx, ev, stream);
    ctx->last_path |= 1;
    count_launch(ctx, stream);
    return slot ? release_slot(ctx, slot, stream) : LORA_OK;
}

// Minimum run of consecutive same-adapter rows that goes to the tensor-core tile
// kernels (shorter runs use the row-gather kernel); 0 disables the tile path.
int tile_min_run(const lora_ctx *ctx, int64_t n_act, int d_in, int d_out, int rank,
                 bool *hit = nullptr)
{
    if (hit)
        *hit = true;
    if (ctx->tile_min_run_override > 0)
        return ctx->tile_min_run_override;
    TileCfg tc;
    if (ctx->tiles.lookup(TileKey{kKindTileFused, pow2_bucket(n_act), 0, d_in, d_out, rank}, tc))
        return tc[0];
    if (hit)
        *hit = false;
    return 128;
}

// Row matrices of a tensor-core call over n_slots adapters (dense.cu): the pools
// when every adapter's pages are consecutive and its rank a multiple of 16 (no
// padding rows to zero), else a dense copy with one rp-row slot per adapter.
struct RowMats {
    const uint16_t *a = nullptr, *b = nullptr;
    int64_t a_ld = 0, a_nrows = 0, b_ld = 0, b_nrows = 0;
    bool staged = false;
    bool early = false;             // the copy may run before the previous kernel ends
    int rp = 0;
    // The copies to make: adapter stage_adapter[i] into slot stage_slot[i], widths and
    // row strides of the destination (the per-call scratch: the call's widths; the
    // table's cache: full pages).
    std::vector<int32_t> stage_adapter, stage_slot;
    int a_width = 0, b_width = 0;
    bool stage_a = false, stage_b = false;
};

// Bytes of the dense rows setup_rows would make for these adapters (0 when the
// pools serve as they are).
size_t dense_rows_bytes(const lora_table *t, const int32_t *adapters, int n_slots, int d_in,
                        int d_out, bool need_a, bool need_b)
{
    bool direct = true;
    int rmax = 0;
    for (int s = 0; s < n_slots; ++s) {
        const size_t k = size_t(adapters[s]);
        rmax = std::max(rmax, t->rank[k]);
        if ((t->rank[k] % 16) != 0 || (need_a && !t->a_contig[k]) || (need_b && !t->b_contig[k]))
            direct = false;
    }
    if (direct)
        return 0;
    const int rp = (rmax + 15) & ~15;
    const size_t a_bytes = need_a ? (size_t(n_slots) * rp * size_t(d_in) * 2u + 255u) & ~size_t(255) : 0;
    return a_bytes + (need_b ? size_t(n_slots) * rp * size_t(d_out) * 2u : 0);
}

// The table's cache of dense rows, for the adapters of a tensor-core call: make
// room (a grow copies the slots kept), give every adapter without a slot one, and
// list the copies of the adapters whose slot is not current.  Returns
// LORA_E_CAPACITY when the cache would pass kDenseCacheBytes (the call then stages
// into per-call scratch).
constexpr size_t kDenseCacheBytes = size_t(1) << 30;

int cache_rows(lora_ctx *ctx, lora_table *t, const int32_t *adapters, int n_slots,
               cudaStream_t stream, RowMats *m, int32_t *a_base, int32_t *b_base)
{
    if (t->dense_rp == 0)
        t->dense_rp = (t->max_rank + 15) & ~15;
    const int rp = t->dense_rp;
    const size_t slot_bytes = size_t(rp) * (size_t(t->a_pw) + size_t(t->b_pw)) * 2u;
    if (t->dense_slot.empty()) {
        t->dense_slot.assign(size_t(t->n_adapters), -1);
        t->dense_valid.assign(size_t(t->n_adapters), 0);
    }
    int need = t->dense_used;
    for (int s = 0; s < n_slots; ++s)
        if (t->dense_slot[size_t(adapters[s])] < 0)
            ++need;
    if (size_t(need) * slot_bytes > kDenseCacheBytes)
        return LORA_E_CAPACITY;
    if (need > t->dense_cap) {
        int cap = std::max(16, t->dense_cap);
        while (cap < need)
            cap *= 2;
        uint16_t *na = nullptr, *nb = nullptr;
        if (cudaMalloc(reinterpret_cast<void **>(&na), size_t(cap) * rp * t->a_pw * 2u) != cudaSuccess)
            return LORA_E_NOMEM;
        if (cudaMalloc(reinterpret_cast<void **>(&nb), size_t(cap) * rp * t->b_pw * 2u) != cudaSuccess) {
            cudaFree(na);
            return LORA_E_NOMEM;
        }
        if (t->dense_used > 0) {
            CUDA_TRY(ctx, cudaMemcpyAsync(na, t->dense_a, size_t(t->dense_used) * rp * t->a_pw * 2u,
                                          cudaMemcpyDeviceToDevice, stream));
            CUDA_TRY(ctx, cudaMemcpyAsync(nb, t->dense_b, size_t(t->dense_used) * rp * t->b_pw * 2u,
                                          cudaMemcpyDeviceToDevice, stream));
        }
        // the old buffers may still be read by launches queued before this call
        CUDA_TRY(ctx, cudaStreamSynchronize(stream));
        cudaFree(t->dense_a);
        cudaFree(t->dense_b);
        t->dense_a = na;
        t->dense_b = nb;
        t->dense_cap = cap;
    }
    m->stage_adapter.clear();
    m->stage_slot.clear();
    for (int s = 0; s < n_slots; ++s) {
        const size_t k = size_t(adapters[s]);
        if (t->dense_slot[k] < 0)
            t->dense_slot[k] = t->dense_used++;
        if (!t->dense_valid[k]) {
            m->stage_adapter.push_back(int32_t(k));
            m->stage_slot.push_back(t->dense_slot[k]);
            t->dense_valid[k] = 1;   // current once the copy queued below has run
        }
        a_base[s] = b_base[s] = t->dense_slot[k] * rp;
    }
    m->staged = !m->stage_adapter.empty();
    m->early = false;                // the copy waits for the kernel before it
    m->rp = rp;
    m->a = t->dense_a;
    m->a_ld = t->a_pw;
    m->a_nrows = int64_t(t->dense_cap) * rp;
    m->b = t->dense_b;
    m->b_ld = t->b_pw;
    m->b_nrows = int64_t(t->dense_cap) * rp;
    m->a_width = t->a_pw;
    m->b_width = t->b_pw;
    m->stage_a = m->stage_b = true;  // a slot holds both sides
    return LORA_OK;
}

// own: a caller-sized buffer for the dense rows (instead of the context's two halves
// or the fixed array), with room for dense_rows_bytes; its copy waits for the kernel
// before it (no early staging).
int setup_rows(lora_ctx *ctx, const lora_table *tc, const int32_t *adapters, int n_slots,
               int d_in, int d_out, bool need_a, bool need_b, const NoAllocScratch *fixed,
               cudaStream_t stream, RowMats *m, int32_t *a_base, int32_t *b_base,
               uint8_t *own = nullptr)
{
    // The table's dense-row cache is the table's own state, kept across calls.
    lora_table *t = const_cast<lora_table *>(tc);
    bool direct = true;
    int rmax = 0;
    for (int s = 0; s < n_slots; ++s) {
        const size_t k = size_t(adapters[s]);
        rmax = std::max(rmax, t->rank[k]);
        if ((t->rank[k] % 16) != 0 || (need_a && !t->a_contig[k]) || (need_b && !t->b_contig[k]))
            direct = false;
    }
    if (direct) {
        m->a = t->a_pool;
        m->a_ld = t->a_pw;
        m->a_nrows = t->a_n_pages;
        m->b = t->b_pool;
        m->b_ld = t->b_pw;
        m->b_nrows = t->b_n_pages;
        for (int s = 0; s < n_slots; ++s) {
            a_base[s] = t->a_pages[size_t(adapters[s]) * t->max_rank];
            b_base[s] = t->b_pages[size_t(adapters[s]) * t->max_rank];
        }
        return LORA_OK;
    }
    const int rp = (rmax + 15) & ~15;
    const size_t a_bytes = need_a ? (size_t(n_slots) * rp * size_t(d_in) * 2u + 255u) & ~size_t(255) : 0;
    const size_t bytes = a_bytes + (need_b ? size_t(n_slots) * rp * size_t(d_out) * 2u : 0);
    if (!fixed && !own) {
        int rc = cache_rows(ctx, t, adapters, n_slots, stream, m, a_base, b_base);
        if (rc != LORA_E_CAPACITY)
            return rc;   // served from the table's cache (or an error); else per call
    }
    m->stage_adapter.assign(adapters, adapters + n_slots);
    m->stage_slot.resize(size_t(n_slots));
    for (int s = 0; s < n_slots; ++s)
        m->stage_slot[size_t(s)] = s;
    m->a_width = d_in;
    m->b_width = d_out;
    m->stage_a = need_a;
    m->stage_b = need_b;
    uint8_t *buf = nullptr;
    if (own) {
        buf = own;
    } else if (fixed) {
        if (bytes > kNoAllocDenseBytes)
            return LORA_E_CAPACITY;
        buf = reinterpret_cast<uint8_t *>(fixed->dense);
    } else {
        if (bytes > ctx->dense_cap) {
            // Grows to the largest need seen; later calls reuse it.
            if (ctx->dense) {
                CUDA_TRY(ctx, cudaStreamSynchronize(stream));
                cudaFree(ctx->dense);
                ctx->dense = nullptr;
                ctx->dense_cap = 0;
            }
            if (cudaMalloc(reinterpret_cast<void **>(&ctx->dense), 2 * bytes) != cudaSuccess)
                return LORA_E_NOMEM;
            ctx->dense_cap = bytes;
        }
        // Consecutive staged calls use the two halves in turn, so a call's copy may
        // run while the previous call's kernels still read theirs (early staging).
        ctx->dense_turn ^= 1;
        buf = ctx->dense + size_t(ctx->dense_turn) * ctx->dense_cap;
        m->early = ctx->call_early != 0;
    }
    m->staged = true;
    m->rp = rp;
    m->a = reinterpret_cast<const uint16_t *>(buf);
    m->a_ld = d_in;
    m->a_nrows = int64_t(n_slots) * rp;
    m->b = reinterpret_cast<const uint16_t *>(buf + a_bytes);
    m->b_ld = d_out;
    m->b_nrows = int64_t(n_slots) * rp;
    for (int s = 0; s < n_slots; ++s)
        a_base[s] = b_base[s] = s * rp;
    return LORA_OK;
}

// The copies setup_rows asked for (a no-op for the pools themselves).
int run_staging(lora_ctx *ctx, const lora_table *t, const RowMats &m, cudaStream_t stream)
{
    if (!m.staged)
        return LORA_OK;
    const int n = int(m.stage_adapter.size());
    for (int s0 = 0; s0 < n; s0 += kStageSlots) {
        StageArgs sa{};
        sa.max_rank = t->max_rank;
        sa.rp = m.rp;
        sa.early = m.early ? 1 : 0;
        sa.n_slots = std::min(kStageSlots, n - s0);
        for (int s = 0; s < sa.n_slots; ++s) {
            sa.adapter[s] = m.stage_adapter[size_t(s0 + s)];
            sa.rank[s] = t->rank[size_t(sa.adapter[s])];
            sa.dst_slot[s] = m.stage_slot[size_t(s0 + s)];
        }
        if (m.stage_a)
            sa.side[0] = StageSide{t->a_pool, t->a_pw, t->d_a_pages, const_cast<uint16_t *>(m.a),
                                   m.a_width, m.a_ld};
        if (m.stage_b)
            sa.side[1] = StageSide{t->b_pool, t->b_pw, t->d_b_pages, const_cast<uint16_t *>(m.b),
                                   m.b_width, m.b_ld};
        CUDA_TRY(ctx, launch_stage_rows(sa, stream));
        count_launch(ctx, stream);
    }
    return LORA_OK;
}

int run_tiles(lora_ctx *ctx, const lora_table *t, int mode, const void *x, int64_t ldx, int d_in,
              float *v, int64_t ldv, void *y, int64_t ldy, int d_out, int64_t n,
              cudaStream_t stream, const NoAllocScratch *fixed = nullptr)
{
    Plan &pl = ctx->plan;
    if (pl.tile_items.empty())
        return LORA_OK;
    // The call's adapters (slots, in order of first tile) and their row matrices.
    const bool need_a = mode != kExpand, need_b = mode != kShrink;
    if (ctx->slot_of.size() < size_t(t->n_adapters))
        ctx->slot_of.resize(size_t(t->n_adapters), -1);
    std::vector<int32_t> &slots = pl.slot_adapter;
    slots.clear();
    for (const TileItem &it : pl.tile_items)
        if (ctx->slot_of[size_t(it.adapter)] < 0) {
            ctx->slot_of[size_t(it.adapter)] = int32_t(slots.size());
            slots.push_back(it.adapter);
        }
    const int n_slots = int(slots.size());
    pl.slot_a_base.resize(slots.size());
    pl.slot_b_base.resize(slots.size());
    RowMats mats;
    int rc = setup_rows(ctx, t, slots.data(), n_slots, d_in, d_out, need_a, need_b, fixed, stream,
                        &mats, pl.slot_a_base.data(), pl.slot_b_base.data());
    if (rc == LORA_OK)
        for (TileItem &it : pl.tile_items) {
            const int32_t sidx = ctx->slot_of[size_t(it.adapter)];
            it.a_row = pl.slot_a_base[size_t(sidx)];
            it.b_row = pl.slot_b_base[size_t(sidx)];
        }
    for (int32_t k : slots)
        ctx->slot_of[size_t(k)] = -1;
    if (rc != LORA_OK)
        return rc;
    const size_t items_bytes = pl.tile_items.size() * sizeof(TileItem);
    Slot *slot = nullptr;
    const TileItem *d_items = nullptr;
    const bool inl = pl.tile_items.size() <= size_t(kInlineTiles);
    if (fixed && !inl)
        return LORA_E_CAPACITY;
    if (!inl) {
        rc = acquire_slot(ctx, items_bytes + 16, &slot);
        if (rc != LORA_OK)
            return rc;
        std::memcpy(slot->host, pl.tile_items.data(), items_bytes);
        CUDA_TRY(ctx, cudaMemcpyAsync(slot->dev, slot->host, items_bytes, cudaMemcpyHostToDevice,
                                      stream));
        d_items = reinterpret_cast<const TileItem *>(slot->dev);
    }
    // K-split of the fused shrink: at most one CTA per SM over all tiles (each with
    // the deeper ring; fewer shares also leave the expand fewer partials to sum),
    // each CTA keeping at least 4 K blocks of 64.
    int ksplit = 1;
    if (mode == kFused) {
        const int64_t tiles = int64_t(pl.tile_items.size());
        const int nkb = (d_in + 63) / 64;
        while (ksplit < 8 && tiles * ksplit * 2 <= kSms && nkb / (ksplit * 2) >= 4 &&
               (!fixed || tiles * ksplit * 2 <= kNoAllocSlots))
            ksplit *= 2;
        const size_t need = size_t(tiles) * size_t(ksplit) * size_t(kVPartBytes);
        if (!fixed && need > ctx->vparts_cap) {
            // Grows to the largest need seen; later calls reuse it.
            if (ctx->vparts) {
                CUDA_TRY(ctx, cudaStreamSynchronize(stream));
                cudaFree(ctx->vparts);
                ctx->vparts = nullptr;
                ctx->vparts_cap = 0;
            }
            if (cudaMalloc(reinterpret_cast<void **>(&ctx->vparts), need) != cudaSuccess)
                return LORA_E_NOMEM;
            ctx->vparts_cap = need;
        }
    }
    // TileParams carries the inline list (8 KB): one per context, reused.
    if (!ctx->tparams) {
        ctx->tparams.reset(new (std::nothrow) TileParams());
        if (!ctx->tparams)
            return LORA_E_NOMEM;
    }
    TileParams &p = *ctx->tparams;
    p = TileParams{};
    if (inl) {
        p.items_inline = 1;
        std::copy(pl.tile_items.begin(), pl.tile_items.end(), p.inl);
    }
    p.x = static_cast<const uint16_t *>(x);
    p.ldx = ldx;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = ldy;
    p.a_rows = mats.a;
    p.a_ld = mats.a_ld;
    p.a_nrows = mats.a_nrows;
    p.b_rows = mats.b;
    p.b_ld = mats.b_ld;
    p.b_nrows = mats.b_nrows;
    p.items = d_items;
    p.vparts = fixed ? fixed->vparts : reinterpret_cast<float *>(ctx->vparts);
    p.ksplit = ksplit;
    p.v = v;
    p.ldv = ldv;
    p.status = ctx->d_status;
    p.max_rank = t->max_rank;
    p.n_rows = int(n);
    p.d_in = d_in;
    p.d_out = d_out;
    p.n_items = int(pl.tile_items.size());
    p.vmode = mode == kFused ? 0 : 1;
    p.max_tile_rank = pl.tile_max_rank;
    // x ahead of the wait when the caller allows it and no copy into the row matrix
    // runs just before; y ahead of the expand's wait when the shrink runs just before.
    p.early_x = (ctx->call_early_x && !mats.staged) ? 1 : 0;
    p.early_tiles = mode == kFused ? 1 : 0;
    // A grid that fits one CTA per SM gets the deeper ring.
    p.wide_ring = (int64_t(pl.tile_items.size()) * ksplit <= kSms) ? 1 : 0;
    // The dense copy (if any) is timed with the kernel that first reads it.
    if (mode != kExpand) {
        const long ev = prof_start(ctx, 1, stream);
        rc = run_staging(ctx, t, mats, stream);
        if (rc != LORA_OK)
            return rc;
        CUDA_TRY(ctx, launch_shrink_tc(p, stream));
        prof_stop(ctx, ev, stream);
        count_launch(ctx, stream);
    }
    if (mode != kShrink) {
        const long ev = prof_start(ctx, 3, stream);
        if (mode == kExpand) {
            rc = run_staging(ctx, t, mats, stream);
            if (rc != LORA_OK)
                return rc;
        }
        CUDA_TRY(ctx, launch_expand_tc(p, stream));
        prof_stop(ctx, ev, stream);
        count_launch(ctx, stream);
    }
    ctx->last_path |= 2;
    return slot ? release_slot(ctx, slot, stream) : LORA_OK;
}

// A repeat of a cached row-gather-only fused call: a table with the same signature
// (ranks, scales, widths: a decode step's layers each have their own pools), the
// same shape, options and ids (their contents).  Returns the entry or nullptr.
lora_ctx::RowCacheEntry *rcache_find(lora_ctx *ctx, const lora_table *t, const int32_t *ids,
                                     int64_t n, int d_in, int d_out)
{
    if (ctx->force_cluster > 0 || ctx->force_rows > 0)
        return nullptr;
    for (auto &e : ctx->rcache)
        if (e.valid && e.table_sig == t->sig && e.n == n && e.d_in == d_in &&
            e.d_out == d_out && e.tiles_gen == ctx->tiles.gen &&
            std::memcmp(e.ids.data(), ids, size_t(n) * sizeof(int32_t)) == 0) {
            // Same ranks and scales, possibly another table (another layer's pools):
            // every adapter of the plan must be one this table can serve.
            for (int32_t k : e.adapters)
                if (t->status[size_t(k)] != LORA_OK)
                    return nullptr;
            return &e;
        }
    return nullptr;
}

void rcache_clear(lora_ctx *ctx)
{
    for (auto &e : ctx->rcache)
        e.valid = false;
}

int delta_call(lora_ctx *ctx, const lora_table *t, int mode, const int32_t *ids, int64_t n,
               const void *x, int64_t ldx, int d_in, float *v, int64_t ldv, void *y,
               int64_t ldy, int d_out, cudaStream_t stream)
{
    if (ctx) {
        ctx->last_path = ctx->last_launches = 0;
        begin_call(ctx, stream);
    }
    if (mode == kFused && ctx && t && t->ctx == ctx && n > 0 && ids && ctx->device >= 0) {
        lora_ctx::RowCacheEntry *e = rcache_find(ctx, t, ids, n, d_in, d_out);
        // A launch laid out without y rows in shared memory needs early input.
        if (e && (e->small ? e->small_args.p.no_y_smem : e->big_args->p.no_y_smem) &&
            !ctx->call_early_x)
            e = nullptr;
        if (e) {
            if (!stride_ok(x, ldx, d_in) || !stride_ok(y, ldy, d_out))
                return LORA_E_INVAL;
            int rc = use_device(ctx);
            if (rc != LORA_OK)
                return rc;
            const long ev = prof_start(ctx, 0, stream);
            auto patch = [&](RowsParams &q) {
                q.x = static_cast<const uint16_t *>(x);
                q.ldx = ldx;
                q.y = static_cast<uint16_t *>(y);
                q.ldy = ldy;
                q.a_pool = t->a_pool;
                q.b_pool = t->b_pool;
                q.a_pages = t->d_a_pages;
                q.b_pages = t->d_b_pages;
                q.rank = t->d_rank;
                q.scale = t->d_scale;
                q.early_pages = ctx->call_early;
                q.early_x = ctx->call_early_x;
            };
            if (e->small) {
                patch(e->small_args.p);
                CUDA_TRY(ctx, launch_rows_inline_small(kFused, e->small_args, e->smem, stream));
            } else {
                patch(e->big_args->p);
                CUDA_TRY(ctx, launch_rows_inline(kFused, *e->big_args, e->smem, stream));
            }
            prof_stop(ctx, ev, stream);
            ctx->last_path = 1;
            ctx->untuned = e->untuned;
            count_launch(ctx, stream);
            return LORA_OK;
        }
    }
    int rc = prepare(ctx, t, ids, n);
    if (rc != LORA_OK)
        return rc;
    Plan &pl = ctx->plan;
    if (pl.active.empty())
        return LORA_OK;
    if (mode != kExpand) {
        if (!stride_ok(x, ldx, d_in) || d_in > t->a_pw)
            return LORA_E_INVAL;
    }
    if (mode != kShrink) {
        if (!stride_ok(y, ldy, d_out) || d_out > t->b_pw)
            return LORA_E_INVAL;
    }
    if (mode != kFused) {
        if (!v || (reinterpret_cast<uintptr_t>(v) & 3u) || ldv < 1)
            return LORA_E_INVAL;
        int32_t rmax = 0;
        for (int32_t k : pl.seg_adapter)
            rmax = std::max(rmax, t->rank[size_t(k)]);
        if (ldv < rmax)
            return LORA_E_INVAL;
    }
    rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    const int kind = mode == kShrink ? kKindShrink : mode == kExpand ? kKindExpand : kKindRowsFused;
    int32_t rmax = 0;
    for (int32_t k : pl.seg_adapter)
        rmax = std::max(rmax, t->rank[size_t(k)]);
    const int64_t n_act = int64_t(pl.active.size());
    bool hit_tiles = true, hit_rows = true;
    const int min_run = (ctx->tile_path && tile_tc_supported(d_in, d_out, rmax))
                            ? tile_min_run(ctx, n_act, d_in, d_out, rmax, &hit_tiles)
                            : 0;
    // Rows-kernel shape from the rows that stay on it (approximated by all rows when
    // the tile path is off).
    RowsCfg cfg = choose_rows_cfg(ctx, mode, kind, n_act, int64_t(pl.seg_adapter.size()), d_in,
                                  d_out, rmax, &hit_rows);
    plan_items(pl, t->rank.data(), t->scale.data(), cfg.rows, min_run);
    if (!pl.tile_items.empty() && pl.row_active > 0 && pl.row_active < n_act)
        cfg = choose_rows_cfg(ctx, mode, kind, pl.row_active, int64_t(pl.row_items.size()), d_in,
                              d_out, pl.row_max_rank, &hit_rows);
    // The minimum run is a tuned decision only where a run could reach a tile (the
    // search's shortest candidate is 32 rows).
    ctx->untuned = (!hit_tiles && pl.max_seg_len >= 32) || (!pl.row_items.empty() && !hit_rows);
    rc = run_tiles(ctx, t, mode, x, ldx, d_in, v, ldv, y, ldy, d_out, n, stream);
    if (rc != LORA_OK)
        return rc;
    rc = run_rows(ctx, t, mode, cfg, x, ldx, d_in, v, ldv, y, ldy, d_out, stream);
    // Keep the launch of a row-gather-only fused call whose plan travelled in the
    // parameters, for the calls that repeat it.
    if (rc == LORA_OK && mode == kFused && pl.tile_items.empty() && !pl.row_items.empty() &&
        ctx->rows_last_inline && ctx->force_cluster == 0 && ctx->force_rows == 0) {
        lora_ctx::RowCacheEntry &e = ctx->rcache[ctx->rcache_next];
        ctx->rcache_next = (ctx->rcache_next + 1) % int(sizeof ctx->rcache / sizeof ctx->rcache[0]);
        e.valid = false;
        e.table_sig = t->sig;
        e.adapters.assign(pl.seg_adapter.begin(), pl.seg_adapter.end());
        e.tiles_gen = ctx->tiles.gen;
        e.n = n;
        e.d_in = d_in;
        e.d_out = d_out;
        e.ids.assign(ids, ids + n);
        e.small = ctx->rows_last_small;
        e.smem = ctx->rows_last_smem;
        e.untuned = ctx->untuned;
        if (e.small) {
            e.small_args = ctx->inline_small;
            e.valid = true;
        } else {
            if (!e.big_args)
                e.big_args.reset(new (std::nothrow) RowsParamsInline());
            if (e.big_args) {
                *e.big_args = ctx->inline_args;
                e.valid = true;
            }
        }
    }
    return rc;
}

int merge_call(lora_ctx *ctx, const lora_table *t, int adapter, void *W, int64_t ldw,
               int d_in, int d_out, float sign, cudaStream_t stream)
{
    if (ctx) {
        ctx->last_path = ctx->last_launches = 0;
        begin_call(ctx, stream);
    }
    if (!ctx || !t || t->ctx != ctx)
        return LORA_E_INVAL;
    if (adapter < 0 || adapter >= t->n_adapters)
        return LORA_E_ADAPTER;
    if (t->status[size_t(adapter)] != LORA_OK)
        return t->status[size_t(adapter)];
    if (!stride_ok(W, ldw, d_out) || d_in <= 0 || d_in > t->a_pw || d_out > t->b_pw)
        return LORA_E_INVAL;
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    MergeParams p{};
    p.W = static_cast<uint16_t *>(W);
    p.ldw = ldw;
    p.a_pool = t->a_pool;
    p.a_pw = t->a_pw;
    p.b_pool = t->b_pool;
    p.b_pw = t->b_pw;
    p.b_n_pages = t->b_n_pages;
    p.a_pages = t->d_a_pages + size_t(adapter) * t->max_rank;
    p.b_pages = t->d_b_pages + size_t(adapter) * t->max_rank;
    p.status = ctx->d_status;
    p.d_in = d_in;
    p.d_out = d_out;
    p.rank = t->rank[size_t(adapter)];
    p.scale = sign * t->scale[size_t(adapter)];
    int path = ctx->merge_path;
    TileCfg tcfg;
    if (path == 0) {
        if (ctx->tiles.lookup(TileKey{kKindMerge, pow2_bucket(d_in), 0, d_in, d_out, p.rank}, tcfg))
            path = tcfg[0];
        else
            ctx->untuned = true;
    }
    const bool tc = merge_tc_supported(d_in, d_out, p.rank) && path != 1;
    RowMats mats;
    if (tc) {
        rc = setup_rows(ctx, t, &adapter, 1, d_in, d_out, true, true, nullptr, stream, &mats,
                        &p.a_row, &p.b_row);
        if (rc != LORA_OK)
            return rc;
        p.a_rows = mats.a;
        p.a_ld = mats.a_ld;
        p.a_nrows = mats.a_nrows;
        p.b_rows = mats.b;
        p.b_ld = mats.b_ld;
        p.b_nrows = mats.b_nrows;
    }
    const long ev = prof_start(ctx, 2, stream);
    if (tc) {
        rc = run_staging(ctx, t, mats, stream);
        if (rc != LORA_OK)
            return rc;
        CUDA_TRY(ctx, launch_merge_tc(p, 0, stream));
    } else {
        CUDA_TRY(ctx, launch_merge_simt(p, stream));
    }
    prof_stop(ctx, ev, stream);
    ctx->last_path = 4;
    count_launch(ctx, stream);
    return LORA_OK;
}

}  // namespace

extern "C" {

int lora_version(void) { return 1; }

const char *lora_strerror(int code)
{
    switch (code) {
    case LORA_OK: return "ok";
    case LORA_E_INVAL: return "invalid argument (null/misaligned pointer, size or stride)";
    case LORA_E_RANK: return "unsupported rank (multiple of 8 in [8, max_rank] required)";
    case LORA_E_ADAPTER: return "adapter id out of range";
    case LORA_E_NOT_RESIDENT: return "referenced adapter is not resident (page id -1)";
    case LORA_E_PAGE: return "page id beyond the pool";
    case LORA_E_CUDA: return "CUDA runtime error";
    case LORA_E_TIMEOUT: return "a bounded device-side wait expired";
    case LORA_E_NOMEM: return "allocation failed";
    case LORA_E_CAPACITY: return "batch beyond the context's max_rows or a fixed scratch limit";
    case LORA_E_UNSUPPORTED: return "shape not supported by the kernels";
    case LORA_E_IO: return "tile-table or shape file could not be read or written";
    case LORA_E_NOTUNED: return "information: a built-in default launch shape was used";
    default: return "unknown status";
    }
}

const char *lora_last_cuda_error(const lora_ctx *ctx) { return ctx ? ctx->cuda_err : ""; }

int lora_ctx_create(int device, int64_t max_rows, int max_rank, lora_ctx **out)
{
    if (!out || max_rows < 0 || max_rank < 8 || max_rank > LORA_MAX_RANK || (max_rank % 8) ||
        device < -1)
        return LORA_E_INVAL;
    *out = nullptr;
    if (device == -1) {
        // Host-only context: plans and tile tables, no device state, no launches.
        lora_ctx *h = new (std::nothrow) lora_ctx();
        if (!h)
            return LORA_E_NOMEM;
        h->device = -1;
        h->max_rows = max_rows;
        h->max_rank = max_rank;
        *out = h;
        return LORA_OK;
    }
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return LORA_E_CUDA;
    cudaDeviceProp prop{};
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
        return LORA_E_CUDA;
    if (prop.major != 10 || prop.minor != 3)
        return LORA_E_UNSUPPORTED;   // built for sm_103a only
    lora_ctx *ctx = new (std::nothrow) lora_ctx();
    if (!ctx)
        return LORA_E_NOMEM;
    ctx->device = device;
    ctx->max_rows = max_rows;
    ctx->max_rank = max_rank;
    // Plans up to max_rows never grow these again.
    Plan &pl = ctx->plan;
    pl.active.reserve(size_t(max_rows));
    pl.perm.reserve(size_t(max_rows));
    pl.seg_offsets.reserve(size_t(max_rows) + 1);
    pl.seg_adapter.reserve(size_t(max_rows));
    pl.row_items.reserve(size_t(max_rows));
    pl.row_perm.reserve(size_t(max_rows));
    pl.tile_items.reserve(size_t(max_rows) / 64 + 64);
    int prev = 0;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&ctx->d_status), 16) != cudaSuccess ||
        cudaMemset(ctx->d_status, 0, 16) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&ctx->d_dplan), size_t(max_rows) * 20 + 64) != cudaSuccess) {
        lora_ctx_destroy(ctx);
        cudaSetDevice(prev);
        return LORA_E_CUDA;
    }
    // Staging slots sized for any plan of up to max_rows rows (row items and the
    // permutation, tile lists, base-projection terms and ids: at most 24 bytes a row
    // and a little more), so that no call allocates in steady state.
    const size_t slot_bytes = (size_t(max_rows) * 24u + 8192u + 255u) & ~size_t(255);
    for (Slot &s : ctx->slots) {
        if (cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming) != cudaSuccess ||
            cudaMallocHost(reinterpret_cast<void **>(&s.host), slot_bytes) != cudaSuccess ||
            cudaMalloc(reinterpret_cast<void **>(&s.dev), slot_bytes) != cudaSuccess) {
            lora_ctx_destroy(ctx);
            cudaSetDevice(prev);
            return LORA_E_CUDA;
        }
        s.cap = slot_bytes;
    }
    // lora_fused_noalloc's fixed scratch: loading the module that holds it commits
    // its memory here, so that no lora_fused_noalloc call is the one that does.
    if (noalloc_scratch(device, true, nullptr) != cudaSuccess) {
        lora_ctx_destroy(ctx);
        cudaSetDevice(prev);
        return LORA_E_CUDA;
    }
    cudaSetDevice(prev);
    *out = ctx;
    return LORA_OK;
}

int lora_ctx_destroy(lora_ctx *ctx)
{
    if (!ctx)
        return LORA_E_INVAL;
    if (ctx->device < 0) {
        delete ctx;
        return LORA_OK;
    }
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    for (auto &e : ctx->prof_ev) {
        cudaEventDestroy(e.a);
        cudaEventDestroy(e.b);
    }
    for (Slot &s : ctx->slots) {
        if (s.ev) {
            if (s.pending)
                cudaEventSynchronize(s.ev);
            cudaEventDestroy(s.ev);
        }
        if (s.host)
            cudaFreeHost(s.host);
        if (s.dev)
            cudaFree(s.dev);
    }
    if (ctx->d_status)
        cudaFree(ctx->d_status);
    if (ctx->d_dplan)
        cudaFree(ctx->d_dplan);
    if (ctx->vparts)
        cudaFree(ctx->vparts);
    if (ctx->vrows)
        cudaFree(ctx->vrows);
    if (ctx->brows)
        cudaFree(ctx->brows);
    if (ctx->aprep)
        cudaFree(ctx->aprep);
    if (ctx->dense)
        cudaFree(ctx->dense);
    if (ctx->flush)
        cudaFree(ctx->flush);
    cudaSetDevice(prev);
    delete ctx;
    return LORA_OK;
}

int lora_table_create(lora_ctx *ctx, const void *a_pool, int64_t a_n_pages, int a_page_width,
                      const void *b_pool, int64_t b_n_pages, int b_page_width, int n_adapters,
                      int max_rank, const int32_t *rank_host, const float *scale_host,
                      const int32_t *a_pages_host, const int32_t *b_pages_host,
                      lora_table **out)
{
    if (!out)
        return LORA_E_INVAL;
    *out = nullptr;
    if (!ctx || !a_pool || !b_pool || !aligned16(a_pool) || !aligned16(b_pool) ||
        a_n_pages <= 0 || b_n_pages <= 0 || a_page_width <= 0 || b_page_width <= 0 ||
        (a_page_width % 8) || (b_page_width % 8) || n_adapters <= 0 || max_rank < 8 ||
        max_rank > LORA_MAX_RANK || !rank_host || !scale_host || !a_pages_host || !b_pages_host)
        return LORA_E_INVAL;
    static std::atomic<uint64_t> serials{0};
    lora_table *t = new (std::nothrow) lora_table();
    if (!t)
        return LORA_E_NOMEM;
    t->serial = ++serials;
    {
        // FNV-1a over the fields a row-gather plan and its launch shape depend on
        // (not the pools or page ids: a cached launch patches those)
        uint64_t h = 1469598103934665603ull;
        auto mix = [&h](const void *d, size_t nb) {
            const unsigned char *c = static_cast<const unsigned char *>(d);
            for (size_t i = 0; i < nb; ++i) {
                h ^= c[i];
                h *= 1099511628211ull;
            }
        };
        const int64_t head[4] = {n_adapters, max_rank, a_page_width, b_page_width};
        mix(head, sizeof head);
        mix(rank_host, size_t(n_adapters) * sizeof(int32_t));
        mix(scale_host, size_t(n_adapters) * sizeof(float));
        t->sig = h;
    }
    t->ctx = ctx;
    t->device = ctx->device;
    t->a_pool = static_cast<const uint16_t *>(a_pool);
    t->b_pool = static_cast<const uint16_t *>(b_pool);
    t->a_n_pages = a_n_pages;
    t->b_n_pages = b_n_pages;
    t->a_pw = a_page_width;
    t->b_pw = b_page_width;
    t->n_adapters = n_adapters;
    t->max_rank = max_rank;
    const size_t np = size_t(n_adapters) * size_t(max_rank);
    t->rank.assign(rank_host, rank_host + n_adapters);
    t->scale.assign(scale_host, scale_host + n_adapters);
    t->a_pages.assign(a_pages_host, a_pages_host + np);
    t->b_pages.assign(b_pages_host, b_pages_host + np);
    t->status.resize(size_t(n_adapters));
    plan_reserve(ctx->plan, n_adapters);
    t->a_contig.assign(size_t(n_adapters), 0);
    t->b_contig.assign(size_t(n_adapters), 0);
    for (int k = 0; k < n_adapters; ++k) {
        t->status[size_t(k)] = adapter_status(t, k);
        if (t->status[size_t(k)] != LORA_OK)
            continue;
        const int32_t *pa = &t->a_pages[size_t(k) * max_rank], *pb = &t->b_pages[size_t(k) * max_rank];
        bool ca = true, cb = true;
        for (int j = 1; j < t->rank[size_t(k)]; ++j) {
            ca = ca && pa[j] == pa[0] + j;
            cb = cb && pb[j] == pb[0] + j;
        }
        t->a_contig[size_t(k)] = ca;
        t->b_contig[size_t(k)] = cb;
    }
    // Device copies; pages of adapters that cannot be used are zeroed so that no
    // kernel could ever form an address from them.
    if (ctx->device < 0) {
        *out = t;   // host-only: bookkeeping without device copies
        return LORA_OK;
    }
    std::vector<int32_t> ap(t->a_pages), bp(t->b_pages);
    std::vector<uint8_t> okv(size_t(n_adapters), 0);
    for (int k = 0; k < n_adapters; ++k) {
        if (t->status[size_t(k)] != LORA_OK) {
            for (int j = 0; j < max_rank; ++j)
                ap[size_t(k) * max_rank + j] = bp[size_t(k) * max_rank + j] = 0;
        } else {
            okv[size_t(k)] = 1;
            t->rank_max_ok = std::max(t->rank_max_ok, t->rank[size_t(k)]);
        }
    }
    int prev = 0;
    cudaGetDevice(&prev);
    bool okk = cudaSetDevice(ctx->device) == cudaSuccess &&
               cudaMalloc(reinterpret_cast<void **>(&t->d_rank), sizeof(int32_t) * n_adapters) == cudaSuccess &&
               cudaMalloc(reinterpret_cast<void **>(&t->d_scale), sizeof(float) * n_adapters) == cudaSuccess &&
               cudaMalloc(reinterpret_cast<void **>(&t->d_a_pages), sizeof(int32_t) * np) == cudaSuccess &&
               cudaMalloc(reinterpret_cast<void **>(&t->d_b_pages), sizeof(int32_t) * np) == cudaSuccess &&
               cudaMemcpy(t->d_rank, rank_host, sizeof(int32_t) * n_adapters, cudaMemcpyHostToDevice) == cudaSuccess &&
               cudaMemcpy(t->d_scale, scale_host, sizeof(float) * n_adapters, cudaMemcpyHostToDevice) == cudaSuccess &&
               cudaMemcpy(t->d_a_pages, ap.data(), sizeof(int32_t) * np, cudaMemcpyHostToDevice) == cudaSuccess &&
               cudaMemcpy(t->d_b_pages, bp.data(), sizeof(int32_t) * np, cudaMemcpyHostToDevice) == cudaSuccess &&
               cudaMalloc(reinterpret_cast<void **>(&t->d_ok), size_t(n_adapters)) == cudaSuccess &&
               cudaMemcpy(t->d_ok, okv.data(), size_t(n_adapters), cudaMemcpyHostToDevice) == cudaSuccess;
    cudaSetDevice(prev);
    if (!okk) {
        lora_table_destroy(t);
        return LORA_E_CUDA;
    }
    *out = t;
    return LORA_OK;
}

int lora_table_invalidate(lora_table *t, int adapter)
{
    if (!t || adapter < -1 || adapter >= t->n_adapters)
        return LORA_E_INVAL;
    if (t->dense_valid.empty())
        return LORA_OK;
    if (adapter == -1)
        std::fill(t->dense_valid.begin(), t->dense_valid.end(), uint8_t(0));
    else
        t->dense_valid[size_t(adapter)] = 0;
    return LORA_OK;
}

int lora_table_destroy(lora_table *t)
{
    if (!t)
        return LORA_E_INVAL;
    // Only the table's own fields are used here: the context may already be gone.
    if (t->device < 0) {
        delete t;
        return LORA_OK;
    }
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(t->device);
    // Launches that read the table may still be queued: wait for the device first.
    cudaDeviceSynchronize();
    cudaFree(t->d_rank);
    cudaFree(t->d_scale);
    cudaFree(t->d_a_pages);
    cudaFree(t->d_b_pages);
    cudaFree(t->d_ok);
    cudaFree(t->dense_a);
    cudaFree(t->dense_b);
    cudaSetDevice(prev);
    delete t;
    return LORA_OK;
}

int lora_plan_build(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
                    lora_plan_view *out)
{
    if (!out)
        return LORA_E_INVAL;
    int rc = prepare(ctx, t, ids, n);
    if (rc != LORA_OK)
        return rc;
    Plan &pl = ctx->plan;
    int32_t rmax = 8;
    for (int32_t k : pl.seg_adapter)
        rmax = std::max(rmax, t->rank[size_t(k)]);
    const int64_t n_act = int64_t(pl.active.size());
    const int min_run = (ctx->tile_path && tile_tc_supported(t->a_pw, t->b_pw, rmax))
                            ? tile_min_run(ctx, n_act, t->a_pw, t->b_pw, rmax)
                            : 0;
    const RowsCfg cfg = choose_rows_cfg(ctx, kFused, kKindRowsFused, n_act,
                                        int64_t(pl.seg_adapter.size()), t->a_pw, t->b_pw, rmax);
    plan_items(pl, t->rank.data(), t->scale.data(), cfg.rows, min_run);
    out->n_active = int64_t(pl.active.size());
    out->active_rows = pl.active.data();
    out->perm = pl.perm.data();
    out->n_segments = int64_t(pl.seg_adapter.size());
    out->seg_offsets = pl.seg_offsets.data();
    out->seg_adapter = pl.seg_adapter.data();
    out->row_items = int64_t(pl.row_items.size());
    out->tile_items = int64_t(pl.tile_items.size());
    out->rows_per_item = cfg.rows;
    out->tile_min_run = min_run;
    return LORA_OK;
}

int lora_shrink(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
                const void *x, int64_t ldx, int d_in, float *v, int64_t ldv, void *stream)
{
    return delta_call(ctx, t, kShrink, ids, n, x, ldx, d_in, v, ldv, nullptr, 0, 8,
                      static_cast<cudaStream_t>(stream));
}

int lora_expand(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
                const float *v, int64_t ldv, void *y, int64_t ldy, int d_out, void *stream)
{
    return delta_call(ctx, t, kExpand, ids, n, nullptr, 0, 8, const_cast<float *>(v), ldv, y,
                      ldy, d_out, static_cast<cudaStream_t>(stream));
}

int lora_fused(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
               const void *x, int64_t ldx, int d_in, void *y, int64_t ldy, int d_out,
               void *stream)
{
    return delta_call(ctx, t, kFused, ids, n, x, ldx, d_in, nullptr, 0, y, ldy, d_out,
                      static_cast<cudaStream_t>(stream));
}

// Grow a context-owned device buffer to `need` bytes (after the stream's work that
// may still use the old one).
static int grow_buffer(lora_ctx *ctx, cudaStream_t stream, void **buf, size_t *cap, size_t need)
{
    if (need <= *cap)
        return LORA_OK;
    if (*buf) {
        CUDA_TRY(ctx, cudaStreamSynchronize(stream));
        cudaFree(*buf);
        *buf = nullptr;
        *cap = 0;
    }
    if (cudaMalloc(buf, need) != cudaSuccess) {
        cudaGetLastError();
        return LORA_E_NOMEM;
    }
    *cap = need;
    return LORA_OK;
}

int lora_base_fused(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
                    const void *x, int64_t ldx, int d_in, const void *W, int64_t ldw, void *y,
                    int64_t ldy, int d_out, void *stream_ptr)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (ctx) {
        ctx->last_path = ctx->last_launches = 0;
        begin_call(ctx, stream);
    }
    int rc = prepare(ctx, t, ids, n);
    if (rc != LORA_OK)
        return rc;
    if (n == 0)
        return LORA_OK;
    if (!stride_ok(x, ldx, d_in) || !stride_ok(W, ldw, d_out) || !stride_ok(y, ldy, d_out))
        return LORA_E_INVAL;
    const bool any_active = !ctx->plan.active.empty();
    if (any_active && (d_in > t->a_pw || d_out > t->b_pw))
        return LORA_E_INVAL;
    rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    int32_t rmax = 8;
    for (int32_t k : ctx->plan.seg_adapter)
        rmax = std::max(rmax, t->rank[size_t(k)]);
    // (a multiple of 4 floats: the prep kernel reads a row's v as 16-byte vectors)
    const int64_t ldv = (rmax + 3) & ~int64_t(3);

    // 1. Per 256-row block, the adapters with rows in it (order of first row), each
    //    cut into chunks of 64 columns of its padded rank.
    const int BM = proj_block_rows(), BN = proj_block_cols(), CK = proj_chunk_cols();
    const int n_mblk = int(ceil_div(n, BM)), n_nblk = int(ceil_div(d_out, BN));
    std::vector<int32_t> &mark = ctx->proj_mark, &off = ctx->proj_off, &slots = ctx->proj_slots;
    std::vector<ProjChunk> &chunks = ctx->proj_chunks;
    mark.assign(size_t(t->n_adapters), -1);
    if (ctx->slot_of.size() < size_t(t->n_adapters))
        ctx->slot_of.resize(size_t(t->n_adapters), -1);
    off.assign(size_t(n_mblk) + 1, 0);
    chunks.clear();
    slots.clear();
    for (int m = 0; m < n_mblk; ++m) {
        off[size_t(m)] = int32_t(chunks.size());
        const int64_t r1 = std::min<int64_t>(n, int64_t(m + 1) * BM);
        for (int64_t i = int64_t(m) * BM; i < r1; ++i) {
            const int32_t k = ids[i];
            if (k < 0 || mark[size_t(k)] == m)
                continue;
            mark[size_t(k)] = m;
            if (ctx->slot_of[size_t(k)] < 0) {
                ctx->slot_of[size_t(k)] = int32_t(slots.size());
                slots.push_back(k);
            }
            const int32_t r = t->rank[size_t(k)], rp = (r + 15) & ~15;
            for (int32_t c = 0; c < rp; c += CK)
                chunks.push_back(ProjChunk{k, 0, r, t->scale[size_t(k)], m, c, std::min(CK, rp - c), 0});
        }
    }
    off[size_t(n_mblk)] = int32_t(chunks.size());
    const int n_chunks = int(chunks.size());
    // 2. The B row matrix of those adapters: the pool itself, or dense rows in the
    //    context's own buffer (rank-padded with zero rows).
    const int n_slots = int(slots.size());
    RowMats mats;
    ctx->proj_bbase.assign(size_t(n_slots), 0);
    std::vector<int32_t> a_unused(size_t(n_slots) + 1, 0);
    if (n_slots > 0) {
        const size_t bytes = dense_rows_bytes(t, slots.data(), n_slots, d_in, d_out, false, true);
        rc = grow_buffer(ctx, stream, reinterpret_cast<void **>(&ctx->brows), &ctx->brows_cap, bytes);
        if (rc == LORA_OK)
            rc = setup_rows(ctx, t, slots.data(), n_slots, d_in, d_out, false, true, nullptr, stream,
                            &mats, a_unused.data(), ctx->proj_bbase.data(), ctx->brows);
        if (rc == LORA_OK)
            for (ProjChunk &ch : chunks)
                ch.b_row = ctx->proj_bbase[size_t(ctx->slot_of[size_t(ch.adapter)])] + ch.c;
    }
    for (int32_t k : slots)
        ctx->slot_of[size_t(k)] = -1;
    if (rc != LORA_OK)
        return rc;
    // 3. Scratch: v rows, and the prepared left operands (per chunk 2 x 256 x 64 bf16).
    if (any_active) {
        rc = grow_buffer(ctx, stream, reinterpret_cast<void **>(&ctx->vrows), &ctx->vrows_cap,
                         size_t(n) * size_t(ldv) * 4u);
        if (rc == LORA_OK)
            rc = grow_buffer(ctx, stream, reinterpret_cast<void **>(&ctx->aprep), &ctx->aprep_cap,
                             size_t(n_chunks) * 2u * size_t(BM) * size_t(CK) * 2u);
        if (rc != LORA_OK)
            return rc;
    }
    // 4. Upload the block chunks and the ids in one copy, ahead of the shrink, so that
    //    nothing stands between the shrink and the GEMM in the stream.
    const size_t off_bytes = (size_t(n_mblk + 1) * 4u + 15u) & ~size_t(15);
    const size_t chunk_bytes = chunks.size() * sizeof(ProjChunk);
    const size_t ids_bytes = size_t(n) * 4u;
    Slot *slot = nullptr;
    rc = acquire_slot(ctx, off_bytes + chunk_bytes + ids_bytes + 16, &slot);
    if (rc != LORA_OK)
        return rc;
    std::memcpy(slot->host, off.data(), size_t(n_mblk + 1) * 4u);
    std::memcpy(slot->host + off_bytes, chunks.data(), chunk_bytes);
    std::memcpy(slot->host + off_bytes + chunk_bytes, ids, ids_bytes);
    CUDA_TRY(ctx, cudaMemcpyAsync(slot->dev, slot->host, off_bytes + chunk_bytes + ids_bytes,
                                  cudaMemcpyHostToDevice, stream));
    // 5. v = x A_k for the active rows (the shrink kernels) into the fp32 scratch rows;
    //    d_out: the call's, so that long runs take the tensor-core shrink and its
    //    launch shape comes from the tile table's entry for this shape.
    int path = 0;
    bool untuned = false;
    if (any_active) {
        rc = delta_call(ctx, t, kShrink, ids, n, x, ldx, d_in, ctx->vrows, ldv, nullptr, 0, d_out,
                        stream);
        if (rc != LORA_OK) {
            release_slot(ctx, slot, stream);
            return rc;
        }
        path = ctx->last_path;
        untuned = ctx->untuned;
    }
    // 6. Stage B if needed, prepare the left operands, run the GEMM.
    const long ev = prof_start(ctx, 4, stream);
    if (n_slots > 0) {
        rc = run_staging(ctx, t, mats, stream);
        if (rc != LORA_OK) {
            release_slot(ctx, slot, stream);
            return rc;
        }
    }
    ProjParams p{};
    p.x = static_cast<const uint16_t *>(x);
    p.ldx = ldx;
    p.W = static_cast<const uint16_t *>(W);
    p.ldw = ldw;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = ldy;
    p.v = any_active ? ctx->vrows : nullptr;
    p.ldv = ldv;
    p.chunk_off = reinterpret_cast<const int32_t *>(slot->dev);
    p.chunks = reinterpret_cast<const ProjChunk *>(slot->dev + off_bytes);
    p.ids = reinterpret_cast<const int32_t *>(slot->dev + off_bytes + chunk_bytes);
    p.a_prep = any_active ? ctx->aprep : nullptr;
    p.b_rows = n_slots > 0 ? mats.b : nullptr;
    p.b_ld = mats.b_ld;
    p.b_nrows = mats.b_nrows;
    p.status = ctx->d_status;
    p.n = int(n);
    p.d_in = d_in;
    p.d_out = d_out;
    p.n_mblk = n_mblk;
    p.n_nblk = n_nblk;
    p.n_chunks = n_chunks;
    p.early = n_chunks > 0 ? 1 : 0;   // the prep kernel runs just before the GEMM
    if (n_chunks > 0) {
        CUDA_TRY(ctx, launch_proj_prep(p, stream));
        count_launch(ctx, stream);
    }
    CUDA_TRY(ctx, launch_proj_tc(p, stream));
    prof_stop(ctx, ev, stream);
    count_launch(ctx, stream);
    ctx->last_path = path | 16;
    ctx->untuned = untuned;
    return release_slot(ctx, slot, stream);
}

int lora_fused_noalloc(lora_ctx *ctx, const lora_table *t, const int32_t *ids, int64_t n,
                       const void *x, int64_t ldx, int d_in, void *y, int64_t ldy, int d_out,
                       void *stream_ptr)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (ctx) {
        ctx->last_path = ctx->last_launches = 0;
        begin_call(ctx, stream);
    }
    int rc = prepare(ctx, t, ids, n);
    if (rc != LORA_OK)
        return rc;
    Plan &pl = ctx->plan;
    if (pl.active.empty())
        return LORA_OK;
    if (!stride_ok(x, ldx, d_in) || d_in > t->a_pw || !stride_ok(y, ldy, d_out) || d_out > t->b_pw)
        return LORA_E_INVAL;
    rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    int32_t rmax = 0;
    for (int32_t k : pl.seg_adapter)
        rmax = std::max(rmax, t->rank[size_t(k)]);
    const int64_t n_act = int64_t(pl.active.size());
    bool hit_tiles = true, hit_rows = true;
    const int min_run = (ctx->tile_path && tile_tc_supported(d_in, d_out, rmax))
                            ? tile_min_run(ctx, n_act, d_in, d_out, rmax, &hit_tiles)
                            : 0;
    RowsCfg cfg = choose_rows_cfg(ctx, kFused, kKindRowsFused, n_act,
                                  int64_t(pl.seg_adapter.size()), d_in, d_out, rmax, &hit_rows);
    plan_items(pl, t->rank.data(), t->scale.data(), cfg.rows, min_run);
    // Everything must fit the fixed arrays and the launch parameter block.
    if (pl.tile_items.size() > size_t(kNoAllocSlots) ||
        pl.row_items.size() > size_t(kInlineItems) || pl.row_perm.size() > size_t(kInlinePerm))
        return LORA_E_CAPACITY;
    if (!pl.tile_items.empty() && pl.row_active > 0 && pl.row_active < n_act)
        cfg = choose_rows_cfg(ctx, kFused, kKindRowsFused, pl.row_active,
                              int64_t(pl.row_items.size()), d_in, d_out, pl.row_max_rank, &hit_rows);
    // The minimum run is a tuned decision only where a run could reach a tile (the
    // search's shortest candidate is 32 rows).
    ctx->untuned = (!hit_tiles && pl.max_seg_len >= 32) || (!pl.row_items.empty() && !hit_rows);
    NoAllocScratch fixed{};
    CUDA_TRY(ctx, noalloc_scratch(ctx->device, false, &fixed));
    const bool prof = ctx->prof;
    ctx->prof = false;   // the event pool could grow
    rc = run_tiles(ctx, t, kFused, x, ldx, d_in, nullptr, 0, y, ldy, d_out, n, stream, &fixed);
    if (rc == LORA_OK)
        rc = run_rows(ctx, t, kFused, cfg, x, ldx, d_in, nullptr, 0, y, ldy, d_out, stream);
    ctx->prof = prof;
    return rc;
}

int lora_fused_args_call(const lora_fused_args *a)
{
    if (!a)
        return LORA_E_INVAL;
    return delta_call(a->ctx, a->table, kFused, a->ids, a->n, a->x, a->ldx, a->d_in, nullptr, 0,
                      a->y, a->ldy, a->d_out, static_cast<cudaStream_t>(a->stream));
}

int lora_fused_device_ids_args_call(const lora_fused_args *a)
{
    if (!a)
        return LORA_E_INVAL;
    return lora_fused_device_ids(a->ctx, a->table, a->ids, a->n, a->x, a->ldx, a->d_in, a->y,
                                 a->ldy, a->d_out, a->stream);
}

int lora_fused_device_ids(lora_ctx *ctx, const lora_table *t, const int32_t *ids_dev, int64_t n,
                          const void *x, int64_t ldx, int d_in, void *y, int64_t ldy, int d_out,
                          void *stream_ptr)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (ctx) {
        ctx->last_path = ctx->last_launches = 0;
        begin_call(ctx, stream);
    }
    if (!ctx || !t || t->ctx != ctx || n < 0 || n > ctx->max_rows ||
        (n > 0 && (!ids_dev || (reinterpret_cast<uintptr_t>(ids_dev) & 3u))))
        return LORA_E_INVAL;
    if (t->n_adapters > kDevPlanMaxAdapters)
        return LORA_E_UNSUPPORTED;
    if (n == 0)
        return LORA_OK;
    if (!stride_ok(x, ldx, d_in) || d_in > t->a_pw || !stride_ok(y, ldy, d_out) || d_out > t->b_pw)
        return LORA_E_INVAL;
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    if (t->rank_max_ok == 0)
        return LORA_E_ADAPTER;   // no adapter of the table can be served
    // Launch shape from what the host knows: the batch size and the table.  Every
    // row may be on its own adapter, so the grid has room for n items; the surplus
    // clusters leave as soon as they read the plan's count (planned mode) or their
    // row's id (direct mode: one row per cluster, no plan kernel).
    const int64_t n_seg = std::min<int64_t>(n, t->n_adapters);
    bool hit_rows = true;
    RowsCfg cfg = choose_rows_cfg(ctx, kFused, kKindRowsFused, n, n_seg, d_in, d_out, t->rank_max_ok,
                                  &hit_rows);
    ctx->untuned = !hit_rows;
    if (!ctx->device_plan)
        cfg.rows = 1;
    RowsParams p{};
    size_t smem = 0;
    rc = rows_launch_params(ctx, kFused, cfg, d_in, d_out, t->rank_max_ok,
                            !ctx->device_plan && ctx->call_early_x, n, p, smem);
    if (rc != LORA_OK)
        return rc;
    p.x = static_cast<const uint16_t *>(x);
    p.ldx = ldx;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = ldy;
    p.a_pool = t->a_pool;
    p.a_pw = t->a_pw;
    p.b_pool = t->b_pool;
    p.b_pw = t->b_pw;
    p.a_pages = t->d_a_pages;
    p.b_pages = t->d_b_pages;
    p.rank = t->d_rank;
    p.scale = t->d_scale;
    p.status = ctx->d_status;
    p.max_rank = t->max_rank;
    p.d_in = d_in;
    p.d_out = d_out;
    p.n_items = int(n);
    p.early_pages = 0;   // planned: the plan is the previous kernel's output
    if (!ctx->device_plan) {
        p.early_pages = ctx->call_early;   // ids and pages read ahead of the wait
        p.early_x = ctx->call_early_x;
        p.ids_dev = ids_dev;
        p.ok = t->d_ok;
        p.n_adapters = t->n_adapters;
        const long ev = prof_start(ctx, 0, stream);
        CUDA_TRY(ctx, launch_rows(kFused, p, smem, stream));
        prof_stop(ctx, ev, stream);
        count_launch(ctx, stream);
        ctx->last_path = 1;
        return LORA_OK;
    }
    RowItem *items = reinterpret_cast<RowItem *>(ctx->d_dplan);
    int32_t *perm = reinterpret_cast<int32_t *>(ctx->d_dplan + size_t(ctx->max_rows) * sizeof(RowItem));
    int32_t *count = reinterpret_cast<int32_t *>(ctx->d_dplan + size_t(ctx->max_rows) * 20);
    DevPlanArgs pa{};
    pa.ids = ids_dev;
    pa.n = int(n);
    pa.rank = t->d_rank;
    pa.scale = t->d_scale;
    pa.ok = t->d_ok;
    pa.n_adapters = t->n_adapters;
    pa.rows_per_item = p.rows_alloc;
    pa.items = items;
    pa.perm = perm;
    pa.n_items = count;
    pa.status = ctx->d_status;
    CUDA_TRY(ctx, launch_plan_dev(pa, stream));
    count_launch(ctx, stream);
    p.items = items;
    p.perm = perm;
    p.n_items_dev = count;
    const long ev = prof_start(ctx, 0, stream);
    CUDA_TRY(ctx, launch_rows(kFused, p, smem, stream));
    prof_stop(ctx, ev, stream);
    count_launch(ctx, stream);
    ctx->last_path = 1;
    return LORA_OK;
}

int lora_merge(lora_ctx *ctx, const lora_table *t, int adapter, void *W, int64_t ldw, int d_in,
               int d_out, void *stream)
{
    return merge_call(ctx, t, adapter, W, ldw, d_in, d_out, +1.f,
                      static_cast<cudaStream_t>(stream));
}

int lora_unmerge(lora_ctx *ctx, const lora_table *t, int adapter, void *W, int64_t ldw,
                 int d_in, int d_out, void *stream)
{
    return merge_call(ctx, t, adapter, W, ldw, d_in, d_out, -1.f,
                      static_cast<cudaStream_t>(stream));
}

int lora_page_in(lora_ctx *ctx, const lora_table *t, int adapter, const void *host_a, int d_in,
                 const void *host_b, int d_out, void *stream_ptr)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (ctx)
        ctx->last_path = ctx->last_launches = 0;
    if (!ctx || !t || t->ctx != ctx)
        return LORA_E_INVAL;
    if (adapter < 0 || adapter >= t->n_adapters)
        return LORA_E_ADAPTER;
    if (t->status[size_t(adapter)] != LORA_OK)
        return t->status[size_t(adapter)];
    if (!host_a || !host_b || !aligned16(host_a) || !aligned16(host_b) || d_in <= 0 || d_out <= 0 ||
        (d_in % 8) || (d_out % 8) || d_in > t->a_pw || d_out > t->b_pw)
        return LORA_E_INVAL;
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    // Both buffers must be page-locked host memory mapped into the device's address
    // space: the kernel reads them directly.  Anything else is refused here, before
    // any launch.
    const void *dev_src[2] = {nullptr, nullptr};
    const void *host[2] = {host_a, host_b};
    for (int side = 0; side < 2; ++side) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, host[side]) != cudaSuccess) {
            (void)cudaGetLastError();
            return LORA_E_INVAL;
        }
        if (at.type != cudaMemoryTypeHost || !at.devicePointer)
            return LORA_E_INVAL;
        dev_src[side] = at.devicePointer;
    }
    const int r = t->rank[size_t(adapter)];
    PageInArgs a{};
    a.rank = r;
    a.side[0].host = static_cast<const uint16_t *>(dev_src[0]);
    a.side[0].pool = const_cast<uint16_t *>(t->a_pool);
    a.side[0].pw = t->a_pw;
    a.side[0].width = d_in;
    a.side[1].host = static_cast<const uint16_t *>(dev_src[1]);
    a.side[1].pool = const_cast<uint16_t *>(t->b_pool);
    a.side[1].pw = t->b_pw;
    a.side[1].width = d_out;
    for (int j = 0; j < r; ++j) {
        a.side[0].page[j] = t->a_pages[size_t(adapter) * t->max_rank + j];
        a.side[1].page[j] = t->b_pages[size_t(adapter) * t->max_rank + j];
    }
    CUDA_TRY(ctx, launch_page_in(a, stream));
    // the adapter's dense rows (if the table keeps them) no longer match its pages
    lora_table *tw = const_cast<lora_table *>(t);
    if (!tw->dense_valid.empty())
        tw->dense_valid[size_t(adapter)] = 0;
    ctx->last_path = 8;
    ctx->last_launches = 1;
    ctx->launches_total += 1;
    ctx->pool_write_stream = stream;
    ctx->pool_write_pending = true;
    return LORA_OK;
}

int lora_selftest_timeout(lora_ctx *ctx, int64_t limit_us, void *stream)
{
    if (!ctx || limit_us < 1 || limit_us > 1000000)
        return LORA_E_INVAL;
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    CUDA_TRY(ctx, launch_wait_selftest(ctx->d_status, uint64_t(limit_us) * 1000u,
                                       static_cast<cudaStream_t>(stream)));
    ctx->launches_total += 1;
    return LORA_OK;
}

int lora_tiles_load(lora_ctx *ctx, const char *path)
{
    if (!ctx || !path)
        return LORA_E_INVAL;
    return ctx->tiles.load(path);
}

int lora_tiles_save(const lora_ctx *ctx, const char *path)
{
    if (!ctx || !path)
        return LORA_E_INVAL;
    return ctx->tiles.save(path);
}

int64_t lora_tiles_count(const lora_ctx *ctx) { return ctx ? int64_t(ctx->tiles.map.size()) : -1; }

int lora_tile_status(const lora_ctx *ctx)
{
    if (!ctx)
        return LORA_E_INVAL;
    return ctx->untuned ? LORA_E_NOTUNED : LORA_OK;
}

int lora_sync_status(lora_ctx *ctx, void *stream)
{
    if (!ctx)
        return LORA_E_INVAL;
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    CUDA_TRY(ctx, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    unsigned word = 0;
    CUDA_TRY(ctx, cudaMemcpy(&word, ctx->d_status, sizeof word, cudaMemcpyDeviceToHost));
    if (word != 0) {
        CUDA_TRY(ctx, cudaMemset(ctx->d_status, 0, sizeof word));
        return word == kDevBadId ? LORA_E_ADAPTER : LORA_E_TIMEOUT;
    }
    return LORA_OK;
}

int lora_ctx_set_option(lora_ctx *ctx, int option, int value)
{
    if (!ctx)
        return LORA_E_INVAL;
    rcache_clear(ctx);
    switch (option) {
    case LORA_OPT_TILE_PATH: ctx->tile_path = value ? 1 : 0; return LORA_OK;
    case LORA_OPT_MERGE_KERNEL:
        if (value < 0 || value > 1)
            return LORA_E_INVAL;
        ctx->merge_path = value;
        return LORA_OK;
    case LORA_OPT_TILE_MIN_RUN:
        if (value < 0)
            return LORA_E_INVAL;
        ctx->tile_min_run_override = value;
        return LORA_OK;
    case LORA_OPT_EARLY_PAGES: ctx->early_pages = value ? 1 : 0; return LORA_OK;
    case LORA_OPT_EARLY_INPUT: ctx->early_input = value ? 1 : 0; return LORA_OK;
    case LORA_OPT_DEVICE_PLAN: ctx->device_plan = value ? 1 : 0; return LORA_OK;
    case LORA_OPT_ROWS_B_OVER_A:
        if (value < -1 || value > 1)
            return LORA_E_INVAL;
        ctx->b_over_a = value;
        return LORA_OK;
    default: return LORA_E_INVAL;
    }
}

int lora_profile_begin(lora_ctx *ctx, int every)
{
    if (!ctx || every < 1)
        return LORA_E_INVAL;
    ctx->prof = true;
    ctx->prof_used = 0;
    ctx->prof_every = every;
    for (int64_t &c : ctx->prof_seen)
        c = 0;
    return LORA_OK;
}

int lora_profile_end(lora_ctx *ctx, double *ms, int64_t *launches)
{
    if (!ctx || !ms || !launches)
        return LORA_E_INVAL;
    ctx->prof = false;
    for (int f = 0; f < kFamilies; ++f) {
        ms[f] = 0.0;
        launches[f] = 0;
    }
    int64_t sampled[kFamilies] = {0, 0, 0, 0, 0};
    for (size_t i = 0; i < ctx->prof_used; ++i) {
        lora_ctx::ProfEv &e = ctx->prof_ev[i];
        CUDA_TRY(ctx, cudaEventSynchronize(e.b));
        float t = 0.f;
        CUDA_TRY(ctx, cudaEventElapsedTime(&t, e.a, e.b));
        ms[e.family] += double(t);
        sampled[e.family] += 1;
    }
    // The bracketed launches stand for all of their family: mean x count.
    for (int f = 0; f < kFamilies; ++f) {
        launches[f] = ctx->prof_seen[f];
        if (sampled[f] > 0)
            ms[f] *= double(ctx->prof_seen[f]) / double(sampled[f]);
    }
    ctx->prof_used = 0;
    return LORA_OK;
}

int64_t lora_launch_count(const lora_ctx *ctx) { return ctx ? ctx->launches_total : -1; }

int lora_last_path(const lora_ctx *ctx, int *n_launches)
{
    if (!ctx)
        return LORA_E_INVAL;
    if (n_launches)
        *n_launches = ctx->last_launches;
    return ctx->last_path;
}

int lora_tune_shape(lora_ctx *ctx, const lora_table *t, int kind, const int32_t *ids, int64_t n,
                    const void *x, int64_t ldx, int d_in, void *y, int64_t ldy, int d_out,
                    int iters, float *best_us, void *stream_ptr)
{
    if (!ctx || !t || !best_us || iters < 1 || kind < 0 || kind > 4 || !ids || n < 1)
        return LORA_E_INVAL;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    // One candidate: warm up twice, then the median of `iters` calls, each timed
    // alone and started with L2 cold (a 256 MB write first), as a serving step meets
    // its adapters after the rest of the model has streamed through the cache.
    constexpr size_t kFlushBytes = size_t(256) << 20;
    if (!ctx->flush && cudaMalloc(reinterpret_cast<void **>(&ctx->flush), kFlushBytes) != cudaSuccess)
        return LORA_E_NOMEM;
    cudaEvent_t e0, e1;
    CUDA_TRY(ctx, cudaEventCreate(&e0));
    CUDA_TRY(ctx, cudaEventCreate(&e1));
    auto call = [&]() -> int {
        switch (kind) {
        case kKindShrink: return LORA_E_UNSUPPORTED;
        case kKindExpand: return LORA_E_UNSUPPORTED;
        case kKindMerge: return lora_merge(ctx, t, ids[0], y, ldy, d_in, d_out, stream);
        default: return lora_fused(ctx, t, ids, n, x, ldx, d_in, y, ldy, d_out, stream);
        }
    };
    auto time_it = [&](float &us) -> int {
        for (int w = 0; w < 2; ++w) {
            int r2 = call();
            if (r2 != LORA_OK)
                return r2;
        }
        std::vector<float> t_ms;
        t_ms.reserve(size_t(iters));
        for (int i = 0; i < iters; ++i) {
            if (cudaMemsetAsync(ctx->flush, i & 0xff, kFlushBytes, stream) != cudaSuccess ||
                cudaEventRecord(e0, stream) != cudaSuccess)
                return LORA_E_CUDA;
            int r2 = call();
            if (r2 != LORA_OK)
                return r2;
            if (cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess)
                return LORA_E_CUDA;
            float ms = 0.f;
            cudaEventElapsedTime(&ms, e0, e1);
            t_ms.push_back(ms);
        }
        std::nth_element(t_ms.begin(), t_ms.begin() + iters / 2, t_ms.end());
        us = 1000.f * t_ms[size_t(iters / 2)];
        return LORA_OK;
    };
    // The key of the shape, as the runtime will look it up.
    rc = prepare(ctx, t, ids, n);
    if (rc != LORA_OK) {
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        return rc;
    }
    int32_t rmax = 8;
    for (int32_t k : ctx->plan.seg_adapter)
        rmax = std::max(rmax, t->rank[size_t(k)]);
    if (kind == kKindMerge)
        rmax = t->rank[size_t(ids[0])];
    const int64_t n_act = int64_t(ctx->plan.active.size());
    const TileKey key{kind, kind == kKindMerge ? pow2_bucket(d_in) : pow2_bucket(n_act),
                      kind == kKindRowsFused ? pow2_bucket(int64_t(ctx->plan.seg_adapter.size())) : 0,
                      d_in, d_out, rmax};
    float best = -1.f;
    TileCfg best_cfg{0, 0, 0, 0};
    const int saved_tile = ctx->tile_path, saved_merge = ctx->merge_path,
              saved_run = ctx->tile_min_run_override;
    if (kind == kKindRowsFused) {
        // Pruned space (VaLoRA blog 4.3.2: hardware limits and dimensions that are
        // multiples of the tile): power-of-two cluster widths whose slices are at
        // least 64 elements and fit shared memory, rows per item up to the longest
        // segment.
        ctx->tile_path = 0;
        const int seg_max = ctx->plan.max_seg_len;
        for (int C = 1; C <= rows_max_cluster(); C *= 2) {
            if (C > 1 && std::min(d_in, d_out) / C < 64)
                break;
            for (int R = 1; R <= 16; R *= 2) {
                if (R > 1 && R / 2 >= seg_max)
                    break;
                if (rows_smem_for(kFused, C, R, rmax, d_in, d_out) > size_t(rows_max_smem()))
                    continue;
                ctx->force_cluster = C;
                ctx->force_rows = R;
                float us = 0.f;
                if (time_it(us) == LORA_OK && (best < 0.f || us < best)) {
                    best = us;
                    best_cfg = TileCfg{C, R, 0, 0};
                }
            }
        }
        ctx->force_cluster = ctx->force_rows = 0;
    } else if (kind == kKindTileFused) {
        // Up to 256: a longer minimum would send prompt-length runs of a batch with
        // mixed lengths to the row-gather kernel, which the tuned shape may not show.
        const int runs[] = {32, 64, 128, 256};
        for (int m : runs) {
            ctx->tile_min_run_override = m;
            float us = 0.f;
            if (time_it(us) == LORA_OK && (best < 0.f || us < best)) {
                best = us;
                best_cfg = TileCfg{m, 0, 0, 0};
            }
        }
    } else if (kind == kKindMerge) {
        for (int path = 0; path <= 1; ++path) {
            ctx->merge_path = path;
            float us = 0.f;
            if (time_it(us) == LORA_OK && (best < 0.f || us < best)) {
                best = us;
                best_cfg = TileCfg{path, 0, 0, 0};
            }
        }
    } else {
        rc = LORA_E_UNSUPPORTED;
    }
    ctx->tile_path = saved_tile;
    ctx->merge_path = saved_merge;
    ctx->tile_min_run_override = saved_run;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (rc != LORA_OK)
        return rc;
    if (best < 0.f)
        return LORA_E_UNSUPPORTED;
    ctx->tiles.put(key, best_cfg);
    *best_us = best;
    return LORA_OK;
}

}  // extern "C"

namespace {

// ---------------------------------------------------------------- lora_tune: shape file

struct TuneShape {
    int kind = 0;             // kKindRowsFused, kKindTileFused or kKindMerge
    int64_t n = 1;
    int d_in = 0, d_out = 0, rank = 0, adapters = 1;
    int64_t run = 0;          // rows per request; 0: ids cycle over the adapters
    bool throughput = false;
    std::string text;
};

// One shape per line: kind n d_in d_out rank adapters [run [objective]], kind one of
// rows / tiles / merge, objective latency (default) or throughput (rows only); '#'
// starts a comment.  Checked in full before anything runs.
int parse_shapes(const char *path, int max_rank, std::vector<TuneShape> &out)
{
    std::FILE *f = std::fopen(path, "r");
    if (!f)
        return LORA_E_IO;
    char buf[512];
    int rc = LORA_OK;
    while (rc == LORA_OK && std::fgets(buf, sizeof buf, f)) {
        std::string line(buf);
        const size_t hash = line.find('#');
        if (hash != std::string::npos)
            line.resize(hash);
        std::vector<std::string> tok;
        size_t i = 0;
        while (i < line.size()) {
            while (i < line.size() && std::isspace(static_cast<unsigned char>(line[i])))
                ++i;
            size_t j = i;
            while (j < line.size() && !std::isspace(static_cast<unsigned char>(line[j])))
                ++j;
            if (j > i)
                tok.push_back(line.substr(i, j - i));
            i = j;
        }
        if (tok.empty())
            continue;
        if (tok.size() < 6 || tok.size() > 8) {
            rc = LORA_E_INVAL;
            break;
        }
        TuneShape sh;
        if (tok[0] == "rows")
            sh.kind = kKindRowsFused;
        else if (tok[0] == "tiles")
            sh.kind = kKindTileFused;
        else if (tok[0] == "merge")
            sh.kind = kKindMerge;
        else
            rc = LORA_E_INVAL;
        int64_t v[7] = {0, 0, 0, 0, 0, 0, 0};
        for (size_t q = 1; q < std::min<size_t>(tok.size(), 7) && rc == LORA_OK; ++q) {
            char *end = nullptr;
            v[q] = std::strtoll(tok[q].c_str(), &end, 10);
            if (!end || *end != '\0')
                rc = LORA_E_INVAL;
        }
        if (rc != LORA_OK)
            break;
        sh.n = v[1];
        sh.d_in = int(v[2]);
        sh.d_out = int(v[3]);
        sh.rank = int(v[4]);
        sh.adapters = int(v[5]);
        sh.run = tok.size() > 6 ? v[6] : 0;
        if (tok.size() > 7) {
            if (tok[7] == "throughput")
                sh.throughput = true;
            else if (tok[7] != "latency")
                rc = LORA_E_INVAL;
        }
        if (sh.n < 1 || sh.n > (int64_t(1) << 24) || v[2] < 8 || v[2] > 65536 || (v[2] % 8) ||
            v[3] < 8 || v[3] > 65536 || (v[3] % 8) || sh.rank < 8 || (sh.rank % 8) ||
            sh.rank > max_rank || sh.adapters < 1 || sh.adapters > 4096 || sh.run < 0 ||
            (sh.throughput && sh.kind != kKindRowsFused))
            rc = LORA_E_INVAL;
        sh.text = tok[0];
        for (size_t q = 1; q < tok.size(); ++q)
            sh.text += " " + tok[q];
        out.push_back(sh);
    }
    std::fclose(f);
    return rc;
}

// Device buffers of one tuning shape, freed when it goes out of scope.
struct TuneBuffers {
    std::vector<void *> mem;
    std::vector<lora_table *> tables;
    ~TuneBuffers()
    {
        for (lora_table *t : tables)
            lora_table_destroy(t);
        for (void *p : mem)
            cudaFree(p);
    }
    uint16_t *alloc(size_t elems)
    {
        void *p = nullptr;
        if (cudaMalloc(&p, elems * 2) != cudaSuccess)
            return nullptr;
        mem.push_back(p);
        return static_cast<uint16_t *>(p);
    }
};

// Run one shape of lora_tune on synthetic data: values uniform with the variances of
// the workloads (x and W unit / 1/d_in, A 1/d_in, B 1/r), filled on the device.
int tune_one(lora_ctx *ctx, const TuneShape &sh, int index, cudaStream_t stream, float *best_us)
{
    const int na = sh.adapters, r = sh.rank;
    const bool merge = sh.kind == kKindMerge;
    const int64_t n = merge ? 1 : sh.n;
    std::vector<int32_t> rank(size_t(na), r), pages(size_t(na) * r);
    std::vector<float> scale(size_t(na), 16.f / float(r));
    for (size_t i = 0; i < pages.size(); ++i)
        pages[i] = int32_t(i);
    std::vector<int32_t> ids(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i)
        ids[size_t(i)] = int32_t((sh.run > 0 ? i / sh.run : i) % na);
    const size_t pool_a = size_t(na) * r * size_t(sh.d_in), pool_b = size_t(na) * r * size_t(sh.d_out);
    const size_t act = merge ? size_t(sh.d_in) * size_t(sh.d_out) : size_t(n) * (sh.d_in + sh.d_out);
    int sets = 1;
    if (sh.throughput)   // inputs over a pass larger than L2, as a decode loop meets them
        sets = int(std::min<size_t>(64, std::max<size_t>(2, ((size_t(256) << 20) + 2 * (pool_a + pool_b + act) - 1) /
                                                               (2 * (pool_a + pool_b + act)))));
    TuneBuffers b;
    std::vector<uint16_t *> xs, ys;
    const uint64_t seed0 = uint64_t(index) * 1000003ull;
    for (int s = 0; s < sets; ++s) {
        uint16_t *a = b.alloc(pool_a), *bb = b.alloc(pool_b);
        uint16_t *x = merge ? nullptr : b.alloc(size_t(n) * sh.d_in);
        uint16_t *y = b.alloc(merge ? size_t(sh.d_in) * sh.d_out : size_t(n) * sh.d_out);
        if (!a || !bb || (!merge && !x) || !y)
            return LORA_E_NOMEM;
        const uint64_t sd = seed0 + uint64_t(s) * 16;
        CUDA_TRY(ctx, launch_fill_bf16(a, pool_a, sd + 1, std::sqrt(3.f / float(sh.d_in)), stream));
        CUDA_TRY(ctx, launch_fill_bf16(bb, pool_b, sd + 2, std::sqrt(3.f / float(r)), stream));
        if (x)
            CUDA_TRY(ctx, launch_fill_bf16(x, size_t(n) * sh.d_in, sd + 3, std::sqrt(3.f), stream));
        CUDA_TRY(ctx, launch_fill_bf16(y, merge ? size_t(sh.d_in) * sh.d_out : size_t(n) * sh.d_out, sd + 4,
                                       merge ? std::sqrt(3.f / float(sh.d_in)) : std::sqrt(3.f), stream));
        lora_table *t = nullptr;
        int rc = lora_table_create(ctx, a, int64_t(na) * r, sh.d_in, bb, int64_t(na) * r, sh.d_out, na, r,
                                   rank.data(), scale.data(), pages.data(), pages.data(), &t);
        if (rc != LORA_OK)
            return rc;
        b.tables.push_back(t);
        xs.push_back(x);
        ys.push_back(y);
    }
    CUDA_TRY(ctx, cudaStreamSynchronize(stream));
    if (!sh.throughput) {
        if (merge)
            return lora_tune_shape(ctx, b.tables[0], kKindMerge, ids.data(), 1, ys[0], sh.d_out,
                                   sh.d_in, ys[0], sh.d_out, sh.d_out, 31, best_us, stream);
        return lora_tune_shape(ctx, b.tables[0], sh.kind, ids.data(), n, xs[0], sh.d_in, sh.d_in, ys[0],
                               sh.d_out, sh.d_out, 31, best_us, stream);
    }
    // Throughput of back-to-back calls over the rotating sets, per candidate launch
    // shape of the row-gather kernel (the space lora_tune_shape searches).
    int seg_max = 0;
    {
        std::vector<int> cnt(size_t(na), 0);
        for (int32_t k : ids)
            seg_max = std::max(seg_max, ++cnt[size_t(k)]);
    }
    cudaEvent_t e0, e1;
    CUDA_TRY(ctx, cudaEventCreate(&e0));
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return LORA_E_CUDA;
    }
    const int saved_tile = ctx->tile_path;
    ctx->tile_path = 0;
    constexpr int kSteps = 1500;
    float best = -1.f;
    TileCfg best_cfg{0, 0, 0, 0};
    int rc = LORA_OK;
    for (int C = 1; C <= rows_max_cluster() && rc == LORA_OK; C *= 2) {
        if (C > 1 && std::min(sh.d_in, sh.d_out) / C < 64)
            break;
        for (int R = 1; R <= 16 && rc == LORA_OK; R *= 2) {
            if (R > 1 && R / 2 >= seg_max)
                break;
            if (rows_smem_for(kFused, C, R, r, sh.d_in, sh.d_out) > size_t(rows_max_smem()))
                continue;
            ctx->force_cluster = C;
            ctx->force_rows = R;
            for (int i = 0; i < 20 && rc == LORA_OK; ++i)
                rc = lora_fused(ctx, b.tables[size_t(i % sets)], ids.data(), n, xs[size_t(i % sets)], sh.d_in,
                                sh.d_in, ys[size_t(i % sets)], sh.d_out, sh.d_out, stream);
            if (rc == LORA_OK && cudaEventRecord(e0, stream) != cudaSuccess)
                rc = LORA_E_CUDA;
            for (int i = 0; i < kSteps && rc == LORA_OK; ++i)
                rc = lora_fused(ctx, b.tables[size_t(i % sets)], ids.data(), n, xs[size_t(i % sets)], sh.d_in,
                                sh.d_in, ys[size_t(i % sets)], sh.d_out, sh.d_out, stream);
            if (rc == LORA_OK &&
                (cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess))
                rc = LORA_E_CUDA;
            float ms = 0.f;
            if (rc == LORA_OK && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess) {
                const float us = 1000.f * ms / float(kSteps);
                if (best < 0.f || us < best) {
                    best = us;
                    best_cfg = TileCfg{C, R, 0, 0};
                }
            }
        }
    }
    ctx->force_cluster = ctx->force_rows = 0;
    ctx->tile_path = saved_tile;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (rc != LORA_OK)
        return rc;
    if (best < 0.f)
        return LORA_E_UNSUPPORTED;
    ctx->tiles.put(TileKey{kKindRowsFused, pow2_bucket(n), pow2_bucket(std::min<int64_t>(na, n)), sh.d_in,
                           sh.d_out, r},
                   best_cfg);
    *best_us = best;
    return LORA_OK;
}

}  // namespace

extern "C" {

int lora_tune(lora_ctx *ctx, const char *shapes_path, const char *out_path, void *stream_ptr)
{
    if (!ctx || !shapes_path)
        return LORA_E_INVAL;
    std::vector<TuneShape> shapes;
    int rc = parse_shapes(shapes_path, ctx->max_rank, shapes);
    if (rc != LORA_OK)
        return rc;
    rc = use_device(ctx);
    if (rc != LORA_OK)
        return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    std::vector<float> best(shapes.size(), 0.f);
    for (size_t i = 0; i < shapes.size(); ++i) {
        rc = tune_one(ctx, shapes[i], int(i), stream, &best[i]);
        if (rc != LORA_OK)
            return rc;
    }
    if (!out_path)
        return LORA_OK;
    rc = ctx->tiles.save(out_path);
    if (rc != LORA_OK)
        return rc;
    std::FILE *f = std::fopen(out_path, "a");
    if (!f)
        return LORA_E_IO;
    for (size_t i = 0; i < shapes.size(); ++i)
        std::fprintf(f, "# tuned: %s -> %.3f us (%s)\n", shapes[i].text.c_str(), double(best[i]),
                     shapes[i].throughput ? "back-to-back calls" : "cold single call, median");
    return std::fclose(f) == 0 ? LORA_OK : LORA_E_IO;
}

}  // extern "C"
