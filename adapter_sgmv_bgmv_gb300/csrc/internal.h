// Host-side structures shared by the C-ABI layer and the kernel launchers.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace lora {

// One work item of the row-gather kernel: `nrows` consecutive entries of the
// by-adapter permutation starting at `p0`, all on adapter `adapter` of rank `rank`
// and scale `scale` (carried here so the kernel needs no lookup before its copies).
struct RowItem {
    int32_t adapter;
    int32_t p0;
    int16_t nrows;
    int16_t rank;
    float scale;
};
static_assert(sizeof(RowItem) == 16, "RowItem is one 16-byte load");

// One tile of the tensor-core kernels: rows [row0, row0 + nrows) of x / y (a run of
// consecutive rows that share adapter `adapter`), nrows <= 128.
struct TileItem {
    int32_t adapter;
    int32_t row0;
    int16_t nrows;
    int16_t rank;
    float scale;
    int32_t a_row;            // row of page 0 of A_k in the A row matrix (pages j: a_row + j)
    int32_t b_row;            // row of page 0 of B_k in the B row matrix
    int32_t pad[2];
};
static_assert(sizeof(TileItem) == 32, "TileItem is two 16-byte loads");

enum Mode : int { kShrink = 0, kExpand = 1, kFused = 2 };

// Everything a row-gather launch needs (passed by value as the kernel parameter).
struct RowsParams {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    float *v;
    int64_t ldv;
    const uint16_t *a_pool;
    int64_t a_pw;
    const uint16_t *b_pool;
    int64_t b_pw;
    const int32_t *a_pages;   // device copy, [n_adapters * max_rank]
    const int32_t *b_pages;
    const int32_t *rank;      // device copy, [n_adapters]
    const float *scale;       // device copy, [n_adapters]
    const RowItem *items;
    const int32_t *perm;
    unsigned *status;
    int max_rank;
    int d_in;
    int d_out;
    int n_items;
    int cluster;              // CTAs per item (split of d_in and of d_out)
    int slice_in;             // elements of d_in per CTA (multiple of 8)
    int slice_out;            // elements of d_out per CTA (multiple of 8)
    int rows_alloc;           // shared-memory rows per item (>= every item's nrows)
    int early_pages;          // 1: adapter page copies issued before the dependency wait
    int early_x;              // 1: x, the shrink and the exchange before it as well
    int no_y_smem;            // 1: every CTA reads y after the wait, straight from memory
                              //    (fused, early_x, one output vector per thread): no y rows
                              //    in shared memory
    int b_over_a;             // 1 (fused): B's page slices are copied into A's shared
                              //    memory once the shrink has read it (half the footprint,
                              //    so more CTAs are resident at once)
    int rank_alloc;           // shared-memory rank slots (>= every item's rank)
    const int32_t *n_items_dev;   // device-side plan: the item count (items past it idle),
                                  // read after the wait for the kernel that wrote the plan
    const int32_t *ids_dev;       // direct mode: one row per item, item i = row i, its
                                  // adapter read from here after the wait (no plan)
    const uint8_t *ok;            // direct mode: 1 where the table can serve the adapter
    int n_adapters;               // direct mode
};

// Small plans travel inside the kernel parameter block (no separate upload), in
// one of two sizes so that a decode batch does not ship an oversized block.
constexpr int kInlineItems = 256;
constexpr int kInlinePerm = 512;
template <int NI, int NP>
struct RowsParamsInlineT {
    RowsParams p;
    RowItem items[NI];
    int32_t perm[NP];
};
using RowsParamsInline = RowsParamsInlineT<kInlineItems, kInlinePerm>;
using RowsParamsInlineSmall = RowsParamsInlineT<64, 128>;

size_t rows_smem_bytes(int mode, int slice_in, int slice_out, int rows_alloc, int rank_alloc,
                       int cluster, bool no_y = false, bool b_over_a = false);
// CTAs of a row-gather launch with this much dynamic shared memory that one SM holds
// at once (shared memory and the kernel instance's register budget).
int rows_ctas_per_sm(int mode, size_t smem);
// Whether a launch with these parameters has every CTA read y after the dependency
// wait (then its shared memory holds no y rows).
bool rows_y_late(int mode, bool early_x, int slice_out, int rows_alloc);
int rows_max_cluster();
cudaError_t launch_rows(int mode, const RowsParams &p, size_t smem, cudaStream_t stream);
cudaError_t launch_rows_inline(int mode, const RowsParamsInline &a, size_t smem,
                               cudaStream_t stream);
cudaError_t launch_rows_inline_small(int mode, const RowsParamsInlineSmall &a, size_t smem,
                                     cudaStream_t stream);
int rows_max_smem();

// Tensor-core tile kernels (tile_tc.cu, stream_tc.cu).  In the fused call the shrink
// splits K over `ksplit` CTAs per tile; each writes its fp32 partial V (128 rows x
// r_pad) into its own 64 KB slot of a scratch that the expand sums in order.
constexpr int kVPartBytes = 128 * 128 * 4;
// Tile lists up to this long travel in the launch parameters (no copy in the
// stream ahead of the kernels); longer ones are copied to the device.
constexpr int kInlineTiles = 256;
struct TileParams {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    // Row matrices of the adapters' pages: row a_row + j holds page j of A_k (its
    // first d_in elements are read), row b_row + j page j of B_k (first d_out).
    // Either the pools themselves (every adapter's pages consecutive) or a dense
    // copy made for the call, rank-padded with zero rows.
    const uint16_t *a_rows;
    int64_t a_ld;             // row stride, elements
    int64_t a_nrows;          // rows (tensor-map extent)
    const uint16_t *b_rows;
    int64_t b_ld;
    int64_t b_nrows;
    const TileItem *items;    // device copy of the list, unless items_inline
    float *vparts;            // fused: [n_items][ksplit] partial V slots
    float *v;                 // shrink / expand only: fp32 rows [n, ldv]
    int64_t ldv;
    unsigned *status;
    int max_rank;
    int n_rows;               // rows of x / y (tensor-map extent)
    int d_in;
    int d_out;
    int n_items;
    int vmode;                // 0: V tiles (fused), 1: fp32 v rows
    int max_tile_rank;        // largest rank among the items (sizes shared memory)
    int ksplit;               // fused: K-split of the shrink (1..8)
    int early_x;              // shrink: x and A loads and MMAs before the dependency wait
    int early_tiles;          // expand right after its shrink: y and B loads before it
    int wide_ring;            // shrink: one CTA per SM, a ring of 200 KB instead of 100 KB
    int items_inline;         // 1: the list is inl[0 .. n_items)
    TileItem inl[kInlineTiles];
};
#ifdef __CUDACC__
__device__ __forceinline__ TileItem tile_item(const TileParams &p, int i)
{
    return p.items_inline ? p.inl[i] : p.items[i];
}
#endif
// Fixed scratch of lora_fused_noalloc (noalloc.cu): device addresses of the
// file-scope arrays on one device, looked up once per device.
constexpr int kNoAllocSlots = 64;
constexpr size_t kNoAllocDenseBytes = size_t(8) << 20;
struct NoAllocScratch {
    float *vparts;            // kNoAllocSlots slots of kVPartBytes
    uint16_t *dense;          // kNoAllocDenseBytes of dense adapter rows
};
static_assert(kNoAllocSlots <= kInlineTiles, "a no-alloc tile list travels in the parameters");
// Looks the addresses up on the first call for `device` (with it current) or when
// `refresh` is set, and caches them; loading the module that holds the arrays is
// what commits their memory.
cudaError_t noalloc_scratch(int device, bool refresh, NoAllocScratch *out);

// Dense adapter rows (dense.cu): for slot s and j < rp, row s*rp + j of dst gets
// the first `width` elements of page j of the slot's adapter, zeros for j >= rank.
constexpr int kStageSlots = 128;           // slots per launch
struct StageSide {
    const uint16_t *pool;
    int64_t pw;
    const int32_t *pages;     // device page table [n_adapters * max_rank]
    uint16_t *dst;            // rows of dst_ld elements; slot s at row s * rp
    int width;                // elements copied per row (<= pw, <= dst_ld)
    int64_t dst_ld;
};
struct StageArgs {
    StageSide side[2];        // A, B (side with dst == nullptr skipped)
    int max_rank;
    int rp;
    int n_slots;              // entries of this launch
    int early;                // copy before waiting for the previous kernel (dense.cu)
    int32_t adapter[kStageSlots];
    int32_t rank[kStageSlots];
    int32_t dst_slot[kStageSlots];   // destination slot of entry s
};
cudaError_t launch_stage_rows(const StageArgs &a, cudaStream_t stream);

// Adapter page-in (pagein.cu): rows j < rank of `host` (device-mapped page-locked
// host memory, `width` elements each) to pool page page[j], for A and for B.
constexpr int kPageInMaxRank = 128;
struct PageInSide {
    const uint16_t *host;     // device address of the host rows [rank][width]
    uint16_t *pool;
    int64_t pw;               // pool page width, elements
    int width;                // elements copied per page (<= pw, multiple of 8)
    int32_t page[kPageInMaxRank];
};
struct PageInArgs {
    PageInSide side[2];       // A, B
    int rank;
};
cudaError_t launch_page_in(const PageInArgs &a, cudaStream_t stream);

// Device-side plan (devplan.cu) of a row-gather call over device-resident ids.
constexpr int kDevPlanMaxAdapters = 16384;
struct DevPlanArgs {
    const int32_t *ids;       // [n], device
    int n;
    const int32_t *rank;      // table's device copies
    const float *scale;
    const uint8_t *ok;        // 1: the table can serve the adapter
    int n_adapters;
    int rows_per_item;
    RowItem *items;           // [n] out
    int32_t *perm;            // [n] out
    int32_t *n_items;         // out
    unsigned *status;
};
size_t dev_plan_smem_bytes(int n_adapters);
cudaError_t launch_wait_selftest(unsigned *status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_plan_dev(const DevPlanArgs &a, cudaStream_t stream);

// Base projection with the adapter term (proj_tc.cu): y = bf16(x W + s_k (x A_k) B_k).
// The adapter terms of a 256-row block m are chunks[chunk_off[m] .. chunk_off[m + 1]):
// one per adapter with rows in the block and 64 columns of its padded rank.
struct ProjChunk {
    int32_t adapter;
    int32_t b_row;            // the B row matrix's row of the chunk's first rank index
    int32_t rank;
    float scale;
    int32_t m;                // the block
    int32_t c;                // the chunk's first rank index (a multiple of 64)
    int32_t kc;               // its K: min(64, padded rank - c), a multiple of 16
    int32_t pad;
};
static_assert(sizeof(ProjChunk) == 32, "ProjChunk is two 16-byte loads");
struct ProjParams {
    const uint16_t *x;
    int64_t ldx;
    const uint16_t *W;
    int64_t ldw;
    uint16_t *y;
    int64_t ldy;
    const float *v;           // the shrink's fp32 rows [n, ldv] (ldv a multiple of 4)
    int64_t ldv;
    const int32_t *ids;       // device copy of the call's ids [n]
    const int32_t *chunk_off; // [n_mblk + 1]
    const ProjChunk *chunks;
    uint16_t *a_prep;         // [n_chunks * 2 * 256, 64] bf16: per chunk hi, then lo
    const uint16_t *b_rows;   // B row matrix (pages as consecutive rows, rank-padded)
    int64_t b_ld;
    int64_t b_nrows;
    unsigned *status;
    int n;
    int d_in;
    int d_out;
    int n_mblk;               // 256-row blocks (one per CTA pair)
    int n_nblk;               // 256-column blocks
    int n_chunks;
    int early;                // launched right after k_proj_prep: x and W loads go ahead of the wait
};
cudaError_t launch_proj_prep(const ProjParams &p, cudaStream_t stream);
cudaError_t launch_proj_tc(const ProjParams &p, cudaStream_t stream);
int proj_block_rows();
int proj_block_cols();
int proj_chunk_cols();

// Offline search (fill.cu): n bf16 values uniform in [-scale, scale) from a hash of
// (seed, index).
cudaError_t launch_fill_bf16(uint16_t *dst, uint64_t n, uint64_t seed, float scale,
                             cudaStream_t stream);

cudaError_t launch_shrink_tc(const TileParams &p, cudaStream_t stream);
cudaError_t launch_expand_tc(const TileParams &p, cudaStream_t stream);
bool tile_tc_supported(int d_in, int d_out, int rank);

// Tensor-core merge (merge_tc.cu).
struct MergeParams {
    uint16_t *W;
    int64_t ldw;
    const uint16_t *a_pool;
    int64_t a_pw;
    const uint16_t *b_pool;
    int64_t b_pw;
    int64_t b_n_pages;        // rows of the B pool (tensor-map extent of the page gather)
    const int32_t *a_pages;   // host-resolved page ids of this adapter, device copy
    const int32_t *b_pages;
    // Row matrices as in TileParams (tensor-core merge), with this adapter's rows.
    const uint16_t *a_rows;
    int64_t a_ld, a_nrows;
    const uint16_t *b_rows;
    int64_t b_ld, b_nrows;
    int32_t a_row, b_row;
    unsigned *status;
    int d_in;
    int d_out;
    int rank;
    float scale;              // signed
    int n_split;              // column groups per 128-row block
};

}  // namespace lora
