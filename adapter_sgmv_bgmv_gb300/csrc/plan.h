// Host-side plan: which rows take part, how they group by adapter, and the work
// items of each kernel.  O(n + n_adapters) per call, no device work.
#pragma once
#include <cstdint>
#include <vector>

#include "internal.h"

namespace lora {

struct Plan {
    std::vector<int32_t> active;       // ascending rows with id >= 0
    std::vector<int32_t> perm;         // active rows stably sorted by adapter id
    std::vector<int32_t> seg_offsets;  // [n_seg + 1]
    std::vector<int32_t> seg_adapter;  // [n_seg]
    std::vector<RowItem> row_items;    // p0 indexes row_perm
    std::vector<int32_t> row_perm;     // the perm entries of the row items only
    std::vector<TileItem> tile_items;
    std::vector<int32_t> slot_adapter; // the tile items' adapters, in order of first tile
    std::vector<int32_t> slot_a_base;  // first row of each slot in the A / B row matrices
    std::vector<int32_t> slot_b_base;
    std::vector<int32_t> count;        // scratch, [>= n_adapters], all zero between calls
    std::vector<int32_t> cursor;       // scratch, [>= n_adapters]
    std::vector<uint64_t> seen;        // scratch bitmap of the adapters in use, all zero
                                       // between calls
    struct Run {
        int32_t row0, len, slot;       // rows [row0, row0 + len) all of adapter slot - 1
    };
    std::vector<Run> runs;             // scratch: the runs of equal active ids (long batches)
    int32_t max_seg_len = 0;
    int32_t max_rank = 0;              // largest rank referenced
    int32_t tile_max_rank = 0;
    int32_t row_max_rank = 0;
    int32_t row_max_rows = 0;
    int64_t row_active = 0;            // active rows routed to the row-gather kernel
    int64_t tile_active = 0;           // active rows routed to the tile kernel
};

// Group rows.  Returns LORA_OK or LORA_E_ADAPTER (an id outside [-1, n_adapters)).
// O(n + n_adapters / 64): only the adapters in use are visited.
int plan_group(Plan &pl, const int32_t *ids, int64_t n, int n_adapters);

// Size the per-adapter scratch for tables of up to n_adapters adapters (so that a
// call allocates nothing for it).
void plan_reserve(Plan &pl, int n_adapters);

// Cut segments into work items.  Runs of consecutive rows of at least
// `tile_min_run` rows go to 128-row tiles (tile_min_run <= 0: none do); everything
// else goes to row items of at most `rows_per_item` rows.
void plan_items(Plan &pl, const int32_t *rank, const float *scale, int rows_per_item,
                int tile_min_run);

}  // namespace lora
