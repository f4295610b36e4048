// Host plan (grouping step).  Punica groups the requests of a batch by adapter
// identity ("BEE-30060 Multi-LoRA serving", Background); LoRazor sizes the LoRA
// launch by the rows whose adapter is still live (LoRazor page, active-row-aware
// kernels).  Here: a stable counting sort of the active rows by adapter id, then
// work items that cover exactly the active rows.
#include "plan.h"

#include <algorithm>

#include "../../include/lora.h"

namespace lora {

int plan_group(Plan &pl, const int32_t *ids, int64_t n, int n_adapters)
{
    pl.active.clear();
    pl.perm.clear();
    pl.seg_offsets.clear();
    pl.seg_adapter.clear();
    pl.max_seg_len = 0;
    pl.count.assign(size_t(n_adapters), 0);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t k = ids[i];
        if (k < -1 || k >= n_adapters)
            return LORA_E_ADAPTER;
        if (k >= 0) {
            pl.active.push_back(int32_t(i));
            pl.count[size_t(k)] += 1;
        }
    }
    pl.cursor.resize(size_t(n_adapters));
    int32_t run = 0;
    for (int k = 0; k < n_adapters; ++k) {
        pl.cursor[size_t(k)] = run;
        const int32_t c = pl.count[size_t(k)];
        if (c > 0) {
            pl.seg_offsets.push_back(run);
            pl.seg_adapter.push_back(k);
            pl.max_seg_len = std::max(pl.max_seg_len, c);
        }
        run += c;
    }
    pl.seg_offsets.push_back(run);
    pl.perm.resize(pl.active.size());
    for (int32_t row : pl.active)
        pl.perm[size_t(pl.cursor[size_t(ids[row])]++)] = row;
    return LORA_OK;
}

void plan_items(Plan &pl, const int32_t *rank, const float *scale, int rows_per_item,
                int tile_min_run)
{
    pl.row_items.clear();
    pl.row_perm.clear();
    pl.tile_items.clear();
    pl.max_rank = pl.tile_max_rank = pl.row_max_rank = pl.row_max_rows = 0;
    pl.row_active = pl.tile_active = 0;
    const size_t nseg = pl.seg_adapter.size();
    for (size_t s = 0; s < nseg; ++s) {
        const int32_t k = pl.seg_adapter[s];
        const int32_t r = rank[k];
        pl.max_rank = std::max(pl.max_rank, r);
        const int32_t b = pl.seg_offsets[s], e = pl.seg_offsets[s + 1];
        // Pending rows of this segment not yet given to a tile: [pend, q).
        int32_t pend = b;
        auto flush_rows = [&](int32_t from, int32_t to) {
            for (int32_t p = from; p < to; p += rows_per_item) {
                const int32_t m = std::min(rows_per_item, to - p);
                const int32_t q0 = int32_t(pl.row_perm.size());
                for (int32_t u = 0; u < m; ++u)
                    pl.row_perm.push_back(pl.perm[size_t(p + u)]);
                pl.row_items.push_back(RowItem{k, q0, int16_t(m), int16_t(r), scale[k]});
                pl.row_max_rows = std::max(pl.row_max_rows, m);
                pl.row_active += m;
            }
            if (to > from)
                pl.row_max_rank = std::max(pl.row_max_rank, r);
        };
        if (tile_min_run > 0) {
            int32_t q = b;
            while (q < e) {
                // maximal run of consecutive row indices starting at perm[q]
                int32_t t = q + 1;
                while (t < e && pl.perm[size_t(t)] == pl.perm[size_t(t - 1)] + 1)
                    ++t;
                if (t - q >= tile_min_run) {
                    flush_rows(pend, q);
                    for (int32_t p = q; p < t; p += 128) {
                        const int32_t m = std::min(128, t - p);
                        pl.tile_items.push_back(
                            TileItem{k, pl.perm[size_t(p)], int16_t(m), int16_t(r), scale[k], -1, -1, {0, 0}});
                        pl.tile_active += m;
                    }
                    pl.tile_max_rank = std::max(pl.tile_max_rank, r);
                    pend = t;
                }
                q = t;
            }
        }
        flush_rows(pend, e);
    }
}

}  // namespace lora
