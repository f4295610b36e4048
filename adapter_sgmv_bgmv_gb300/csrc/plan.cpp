// Host plan (grouping step).  Punica groups the requests of a batch by adapter
// identity ("BEE-30060 Multi-LoRA serving", Background); LoRazor sizes the LoRA
// launch by the rows whose adapter is still live (LoRazor page, active-row-aware
// kernels).  Here: a stable counting sort of the active rows by adapter id, then
// work items that cover exactly the active rows.
#include "plan.h"

#include <algorithm>

#include "../../include/lora.h"

namespace lora {

// count and seen are indexed by adapter + 1: slot 0 takes the released rows (and,
// until the check after the loop, ids out of range), so the counting loop has no
// data-dependent branch (half-released decode batches would mispredict on every row).
void plan_reserve(Plan &pl, int n_adapters)
{
    const size_t slots = size_t(std::max(n_adapters, 0)) + 1;
    if (pl.count.size() < slots)
        pl.count.resize(slots, 0);
    if (pl.cursor.size() < slots)
        pl.cursor.resize(slots, 0);
    if (pl.seen.size() < (slots + 63) / 64)
        pl.seen.resize((slots + 63) / 64, 0);
}

// Batches up to this long are grouped row by row without data-dependent branches
// (decode: short runs, many released rows); longer ones run by run (prefill: a
// request's rows sit together, so a run costs one count update and one block of
// consecutive row indices instead of a read-modify-write per row).
constexpr int64_t kRowByRowMax = 1024;

int plan_group(Plan &pl, const int32_t *ids, int64_t n, int n_adapters)
{
    pl.seg_offsets.clear();
    pl.seg_adapter.clear();
    pl.max_seg_len = 0;
    plan_reserve(pl, n_adapters);
    pl.active.resize(size_t(n));
    int32_t *__restrict active = pl.active.data();
    int32_t *__restrict count = pl.count.data();
    uint64_t *__restrict seen = pl.seen.data();
    const size_t words = (size_t(n_adapters) + 1 + 63) / 64;
    const bool by_row = n <= kRowByRowMax;
    // Count the rows of each adapter, mark the adapters in use and list the active rows.
    int64_t n_act = 0;
    bool bad = false;
    if (by_row) {
        // every row is written, the length advances only for an active one
        for (int64_t i = 0; i < n; ++i) {
            const int32_t k = ids[i];
            const bool in_range = k >= -1 && k < n_adapters;
            bad |= !in_range;
            const int32_t slot = in_range ? k + 1 : 0;
            active[n_act] = int32_t(i);
            n_act += slot > 0;
            count[slot] += 1;
            seen[slot >> 6] |= uint64_t(1) << (slot & 63);
        }
    } else {
        pl.runs.clear();
        for (int64_t i = 0; i < n;) {
            const int32_t k = ids[i];
            int64_t j = i + 1;
            for (; j + 16 <= n; j += 16) {   // whole blocks of 16 first (vector compares)
                int32_t diff = 0;
                for (int u = 0; u < 16; ++u)
                    diff |= ids[j + u] ^ k;
                if (diff != 0)
                    break;
            }
            while (j < n && ids[j] == k)
                ++j;
            if (k < -1 || k >= n_adapters) {
                bad = true;
                break;
            }
            if (k >= 0) {
                const int32_t len = int32_t(j - i), row0 = int32_t(i);
                for (int32_t t = 0; t < len; ++t)
                    active[n_act + t] = row0 + t;
                n_act += len;
                count[k + 1] += len;
                seen[(k + 1) >> 6] |= uint64_t(1) << ((k + 1) & 63);
                pl.runs.push_back(Plan::Run{row0, len, k + 1});
            }
            i = j;
        }
    }
    if (bad) {   // leave the scratch all zero
        if (by_row) {
            for (int64_t i = 0; i < n; ++i) {
                const int32_t k = ids[i];
                count[(k >= -1 && k < n_adapters) ? k + 1 : 0] = 0;
            }
        } else {
            for (const Plan::Run &r : pl.runs)
                count[r.slot] = 0;
        }
        std::fill(seen, seen + words, uint64_t(0));
        pl.active.clear();
        pl.perm.clear();
        return LORA_E_ADAPTER;
    }
    pl.active.resize(size_t(n_act));
    count[0] = 0;
    seen[0] &= ~uint64_t(1);
    // Segments in ascending adapter order: the set bits, word by word.
    int32_t run = 0;
    for (size_t w = 0; w < words; ++w) {
        uint64_t m = seen[w];
        if (m == 0)
            continue;
        seen[w] = 0;
        while (m != 0) {
            const int32_t slot = int32_t(w * 64 + size_t(__builtin_ctzll(m)));
            m &= m - 1;
            const int32_t c = count[slot];
            count[slot] = 0;
            pl.cursor[size_t(slot)] = run;
            pl.seg_offsets.push_back(run);
            pl.seg_adapter.push_back(slot - 1);
            pl.max_seg_len = std::max(pl.max_seg_len, c);
            run += c;
        }
    }
    pl.seg_offsets.push_back(run);
    // Stable placement: rows in ascending order, each at its adapter's cursor.
    pl.perm.resize(size_t(n_act));
    int32_t *__restrict cursor = pl.cursor.data();
    int32_t *__restrict perm = pl.perm.data();
    if (by_row) {
        for (int64_t q = 0; q < n_act; ++q) {
            const int32_t row = active[q];
            perm[cursor[ids[row] + 1]++] = row;
        }
    } else {
        for (const Plan::Run &r : pl.runs) {
            const int32_t c = cursor[r.slot];
            for (int32_t t = 0; t < r.len; ++t)
                perm[c + t] = r.row0 + t;
            cursor[r.slot] = c + r.len;
        }
    }
    return LORA_OK;
}

// Row items only (no run can reach a tile): one pass over the active rows, an item
// starting at every rows_per_item-th row of a segment.  Written without
// data-dependent branches, since decode segments of one to a few rows would make a
// per-segment loop mispredict on almost every segment.
static void plan_row_items_only(Plan &pl, const int32_t *rank, const float *scale,
                                int rows_per_item)
{
    const int32_t n_act = int32_t(pl.perm.size());
    pl.row_perm.assign(pl.perm.begin(), pl.perm.end());
    pl.row_items.resize(size_t(n_act));
    RowItem *items = pl.row_items.data();
    const int32_t *offs = pl.seg_offsets.data();
    const int32_t *seg_adapter = pl.seg_adapter.data();
    int32_t s = 0, end = offs[1], cnt = 0, n_items = 0, max_rows = 0;
    for (int32_t q = 0; q < n_act; ++q) {
        const bool next = q == end;               // first row of the next segment
        s += next ? 1 : 0;
        end = next ? offs[s + 1] : end;
        cnt = next ? 0 : cnt;
        const int32_t k = seg_adapter[s];
        const int32_t m = std::min(rows_per_item, end - q);
        items[n_items] = RowItem{k, q, int16_t(m), int16_t(rank[k]), scale[k]};
        n_items += cnt == 0 ? 1 : 0;
        max_rows = std::max(max_rows, cnt == 0 ? m : 0);
        cnt = cnt + 1 == rows_per_item ? 0 : cnt + 1;
    }
    pl.row_items.resize(size_t(n_items));
    int32_t max_rank = 0;
    for (const int32_t k : pl.seg_adapter)
        max_rank = std::max(max_rank, rank[k]);
    pl.max_rank = pl.row_max_rank = max_rank;
    pl.row_max_rows = max_rows;
    pl.row_active = n_act;
}

// End of the maximal run of consecutive row indices that starts at perm[q], within a
// segment [.., e).  The segment's rows ascend, so [q, t) is one run exactly when
// perm[t - 1] - perm[q] == t - 1 - q, a property that holds up to the run's end and
// fails after it: found by doubling the step, then bisecting (a prefill request's
// thousand rows take about twenty probes, not a thousand).
static int32_t consecutive_end(const int32_t *perm, int32_t q, int32_t e)
{
    auto whole = [&](int32_t t) { return perm[t - 1] - perm[q] == t - 1 - q; };
    int32_t lo = q + 1, step = 1;   // [q, lo) is known to be one run
    while (lo < e) {
        const int32_t hi = std::min(e, lo + step);
        if (!whole(hi)) {
            int32_t a = lo, b = hi - 1;   // the end lies in [lo, hi - 1]
            while (a < b) {
                const int32_t m = a + (b - a + 1) / 2;
                if (whole(m))
                    a = m;
                else
                    b = m - 1;
            }
            return a;
        }
        lo = hi;
        step *= 2;
    }
    return e;
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
    if (nseg > 0 && (tile_min_run <= 0 || pl.max_seg_len < tile_min_run)) {
        plan_row_items_only(pl, rank, scale, rows_per_item);
        return;
    }
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
        if (tile_min_run > 0 && e - b >= tile_min_run) {   // else no run can reach a tile
            int32_t q = b;
            while (q < e) {
                const int32_t t = consecutive_end(pl.perm.data(), q, e);
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
