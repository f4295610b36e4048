// Shape -> launch-configuration table (VaLoRA blog, section 4.3.2: the best tiling
// for each input shape is found offline, kept in a hash table and looked up at run
// time).  Keys bucket the row count to the next power of two; row-gather keys also
// bucket the number of distinct adapters (one segment per adapter), which decides
// how many rows a work item can hold.
#pragma once
#include <array>
#include <cstdint>
#include <string>
#include <unordered_map>

namespace lora {

enum Kind : int { kKindRowsFused = 0, kKindShrink = 1, kKindExpand = 2, kKindTileFused = 3,
                  kKindMerge = 4 };

struct TileKey {
    int kind;
    int64_t m_bucket;
    int64_t s_bucket;         // row-gather kinds: distinct adapters, bucketed; else 0
    int d_in, d_out, rank;
    bool operator==(const TileKey &o) const
    {
        return kind == o.kind && m_bucket == o.m_bucket && s_bucket == o.s_bucket &&
               d_in == o.d_in && d_out == o.d_out && rank == o.rank;
    }
};

struct TileKeyHash {
    size_t operator()(const TileKey &k) const
    {
        uint64_t h = 1469598103934665603ull;
        const int64_t parts[6] = {k.kind, k.m_bucket, k.s_bucket, k.d_in, k.d_out, k.rank};
        for (int64_t p : parts) {
            h ^= uint64_t(p);
            h *= 1099511628211ull;
        }
        return size_t(h);
    }
};

using TileCfg = std::array<int, 4>;

struct TileTable {
    std::unordered_map<TileKey, TileCfg, TileKeyHash> map;
    bool lookup(const TileKey &k, TileCfg &out) const
    {
        auto it = map.find(k);
        if (it == map.end())
            return false;
        out = it->second;
        return true;
    }
    void put(const TileKey &k, const TileCfg &c)
    {
        map[k] = c;
        ++gen;
    }
    uint64_t gen = 0;                         // bumped by every change (put, load)
    int load(const std::string &path);        // LORA_OK / LORA_E_IO / LORA_E_INVAL
    int save(const std::string &path) const;
};

inline int64_t pow2_bucket(int64_t m)
{
    int64_t b = 1;
    while (b < m)
        b <<= 1;
    return b;
}

}  // namespace lora
