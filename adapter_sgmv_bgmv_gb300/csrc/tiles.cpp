// Text form of the shape -> configuration table: one entry per line,
//   kind m_bucket s_bucket d_in d_out rank cfg0 cfg1 cfg2 cfg3
// '#' starts a comment.  Lines without s_bucket (nine fields) read it as 0.
#include "tiles.h"

#include <cstdio>
#include <fstream>
#include <sstream>
#include <vector>

#include "../../include/lora.h"

namespace lora {

int TileTable::load(const std::string &path)
{
    std::ifstream in(path);
    if (!in)
        return LORA_E_IO;
    std::string line;
    std::unordered_map<TileKey, TileCfg, TileKeyHash> fresh;
    while (std::getline(in, line)) {
        const size_t hash = line.find('#');
        if (hash != std::string::npos)
            line.resize(hash);
        std::istringstream ss(line);
        std::vector<int64_t> f;
        int64_t v = 0;
        while (ss >> v)
            f.push_back(v);
        if (!ss.eof())
            return LORA_E_INVAL;   // a field that is not an integer
        if (f.empty())
            continue;              // blank line
        if (f.size() == 9)
            f.insert(f.begin() + 2, 0);
        if (f.size() != 10)
            return LORA_E_INVAL;
        TileKey k{int(f[0]), f[1], f[2], int(f[3]), int(f[4]), int(f[5])};
        TileCfg c{int(f[6]), int(f[7]), int(f[8]), int(f[9])};
        if (k.kind < 0 || k.kind > 4 || k.m_bucket < 0 || k.s_bucket < 0)
            return LORA_E_INVAL;
        fresh[k] = c;
    }
    for (auto &kv : fresh)
        map[kv.first] = kv.second;
    ++gen;
    return LORA_OK;
}

int TileTable::save(const std::string &path) const
{
    std::ofstream out(path);
    if (!out)
        return LORA_E_IO;
    out << "# kind m_bucket s_bucket d_in d_out rank cfg0 cfg1 cfg2 cfg3\n";
    for (const auto &kv : map) {
        const TileKey &k = kv.first;
        const TileCfg &c = kv.second;
        out << k.kind << ' ' << k.m_bucket << ' ' << k.s_bucket << ' ' << k.d_in << ' ' << k.d_out
            << ' ' << k.rank
            << ' ' << c[0] << ' ' << c[1] << ' ' << c[2] << ' ' << c[3] << '\n';
    }
    return out ? LORA_OK : LORA_E_IO;
}

}  // namespace lora
