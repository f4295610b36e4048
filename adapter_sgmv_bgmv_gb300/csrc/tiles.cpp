// Text form of the shape -> configuration table: one entry per line,
//   kind m_bucket d_in d_out rank cfg0 cfg1 cfg2 cfg3
// '#' starts a comment.
#include "tiles.h"

#include <cstdio>
#include <fstream>
#include <sstream>

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
        TileKey k{};
        TileCfg c{};
        if (!(ss >> k.kind))
            continue;   // blank line
        if (!(ss >> k.m_bucket >> k.d_in >> k.d_out >> k.rank >> c[0] >> c[1] >> c[2] >> c[3]))
            return LORA_E_INVAL;
        if (k.kind < 0 || k.kind > 4 || k.m_bucket < 0)
            return LORA_E_INVAL;
        fresh[k] = c;
    }
    for (auto &kv : fresh)
        map[kv.first] = kv.second;
    return LORA_OK;
}

int TileTable::save(const std::string &path) const
{
    std::ofstream out(path);
    if (!out)
        return LORA_E_IO;
    out << "# kind m_bucket d_in d_out rank cfg0 cfg1 cfg2 cfg3\n";
    for (const auto &kv : map) {
        const TileKey &k = kv.first;
        const TileCfg &c = kv.second;
        out << k.kind << ' ' << k.m_bucket << ' ' << k.d_in << ' ' << k.d_out << ' ' << k.rank
            << ' ' << c[0] << ' ' << c[1] << ' ' << c[2] << ' ' << c[3] << '\n';
    }
    return out ? LORA_OK : LORA_E_IO;
}

}  // namespace lora
