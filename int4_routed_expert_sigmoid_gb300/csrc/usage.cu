// usage.cu -- Learn, persisted: the per-expert hit counters of every layer
// saved to a file and loaded back, and the most used experts of a layer (the
// set an expert tier pins in device memory).
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction" (the Learn stage counts, per expert, how
// often the router chose it; the experts chosen most are kept in a cache
// whose contents are saved to a usage file between runs) and "Failure, Corruption, and Restart Behavior" (on restart the usage
// file decides which experts are pinned; the engine does not check that the
// file belongs to the model it runs, so a changed model can be given a wrong
// hot set).  Here the file carries a model id, its shape and a checksum, and a
// file written for another model or shape is refused (MOE_ERR_STALE) rather
// than used.
//
// File layout (all integers little-endian):
//   bytes  0..7    magic "MOEUSAGE"
//   bytes  8..11   version (1)
//   bytes 12..15   layers
//   bytes 16..19   E (experts per layer)
//   bytes 20..23   zero
//   bytes 24..31   model id (chosen by the caller, e.g. a hash of the weights)
//   then layers * E uint64 counts, layer-major
//   then a uint64 FNV-1a hash of every byte before it.
// A file is written to "<path>.tmp" and renamed over <path>, so a reader never
// sees half a file.  Host code only.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "moe_internal.h"

namespace {

constexpr char kMagic[8] = {'M', 'O', 'E', 'U', 'S', 'A', 'G', 'E'};
constexpr uint32_t kVersion = 1;
constexpr size_t kHeader = 32;

uint64_t fnv1a(const uint8_t *p, size_t n)
{
    uint64_t h = 14695981039346656037ull;
    for (size_t i = 0; i < n; i++) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

void put_u32(uint8_t *p, uint32_t v)
{
    for (int i = 0; i < 4; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}

void put_u64(uint8_t *p, uint64_t v)
{
    for (int i = 0; i < 8; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}

uint32_t get_u32(const uint8_t *p)
{
    uint32_t v = 0;
    for (int i = 0; i < 4; i++)
        v |= (uint32_t)p[i] << (8 * i);
    return v;
}

uint64_t get_u64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 0; i < 8; i++)
        v |= (uint64_t)p[i] << (8 * i);
    return v;
}

}  // namespace

extern "C" {

int moe_usage_save(const char *path, const uint64_t *hits, int layers, int E, uint64_t model_id)
{
    if (path == nullptr || hits == nullptr || layers < 1 || E < 1 || (size_t)layers * E > (size_t)1 << 26)
        return MOE_ERR_INVALID_ARG;
    const size_t n = (size_t)layers * E;
    std::vector<uint8_t> buf(kHeader + 8 * n + 8);
    std::memcpy(buf.data(), kMagic, 8);
    put_u32(&buf[8], kVersion);
    put_u32(&buf[12], (uint32_t)layers);
    put_u32(&buf[16], (uint32_t)E);
    put_u32(&buf[20], 0);
    put_u64(&buf[24], model_id);
    for (size_t i = 0; i < n; i++)
        put_u64(&buf[kHeader + 8 * i], hits[i]);
    put_u64(&buf[kHeader + 8 * n], fnv1a(buf.data(), kHeader + 8 * n));
    const std::string tmp = std::string(path) + ".tmp";
    FILE *fp = std::fopen(tmp.c_str(), "wb");
    if (fp == nullptr)
        return MOE_ERR_INVALID_ARG;
    const bool ok = std::fwrite(buf.data(), 1, buf.size(), fp) == buf.size();
    if (std::fclose(fp) != 0 || !ok) {
        std::remove(tmp.c_str());
        return MOE_ERR_INVALID_ARG;
    }
    if (std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

int moe_usage_load(const char *path, uint64_t *hits, int layers, int E, uint64_t model_id)
{
    if (path == nullptr || hits == nullptr || layers < 1 || E < 1 || (size_t)layers * E > (size_t)1 << 26)
        return MOE_ERR_INVALID_ARG;
    FILE *fp = std::fopen(path, "rb");
    if (fp == nullptr)
        return MOE_ERR_INVALID_ARG;
    std::vector<uint8_t> buf;
    uint8_t chunk[1 << 16];
    size_t got;
    while ((got = std::fread(chunk, 1, sizeof(chunk), fp)) > 0) {
        buf.insert(buf.end(), chunk, chunk + got);
        if (buf.size() > kHeader + 8 * ((size_t)1 << 26) + 8)
            break;
    }
    std::fclose(fp);
    if (buf.size() < kHeader + 8 || std::memcmp(buf.data(), kMagic, 8) != 0)
        return MOE_ERR_INVALID_ARG;   // not a usage file
    const uint32_t ver = get_u32(&buf[8]), fl = get_u32(&buf[12]), fe = get_u32(&buf[16]);
    const size_t n = (size_t)fl * fe;
    if (ver != kVersion || get_u32(&buf[20]) != 0 || n > ((size_t)1 << 26) || buf.size() != kHeader + 8 * n + 8)
        return MOE_ERR_INVALID_ARG;   // another version, or cut short / padded
    if (get_u64(&buf[kHeader + 8 * n]) != fnv1a(buf.data(), kHeader + 8 * n))
        return MOE_ERR_INVALID_ARG;   // corrupted
    if (get_u64(&buf[24]) != model_id || (int)fl != layers || (int)fe != E)
        return MOE_ERR_STALE;         // a sound file of another model or shape: not used
    for (size_t i = 0; i < n; i++)
        hits[i] = get_u64(&buf[kHeader + 8 * i]);
    return MOE_OK;
}

int moe_usage_top(const uint64_t *hits, int E, int n, int32_t *experts)
{
    if (hits == nullptr || experts == nullptr || E < 1 || n < 0 || n > E)
        return MOE_ERR_INVALID_ARG;
    // selection by repeated maximum: count descending, equal counts -> lower id first
    std::vector<uint8_t> taken(E, 0);
    for (int j = 0; j < n; j++) {
        int best = -1;
        for (int e = 0; e < E; e++) {
            if (taken[e])
                continue;
            if (best < 0 || hits[e] > hits[best])
                best = e;
        }
        taken[best] = 1;
        experts[j] = best;
    }
    return MOE_OK;
}

}  // extern "C"
