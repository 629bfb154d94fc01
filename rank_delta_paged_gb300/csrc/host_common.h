// Host-only helpers of libslora.so (no CUDA types).
#pragma once

#include <cstdint>
#include <map>
#include <set>
#include <unordered_map>
#include <unordered_set>
#include <string>
#include <vector>

#include "slora.h"

namespace slora {

extern thread_local std::string g_last_error;
slora_status fail(slora_status s, const char *fmt, ...);
uint64_t splitmix64(uint64_t &state);

// Free list of pool slots.  allocated[p]: 0 free, 1 in use.
struct PageAlloc {
    int64_t num_pages = 0;
    std::vector<int32_t> free_stack;
    std::vector<uint8_t> allocated;
    void init(int64_t n, uint64_t seed);
    slora_status alloc(int64_t n, int32_t *out);
    slora_status release(int64_t n, const int32_t *pages);
    int64_t num_free() const { return (int64_t)free_stack.size(); }
};

// First-fit allocator of contiguous ranges (the device page-table arena).
struct RangeAlloc {
    std::map<int64_t, int64_t> free_ranges;  // start -> length
    void init(int64_t capacity);
    int64_t alloc(int64_t n);                 // -1 if no range fits
    void release(int64_t start, int64_t n);
};

// Recency index of resident adapters for eviction under pool pressure: adapters that are
// not pinned are kept in order of last use; the victims are taken from the least recently
// used end.  Pinned adapters (in use by a batch) are never victims.
struct LruIndex {
    struct Ent {
        uint64_t last = 0;
        int32_t pins = 0;
    };
    uint64_t clock = 0;
    std::unordered_map<int32_t, Ent> ents;                // present adapters
    std::set<std::pair<uint64_t, int32_t>> unpinned;      // (last use, id) of present, unpinned adapters

    bool present(int32_t id) const { return ents.count(id) != 0; }
    int32_t pins(int32_t id) const;
    void insert(int32_t id);   // present, unpinned, most recently used (no-op if present)
    void remove(int32_t id);   // no-op if absent
    void touch(int32_t id);    // most recently used; present ids only
    void pin(int32_t id);      // present ids only
    bool unpin(int32_t id);    // false if the id was not pinned
    // Least recently used first: unpinned present ids not in `exclude` until `enough`
    // returns true for the list so far (it is called after each id is added).  Returns
    // false (and an incomplete list) if the unpinned ids run out first.
    template <class Enough>
    bool victims(const std::unordered_set<int32_t> &exclude, Enough enough, std::vector<int32_t> *out) const
    {
        out->clear();
        if (enough(*out))
            return true;
        for (const auto &e : unpinned) {
            if (exclude.count(e.second))
                continue;
            out->push_back(e.second);
            if (enough(*out))
                return true;
        }
        return false;
    }
};

}  // namespace slora
