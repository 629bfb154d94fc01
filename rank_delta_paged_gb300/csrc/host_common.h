// Host-only helpers of libslora.so (no CUDA types).
#pragma once

#include <cstdint>
#include <map>
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

}  // namespace slora
