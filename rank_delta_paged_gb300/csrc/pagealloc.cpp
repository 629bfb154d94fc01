// Host page allocator of the unified pool: one free list shared by adapter rows and KV
// blocks (S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "The
// mechanism": Unified Paging -- one pool allocates pages for KV blocks of varying
// length and LoRA tiles of varying rank; "What to notice when reading": adapters and KV
// share the allocator).  Needs no GPU.
#include <cstdint>
#include <cstdio>
#include <cstdarg>
#include <iterator>
#include <utility>
#include <new>
#include <string>
#include <vector>

#include "slora.h"
#include "host_common.h"

namespace slora {

thread_local std::string g_last_error;

slora_status fail(slora_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = std::string(slora_status_str(s)) + ": " + buf;
    return s;
}

uint64_t splitmix64(uint64_t &state)
{
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void PageAlloc::init(int64_t n, uint64_t seed)
{
    num_pages = n;
    free_stack.resize((size_t)n);
    allocated.assign((size_t)n, 0);
    // The stack pops from the back: fill it so that an unshuffled list hands out
    // pages 0, 1, 2, ... in order.
    for (int64_t i = 0; i < n; ++i)
        free_stack[(size_t)i] = (int32_t)(n - 1 - i);
    if (seed != 0) {
        uint64_t st = seed;
        for (int64_t i = n - 1; i > 0; --i) {
            int64_t j = (int64_t)(splitmix64(st) % (uint64_t)(i + 1));
            std::swap(free_stack[(size_t)i], free_stack[(size_t)j]);
        }
    }
}

slora_status PageAlloc::alloc(int64_t n, int32_t *out)
{
    if (n < 0 || (n > 0 && out == nullptr))
        return fail(SLORA_ERR_INVALID_ARG, "page alloc: n=%lld", (long long)n);
    if ((int64_t)free_stack.size() < n)
        return fail(SLORA_ERR_POOL_FULL, "page alloc: need %lld pages, %lld free", (long long)n,
                    (long long)free_stack.size());
    for (int64_t i = 0; i < n; ++i) {
        int32_t p = free_stack.back();
        free_stack.pop_back();
        allocated[(size_t)p] = 1;
        out[i] = p;
    }
    return SLORA_OK;
}

slora_status PageAlloc::release(int64_t n, const int32_t *pages)
{
    if (n < 0 || (n > 0 && pages == nullptr))
        return fail(SLORA_ERR_INVALID_ARG, "page free: n=%lld", (long long)n);
    // validate everything first (also catches a page listed twice)
    std::vector<int32_t> seen;
    seen.reserve((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        int32_t p = pages[i];
        const char *why = nullptr;
        if (p < 0 || p >= num_pages)
            why = "out of range";
        else if (allocated[(size_t)p] != 1)
            why = allocated[(size_t)p] == 2 ? "listed twice" : "not allocated";
        if (why) {
            for (int32_t q : seen)
                allocated[(size_t)q] = 1;  // undo the marks: nothing is returned
            return fail(SLORA_ERR_INVALID_ARG, "page free: page %d %s", p, why);
        }
        allocated[(size_t)p] = 2;  // mark while validating
        seen.push_back(p);
    }
    for (int32_t p : seen) {
        allocated[(size_t)p] = 0;
        free_stack.push_back(p);
    }
    return SLORA_OK;
}

// ---- page-table arena: first-fit ranges with coalescing -------------------------
void RangeAlloc::init(int64_t capacity)
{
    free_ranges.clear();
    if (capacity > 0)
        free_ranges[0] = capacity;
}

int64_t RangeAlloc::alloc(int64_t n)
{
    for (auto it = free_ranges.begin(); it != free_ranges.end(); ++it) {
        if (it->second >= n) {
            int64_t start = it->first;
            int64_t len = it->second;
            free_ranges.erase(it);
            if (len > n)
                free_ranges[start + n] = len - n;
            return start;
        }
    }
    return -1;
}

void RangeAlloc::release(int64_t start, int64_t n)
{
    if (n <= 0)
        return;
    auto next = free_ranges.lower_bound(start);
    if (next != free_ranges.end() && start + n == next->first) {
        n += next->second;
        next = free_ranges.erase(next);
    }
    if (next != free_ranges.begin()) {
        auto prev = std::prev(next);
        if (prev->first + prev->second == start) {
            prev->second += n;
            return;
        }
    }
    free_ranges[start] = n;
}

}  // namespace slora

using namespace slora;

struct slora_pagealloc {
    PageAlloc a;
};

extern "C" {

const char *slora_status_str(slora_status s)
{
    switch (s) {
    case SLORA_OK: return "SLORA_OK";
    case SLORA_ERR_INVALID_ARG: return "SLORA_ERR_INVALID_ARG";
    case SLORA_ERR_POOL_FULL: return "SLORA_ERR_POOL_FULL";
    case SLORA_ERR_NOT_REGISTERED: return "SLORA_ERR_NOT_REGISTERED";
    case SLORA_ERR_NOT_RESIDENT: return "SLORA_ERR_NOT_RESIDENT";
    case SLORA_ERR_ALREADY_RESIDENT: return "SLORA_ERR_ALREADY_RESIDENT";
    case SLORA_ERR_CUDA: return "SLORA_ERR_CUDA";
    case SLORA_ERR_DEVICE_CHECK: return "SLORA_ERR_DEVICE_CHECK";
    case SLORA_ERR_DEVICE_TIMEOUT: return "SLORA_ERR_DEVICE_TIMEOUT";
    case SLORA_ERR_HOST_ALLOC: return "SLORA_ERR_HOST_ALLOC";
    case SLORA_ERR_ALREADY_REGISTERED: return "SLORA_ERR_ALREADY_REGISTERED";
    case SLORA_ERR_UNSUPPORTED: return "SLORA_ERR_UNSUPPORTED";
    }
    return "SLORA_ERR_UNKNOWN";
}

const char *slora_last_error(void) { return g_last_error.c_str(); }

int32_t slora_version(void) { return 200; }

slora_status slora_pagealloc_create(int64_t num_pages, uint64_t shuffle_seed, slora_pagealloc_t *out)
{
    if (out == nullptr || num_pages < 1 || num_pages >= (int64_t)INT32_MAX)
        return fail(SLORA_ERR_INVALID_ARG, "pagealloc_create: num_pages=%lld", (long long)num_pages);
    auto *p = new (std::nothrow) slora_pagealloc;
    if (!p)
        return fail(SLORA_ERR_HOST_ALLOC, "pagealloc_create");
    try {
        p->a.init(num_pages, shuffle_seed);
    } catch (...) {
        delete p;
        return fail(SLORA_ERR_HOST_ALLOC, "pagealloc_create: %lld pages", (long long)num_pages);
    }
    *out = p;
    return SLORA_OK;
}

slora_status slora_pagealloc_destroy(slora_pagealloc_t a)
{
    delete a;
    return SLORA_OK;
}

slora_status slora_pagealloc_alloc(slora_pagealloc_t a, int64_t n, int32_t *out_pages)
{
    if (!a)
        return fail(SLORA_ERR_INVALID_ARG, "pagealloc_alloc: null allocator");
    return a->a.alloc(n, out_pages);
}

slora_status slora_pagealloc_free(slora_pagealloc_t a, int64_t n, const int32_t *pages)
{
    if (!a)
        return fail(SLORA_ERR_INVALID_ARG, "pagealloc_free: null allocator");
    return a->a.release(n, pages);
}

slora_status slora_pagealloc_num_free(slora_pagealloc_t a, int64_t *out)
{
    if (!a || !out)
        return fail(SLORA_ERR_INVALID_ARG, "pagealloc_num_free");
    *out = (int64_t)a->a.free_stack.size();
    return SLORA_OK;
}

}  // extern "C"
