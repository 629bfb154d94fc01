// The Unified Paging pool, the pinned host adapter store, adapter load / evict and the
// host side of the hot path (S-LoRA: Serving Thousands of Concurrent LoRA Adapters
// (explainer), "The mechanism" and "Algorithm / figure walkthrough"; S-LoRA:
// Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU, section 2).
#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <cstring>
#include <memory>
#include <new>
#include <unordered_set>
#include <vector>

#include <cuda_runtime.h>

#include "host_common.h"
#include "internal.h"
#include "slora.h"

using namespace slora;

namespace {

struct AdapterRec {
    bool registered = false;
    bool resident = false;
    int32_t rank = 0;
    float scaling = 0.f;
    uint16_t *store = nullptr;     // pinned [n_proj][2*rank][hidden]: A^T rows then B rows
    int32_t *pt_host = nullptr;    // pinned [n_proj][2*rank] page table
    const void *store_dev = nullptr;      // device views of the two (read by the load kernel)
    const int32_t *pt_host_dev = nullptr;
    bool pt_read_pending = false;  // a load kernel may still read pt_host (the pool's load event covers it)
    int64_t pt_off = -1;           // arena offset while resident
};

}  // namespace

struct slora_pool {
    int device = 0;
    int32_t hidden = 0;
    int64_t num_pages = 0;
    int32_t n_proj = 0;
    int32_t max_adapters = 0;
    int num_sms = 0;

    PageAlloc pages;
    RangeAlloc arena;
    int64_t arena_cap = 0;

    uint16_t *pool_dev = nullptr;
    int32_t *pt_dev = nullptr;
    DirEntry *dir_dev = nullptr;
    int32_t *status_dev = nullptr;

    cudaStream_t side = nullptr;
    cudaEvent_t release_event = nullptr;
    bool release_pending = false;
    cudaEvent_t load_event = nullptr;


    PlanScratch plan;
    std::vector<AdapterRec> adapters;
    int64_t launches = 0;  // kernels launched by this pool
    cudaEvent_t stage_event = nullptr;   // measurement hook: recorded between plan and delta
    cudaEvent_t load_start_event = nullptr;   // measurement hook: recorded before a load's work
    int32_t load_mode = SLORA_LOAD_ZERO_COPY;
    uint8_t *staging = nullptr;          // copy-engine mode: device staging ring
    int64_t staging_bytes = 0;
    int32_t max_rank = 0;  // largest registered rank (sizes the plan scratch)
    LruIndex lru;          // resident adapters by last acquire / load; pins of running batches
    int64_t n_loaded = 0, n_evicted = 0;
    uint64_t residency_gen = 0;   // bumped whenever the adapter directory changes (plans check it)
};

namespace {

#define CUDA_TRY(expr)                                                                    \
    do {                                                                                  \
        cudaError_t _e = (expr);                                                          \
        if (_e != cudaSuccess)                                                            \
            return fail(SLORA_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(_e), \
                        __FILE__, __LINE__);                                              \
    } while (0)

// The pool's device is current until the end of the enclosing scope; the caller's
// current device is restored then.
#define DEVICE_SCOPE(p)                                                                         \
    DeviceScope _dev_scope((p)->device);                                                        \
    if (_dev_scope.error() != cudaSuccess)                                                      \
        return fail(SLORA_ERR_CUDA, "cudaSetDevice(%d) failed: %s", (p)->device,                 \
                    cudaGetErrorString(_dev_scope.error()))

bool valid_id(const slora_pool *p, int32_t id) { return id >= 0 && id < p->max_adapters; }

int64_t adapter_rows(const slora_pool *p, const AdapterRec &a)
{
    return 2ll * a.rank * p->n_proj;
}

void free_pool_memory(slora_pool *p)
{
    if (p->side)
        cudaStreamSynchronize(p->side);
    cudaDeviceSynchronize();
    for (auto &a : p->adapters) {
        if (a.store) cudaFreeHost(a.store);
        if (a.pt_host) cudaFreeHost(a.pt_host);
        a = AdapterRec();
    }
    if (p->pool_dev) cudaFree(p->pool_dev);
    if (p->pt_dev) cudaFree(p->pt_dev);
    if (p->dir_dev) cudaFree(p->dir_dev);
    if (p->status_dev) cudaFree(p->status_dev);
    if (p->plan.base) cudaFree(p->plan.base);
    if (p->staging) cudaFree(p->staging);
    if (p->release_event) cudaEventDestroy(p->release_event);
    if (p->load_event) cudaEventDestroy(p->load_event);
    if (p->side) cudaStreamDestroy(p->side);
}

constexpr int64_t kDefaultStagingBytes = 256ll << 20;

// Test hook: the nth later load-path operation of one kind fails as if its CUDA call (or,
// for the arena, its allocation) had failed.  Process-wide; one injection at a time.
std::mutex g_fault_mu;
int32_t g_fault_kind = SLORA_FAULT_NONE;
int32_t g_fault_left = 0;
bool inject_fault(int32_t kind)
{
    std::lock_guard<std::mutex> lk(g_fault_mu);
    if (g_fault_kind != kind || g_fault_left <= 0)
        return false;
    if (--g_fault_left > 0)
        return false;
    g_fault_kind = SLORA_FAULT_NONE;
    return true;
}

}  // namespace

extern "C" {

slora_status slora_pool_create(int device, int32_t hidden, int64_t num_pages, int32_t n_proj,
                               int32_t max_adapters, uint64_t shuffle_seed, slora_pool_t *out)
{
    if (!out)
        return fail(SLORA_ERR_INVALID_ARG, "pool_create: out is NULL");
    *out = nullptr;
    if (hidden < 64 || hidden > 8192 || hidden % 64 != 0)
        return fail(SLORA_ERR_INVALID_ARG, "pool_create: hidden=%d (multiple of 64 in [64, 8192])", hidden);
    if (num_pages < 1 || num_pages >= (int64_t)INT32_MAX)
        return fail(SLORA_ERR_INVALID_ARG, "pool_create: num_pages=%lld", (long long)num_pages);
    if (n_proj < 1 || max_adapters < 1 || max_adapters > (1 << 24))
        return fail(SLORA_ERR_INVALID_ARG, "pool_create: n_proj=%d max_adapters=%d", n_proj, max_adapters);
    int ndev = 0;
    CUDA_TRY(cudaGetDeviceCount(&ndev));
    if (device < 0 || device >= ndev)
        return fail(SLORA_ERR_INVALID_ARG, "pool_create: device %d of %d", device, ndev);
    cudaDeviceProp prop;
    CUDA_TRY(cudaGetDeviceProperties(&prop, device));
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(SLORA_ERR_UNSUPPORTED, "pool_create: device %d is sm_%d%d; this library is built for sm_103a",
                    device, prop.major, prop.minor);

    auto *p = new (std::nothrow) slora_pool;
    if (!p)
        return fail(SLORA_ERR_HOST_ALLOC, "pool_create");
    p->device = device;
    p->hidden = hidden;
    p->num_pages = num_pages;
    p->n_proj = n_proj;
    p->max_adapters = max_adapters;
    p->num_sms = prop.multiProcessorCount;
    slora_status st = SLORA_OK;
    try {
        p->pages.init(num_pages, shuffle_seed);
        p->adapters.resize((size_t)max_adapters);
    } catch (...) {
        delete p;
        return fail(SLORA_ERR_HOST_ALLOC, "pool_create: host bookkeeping for %lld pages", (long long)num_pages);
    }
    // Each page belongs to at most one adapter, so num_pages arena entries always
    // suffice in total; twice that leaves room for fragmentation.
    p->arena_cap = 2 * num_pages;
    p->arena.init(p->arena_cap);

    auto cuda_fail = [&](cudaError_t e, const char *what) {
        st = fail(SLORA_ERR_CUDA, "pool_create: %s: %s", what, cudaGetErrorString(e));
    };
    DeviceScope dev_scope(device);
    cudaError_t e;
    if ((e = dev_scope.error()) != cudaSuccess) cuda_fail(e, "cudaSetDevice");
    else if ((e = cudaMalloc(&p->pool_dev, (size_t)num_pages * (size_t)hidden * 2)) != cudaSuccess) cuda_fail(e, "pool");
    else if ((e = cudaMalloc(&p->pt_dev, (size_t)p->arena_cap * 4)) != cudaSuccess) cuda_fail(e, "page-table arena");
    else if ((e = cudaMalloc(&p->dir_dev, (size_t)max_adapters * sizeof(DirEntry))) != cudaSuccess) cuda_fail(e, "directory");
    else if ((e = cudaMalloc(&p->status_dev, 4)) != cudaSuccess) cuda_fail(e, "status");
    else if ((e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking)) != cudaSuccess) cuda_fail(e, "side stream");
    else if ((e = cudaEventCreateWithFlags(&p->release_event, cudaEventDisableTiming)) != cudaSuccess) cuda_fail(e, "event");
    else if ((e = cudaEventCreateWithFlags(&p->load_event, cudaEventDisableTiming)) != cudaSuccess) cuda_fail(e, "event");
    else if ((e = cudaMemset(p->status_dev, 0, 4)) != cudaSuccess) cuda_fail(e, "memset");
    else if ((e = cudaMemset(p->dir_dev, 0xff, (size_t)max_adapters * sizeof(DirEntry))) != cudaSuccess) cuda_fail(e, "memset");
    else if ((e = cudaDeviceSynchronize()) != cudaSuccess) cuda_fail(e, "sync");
    if (st != SLORA_OK) {
        free_pool_memory(p);
        delete p;
        return st;
    }
    *out = p;
    return SLORA_OK;
}

slora_status slora_pool_destroy(slora_pool_t p)
{
    if (!p)
        return SLORA_OK;
    {
        DeviceScope dev_scope(p->device);
        free_pool_memory(p);
    }
    delete p;
    return SLORA_OK;
}

slora_status slora_pool_num_free(slora_pool_t p, int64_t *out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "pool_num_free");
    *out = p->pages.num_free();
    return SLORA_OK;
}

slora_status slora_pool_base(slora_pool_t p, void **out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "pool_base");
    *out = p->pool_dev;
    return SLORA_OK;
}

slora_status slora_pages_alloc(slora_pool_t p, int64_t n, int32_t *out_pages)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "pages_alloc: null pool");
    return p->pages.alloc(n, out_pages);
}

slora_status slora_pages_free(slora_pool_t p, int64_t n, const int32_t *pages, slora_stream_t stream)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "pages_free: null pool");
    slora_status st = p->pages.release(n, pages);
    if (st != SLORA_OK)
        return st;
    DEVICE_SCOPE(p);
    CUDA_TRY(cudaEventRecord(p->release_event, (cudaStream_t)stream));
    p->release_pending = true;
    return SLORA_OK;
}

slora_status slora_adapter_register(slora_pool_t p, int32_t id, int32_t rank, float scaling,
                                    const uint16_t *At_host, const uint16_t *B_host)
{
    if (!p || !valid_id(p, id) || rank < 1 || rank > 1024 || !At_host || !B_host)
        return fail(SLORA_ERR_INVALID_ARG, "adapter_register: id=%d rank=%d", id, rank);
    AdapterRec &a = p->adapters[(size_t)id];
    if (a.registered)
        return fail(SLORA_ERR_ALREADY_REGISTERED, "adapter_register: id=%d", id);
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    const size_t row = (size_t)p->hidden;
    const size_t rows = 2ull * (size_t)rank * (size_t)p->n_proj;
    AdapterRec n;
    n.rank = rank;
    n.scaling = scaling;
    if (cudaHostAlloc((void **)&n.store, rows * row * 2, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        return fail(SLORA_ERR_HOST_ALLOC, "adapter_register: %zu pinned bytes", rows * row * 2);
    }
    if (cudaHostAlloc((void **)&n.pt_host, rows * 4, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(n.store);
        return fail(SLORA_ERR_HOST_ALLOC, "adapter_register: page table");
    }
    void *sd = nullptr, *pd = nullptr;
    if (cudaHostGetDevicePointer(&sd, n.store, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&pd, n.pt_host, 0) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(n.store);
        cudaFreeHost(n.pt_host);
        return fail(SLORA_ERR_CUDA, "adapter_register: no device view of the pinned store");
    }
    n.store_dev = sd;
    n.pt_host_dev = static_cast<const int32_t *>(pd);
    // store layout per projection: A^T rows 0..r-1 then B rows 0..r-1, the page-table order
    for (int32_t pr = 0; pr < p->n_proj; ++pr) {
        uint16_t *dst = n.store + (size_t)pr * 2 * rank * row;
        memcpy(dst, At_host + (size_t)pr * rank * row, (size_t)rank * row * 2);
        memcpy(dst + (size_t)rank * row, B_host + (size_t)pr * rank * row, (size_t)rank * row * 2);
    }
    n.registered = true;
    a = n;
    if (rank > p->max_rank)
        p->max_rank = rank;
    return SLORA_OK;
}

slora_status slora_adapter_evict(slora_pool_t p, int32_t id, slora_stream_t stream);

slora_status slora_adapter_unregister(slora_pool_t p, int32_t id, slora_stream_t stream)
{
    if (!p || !valid_id(p, id))
        return fail(SLORA_ERR_INVALID_ARG, "adapter_unregister: id=%d", id);
    AdapterRec &a = p->adapters[(size_t)id];
    if (!a.registered)
        return fail(SLORA_ERR_NOT_REGISTERED, "adapter_unregister: id=%d", id);
    if (a.resident) {
        slora_status st = slora_adapter_evict(p, id, stream);
        if (st != SLORA_OK)
            return st;
    }
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    // the side stream may still copy out of the store
    CUDA_TRY(cudaStreamSynchronize(p->side));
    cudaFreeHost(a.store);
    cudaFreeHost(a.pt_host);
    a = AdapterRec();
    return SLORA_OK;
}

slora_status slora_adapters_load(slora_pool_t p, int32_t n, const int32_t *ids, slora_stream_t stream)
{
    if (!p || n < 0 || (n > 0 && !ids))
        return fail(SLORA_ERR_INVALID_ARG, "adapters_load: n=%d", n);
    std::vector<int32_t> todo;
    std::unordered_set<int32_t> seen;
    int64_t need_pages = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (!valid_id(p, id))
            return fail(SLORA_ERR_INVALID_ARG, "adapters_load: id=%d", id);
        const AdapterRec &a = p->adapters[(size_t)id];
        if (!a.registered)
            return fail(SLORA_ERR_NOT_REGISTERED, "adapters_load: id=%d", id);
        if (a.resident || !seen.insert(id).second)
            continue;
        todo.push_back(id);
        need_pages += adapter_rows(p, a);
    }
    if (todo.empty())
        return SLORA_OK;
    if (need_pages > p->pages.num_free())
        return fail(SLORA_ERR_POOL_FULL, "adapters_load: %lld pages needed, %lld free",
                    (long long)need_pages, (long long)p->pages.num_free());
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;

    // Host bookkeeping first (pages + arena), taken back if the arena is too fragmented.
    std::vector<int32_t> done;
    auto undo_host = [&]() {
        for (int32_t d : done) {
            AdapterRec &b = p->adapters[(size_t)d];
            p->pages.release(adapter_rows(p, b), b.pt_host);
            p->arena.release(b.pt_off, adapter_rows(p, b));
            b.pt_off = -1;
        }
    };
    for (int32_t id : todo) {
        AdapterRec &a = p->adapters[(size_t)id];
        int64_t rows = adapter_rows(p, a);
        int64_t off = inject_fault(SLORA_FAULT_ARENA) ? -1 : p->arena.alloc(rows);
        if (off < 0) {
            undo_host();
            return fail(SLORA_ERR_POOL_FULL, "adapters_load: page-table arena fragmented");
        }
        if (a.pt_read_pending) {   // a previous load kernel may still read pt_host
            const cudaError_t e = cudaEventSynchronize(p->load_event);   // recorded after every load's work
            if (e != cudaSuccess) {
                p->arena.release(off, rows);
                undo_host();
                return fail(SLORA_ERR_CUDA, "adapters_load: cudaEventSynchronize failed: %s", cudaGetErrorString(e));
            }
            for (int32_t t : todo) p->adapters[(size_t)t].pt_read_pending = false;
        }
        p->pages.alloc(rows, a.pt_host);  // cannot fail: counted above
        a.pt_off = off;
        done.push_back(id);
    }

    cudaStream_t side = p->side;
    // From here on a failure takes the load back: the side stream's work so far completes,
    // the directory entries of the load's adapters are cleared, and their pages and arena
    // ranges return to the free lists (nothing is left half loaded).
    auto rollback = [&](slora_status err) -> slora_status {
        cudaStreamSynchronize(side);
        DirArgs clr;
        clr.n = 0;
        for (size_t i = 0; i < todo.size(); ++i) {
            DirUpdate &u = clr.upd[clr.n++];
            u.adapter_id = todo[i];
            u.rank = 0;
            u.scaling = 0.f;
            u.pad = 0;
            u.pt_off = -1;
            if (clr.n == kMaxDirUpdatesPerLaunch || i + 1 == todo.size()) {
                ++p->residency_gen;
                if (launch_dir_update(p->dir_dev, clr, side) == cudaSuccess)
                    p->launches += 1;
                clr.n = 0;
            }
        }
        cudaStreamSynchronize(side);
        for (int32_t d : done) {
            AdapterRec &b = p->adapters[(size_t)d];
            p->pages.release(adapter_rows(p, b), b.pt_host);
            p->arena.release(b.pt_off, adapter_rows(p, b));
            b.pt_off = -1;
            b.pt_read_pending = false;
        }
        return err;
    };
#define LOAD_TRY(expr, kind)                                                                     \
    do {                                                                                        \
        const bool _inj = inject_fault(kind);                                                   \
        cudaError_t _e = _inj ? cudaErrorLaunchFailure : (expr);                                 \
        if (_e != cudaSuccess)                                                                  \
            return rollback(fail(SLORA_ERR_CUDA, "%s failed: %s%s (%s:%d)", #expr, cudaGetErrorString(_e), \
                                 _inj ? " (injected)" : "", __FILE__, __LINE__));               \
    } while (0)
    if (p->release_pending)
        LOAD_TRY(cudaStreamWaitEvent(side, p->release_event, 0), SLORA_FAULT_NONE);
    if (p->load_start_event)
        LOAD_TRY(cudaEventRecord(p->load_start_event, side), SLORA_FAULT_NONE);
    ScatterArgs sargs;
    sargs.n_runs = 0;
    auto flush = [&]() -> slora_status {
        if (sargs.n_runs == 0)
            return SLORA_OK;
        LOAD_TRY(launch_scatter(p->pt_dev, p->pool_dev, p->num_pages, p->hidden, sargs, p->status_dev,
                                p->num_sms, side),
                 SLORA_FAULT_SCATTER);
        p->launches += 1;
        sargs.n_runs = 0;
        return SLORA_OK;
    };
    if (p->load_mode == SLORA_LOAD_COPY_ENGINE) {
        // One cudaMemcpyAsync per adapter moves its pinned store block (all its rows,
        // contiguous) into the staging ring; one load kernel per ring-full writes the rows
        // from the ring to their pages.  Copies into a reused part of the ring are ordered
        // after the kernel that read it (one stream).
        int64_t largest = 0;
        for (int32_t id : todo)
            largest = std::max(largest, adapter_rows(p, p->adapters[(size_t)id]) * p->hidden * 2);
        if (largest > p->staging_bytes) {
            LOAD_TRY(cudaStreamSynchronize(side), SLORA_FAULT_NONE);
            if (p->staging) cudaFree(p->staging);
            p->staging = nullptr;
            p->staging_bytes = 0;
            LOAD_TRY(cudaMalloc(&p->staging, (size_t)largest), SLORA_FAULT_STAGING);
            p->staging_bytes = largest;
        }
        int64_t off = 0;
        for (int32_t id : todo) {
            AdapterRec &a = p->adapters[(size_t)id];
            const int64_t rows = adapter_rows(p, a), bytes = rows * p->hidden * 2;
            if (off + bytes > p->staging_bytes || sargs.n_runs == kMaxRunsPerLaunch) {
                if ((st = flush()) != SLORA_OK)
                    return st;
                off = 0;
            }
            LOAD_TRY(cudaMemcpyAsync(p->staging + off, a.store, (size_t)bytes, cudaMemcpyHostToDevice, side),
                     SLORA_FAULT_COPY);
            ScatterRun &run = sargs.runs[sargs.n_runs++];
            run.src = p->staging + off;
            run.pt_src = a.pt_host_dev;
            run.pt_index0 = a.pt_off;
            run.nrows = rows;
            off += (bytes + 255) / 256 * 256;
        }
    } else {
        // One kernel per kMaxRunsPerLaunch adapters reads the rows and their page ids
        // straight from the pinned store and page table, writes the pages and the
        // page-table arena.
        for (int32_t id : todo) {
            AdapterRec &a = p->adapters[(size_t)id];
            ScatterRun &run = sargs.runs[sargs.n_runs++];
            run.src = a.store_dev;
            run.pt_src = a.pt_host_dev;
            run.pt_index0 = a.pt_off;
            run.nrows = adapter_rows(p, a);
            if (sargs.n_runs == kMaxRunsPerLaunch && (st = flush()) != SLORA_OK)
                return st;
        }
    }
    if ((st = flush()) != SLORA_OK)
        return st;
    for (int32_t id : todo)   // read by the kernels above until the load event below
        p->adapters[(size_t)id].pt_read_pending = true;
    DirArgs dargs;
    dargs.n = 0;
    for (size_t i = 0; i < todo.size(); ++i) {
        AdapterRec &a = p->adapters[(size_t)todo[i]];
        DirUpdate &u = dargs.upd[dargs.n++];
        u.adapter_id = todo[i];
        u.rank = a.rank;
        u.scaling = a.scaling;
        u.pad = 0;
        u.pt_off = a.pt_off;
        if (dargs.n == kMaxDirUpdatesPerLaunch || i + 1 == todo.size()) {
            ++p->residency_gen;
            LOAD_TRY(launch_dir_update(p->dir_dev, dargs, side), SLORA_FAULT_DIRECTORY);
            p->launches += 1;
            dargs.n = 0;
        }
    }
    LOAD_TRY(cudaEventRecord(p->load_event, side), SLORA_FAULT_NONE);
    LOAD_TRY(cudaStreamWaitEvent((cudaStream_t)stream, p->load_event, 0), SLORA_FAULT_NONE);
#undef LOAD_TRY
    for (int32_t id : todo) {
        p->adapters[(size_t)id].resident = true;
        p->lru.insert(id);
    }
    p->n_loaded += (int64_t)todo.size();
    return SLORA_OK;
}

slora_status slora_adapter_load(slora_pool_t p, int32_t id, slora_stream_t stream)
{
    if (!p || !valid_id(p, id))
        return fail(SLORA_ERR_INVALID_ARG, "adapter_load: id=%d", id);
    const AdapterRec &a = p->adapters[(size_t)id];
    if (!a.registered)
        return fail(SLORA_ERR_NOT_REGISTERED, "adapter_load: id=%d", id);
    if (a.resident)
        return fail(SLORA_ERR_ALREADY_RESIDENT, "adapter_load: id=%d", id);
    return slora_adapters_load(p, 1, &id, stream);
}

slora_status slora_adapter_evict(slora_pool_t p, int32_t id, slora_stream_t stream)
{
    if (!p || !valid_id(p, id))
        return fail(SLORA_ERR_INVALID_ARG, "adapter_evict: id=%d", id);
    AdapterRec &a = p->adapters[(size_t)id];
    if (!a.registered)
        return fail(SLORA_ERR_NOT_REGISTERED, "adapter_evict: id=%d", id);
    if (!a.resident)
        return fail(SLORA_ERR_NOT_RESIDENT, "adapter_evict: id=%d", id);
    if (p->lru.pins(id) > 0)
        return fail(SLORA_ERR_INVALID_ARG, "adapter_evict: id=%d is pinned by an acquire", id);
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    DirArgs dargs;
    dargs.n = 1;
    dargs.upd[0] = DirUpdate{id, a.rank, a.scaling, 0, -1};
    ++p->residency_gen;
    CUDA_TRY(launch_dir_update(p->dir_dev, dargs, (cudaStream_t)stream));
    p->launches += 1;
    int64_t rows = adapter_rows(p, a);
    // pt_host still holds the pages handed out at load time
    if ((st = p->pages.release(rows, a.pt_host)) != SLORA_OK)
        return st;
    p->arena.release(a.pt_off, rows);
    a.pt_off = -1;
    a.resident = false;
    p->lru.remove(id);
    p->n_evicted += 1;
    CUDA_TRY(cudaEventRecord(p->release_event, (cudaStream_t)stream));
    p->release_pending = true;
    return SLORA_OK;
}

slora_status slora_adapters_evict(slora_pool_t p, int32_t n, const int32_t *ids, slora_stream_t stream)
{
    if (!p || n < 0 || (n > 0 && !ids))
        return fail(SLORA_ERR_INVALID_ARG, "adapters_evict: n=%d", n);
    std::vector<int32_t> todo;
    std::unordered_set<int32_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (!valid_id(p, id))
            return fail(SLORA_ERR_INVALID_ARG, "adapters_evict: id=%d", id);
        const AdapterRec &a = p->adapters[(size_t)id];
        if (!a.registered)
            return fail(SLORA_ERR_NOT_REGISTERED, "adapters_evict: id=%d", id);
        if (a.resident && p->lru.pins(id) > 0)
            return fail(SLORA_ERR_INVALID_ARG, "adapters_evict: id=%d is pinned by an acquire", id);
        if (a.resident && seen.insert(id).second)
            todo.push_back(id);
    }
    if (todo.empty())
        return SLORA_OK;
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    DirArgs dargs;
    dargs.n = 0;
    for (size_t i = 0; i < todo.size(); ++i) {
        const AdapterRec &a = p->adapters[(size_t)todo[i]];
        dargs.upd[dargs.n++] = DirUpdate{todo[i], a.rank, a.scaling, 0, -1};
        if (dargs.n == kMaxDirUpdatesPerLaunch || i + 1 == todo.size()) {
            ++p->residency_gen;
            CUDA_TRY(launch_dir_update(p->dir_dev, dargs, (cudaStream_t)stream));
            p->launches += 1;
            dargs.n = 0;
        }
    }
    for (int32_t id : todo) {
        AdapterRec &a = p->adapters[(size_t)id];
        const int64_t rows = adapter_rows(p, a);
        // pt_host still holds the pages handed out at load time
        if ((st = p->pages.release(rows, a.pt_host)) != SLORA_OK)
            return st;
        p->arena.release(a.pt_off, rows);
        a.pt_off = -1;
        a.resident = false;
        p->lru.remove(id);
    }
    p->n_evicted += (int64_t)todo.size();
    CUDA_TRY(cudaEventRecord(p->release_event, (cudaStream_t)stream));
    p->release_pending = true;
    return SLORA_OK;
}

// Least recently used unpinned adapters outside `exclude` whose pages, added to the free
// ones, reach `need`; false if even all of them do not.
static bool lru_victims(slora_pool_t p, const std::unordered_set<int32_t> &exclude, int64_t need,
                        std::vector<int32_t> *out)
{
    int64_t avail = p->pages.num_free();
    return p->lru.victims(exclude,
                          [&](const std::vector<int32_t> &v) {
                              if (!v.empty()) avail += adapter_rows(p, p->adapters[(size_t)v.back()]);
                              return avail >= need;
                          },
                          out);
}

slora_status slora_adapters_acquire(slora_pool_t p, int32_t n, const int32_t *ids, slora_stream_t stream)
{
    if (!p || n < 0 || (n > 0 && !ids))
        return fail(SLORA_ERR_INVALID_ARG, "adapters_acquire: n=%d", n);
    std::unordered_set<int32_t> want;
    std::vector<int32_t> missing;
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (!valid_id(p, id))
            return fail(SLORA_ERR_INVALID_ARG, "adapters_acquire: id=%d", id);
        const AdapterRec &a = p->adapters[(size_t)id];
        if (!a.registered)
            return fail(SLORA_ERR_NOT_REGISTERED, "adapters_acquire: id=%d", id);
        if (!want.insert(id).second)
            continue;
        if (!a.resident) {
            missing.push_back(id);
            need += adapter_rows(p, a);
        }
    }
    std::vector<int32_t> victims;
    if (!lru_victims(p, want, need, &victims))
        return fail(SLORA_ERR_POOL_FULL,
                    "adapters_acquire: %lld pages needed, %lld free, the rest held by pinned or requested adapters",
                    (long long)need, (long long)p->pages.num_free());
    slora_status st;
    if (!victims.empty() &&
        (st = slora_adapters_evict(p, (int32_t)victims.size(), victims.data(), stream)) != SLORA_OK)
        return st;
    if (!missing.empty() &&
        (st = slora_adapters_load(p, (int32_t)missing.size(), missing.data(), stream)) != SLORA_OK)
        return st;
    for (int32_t i = 0; i < n; ++i) {   // in the caller's order: later ids are more recent
        p->lru.touch(ids[i]);
    }
    for (int32_t id : want)
        p->lru.pin(id);
    return SLORA_OK;
}

slora_status slora_adapters_release(slora_pool_t p, int32_t n, const int32_t *ids)
{
    if (!p || n < 0 || (n > 0 && !ids))
        return fail(SLORA_ERR_INVALID_ARG, "adapters_release: n=%d", n);
    std::unordered_set<int32_t> seen;
    for (int32_t i = 0; i < n; ++i)
        if (seen.insert(ids[i]).second && (!valid_id(p, ids[i]) || p->lru.pins(ids[i]) == 0))
            return fail(SLORA_ERR_INVALID_ARG, "adapters_release: id=%d is not acquired", ids[i]);
    for (int32_t id : seen)
        p->lru.unpin(id);
    return SLORA_OK;
}

slora_status slora_pages_alloc_evict(slora_pool_t p, int64_t n, int32_t *out_pages, slora_stream_t stream)
{
    if (!p || n < 0 || (n > 0 && !out_pages))
        return fail(SLORA_ERR_INVALID_ARG, "pages_alloc_evict: n=%lld", (long long)n);
    std::vector<int32_t> victims;
    if (!lru_victims(p, {}, n, &victims))
        return fail(SLORA_ERR_POOL_FULL, "pages_alloc_evict: %lld pages needed, %lld free, the rest pinned",
                    (long long)n, (long long)p->pages.num_free());
    slora_status st;
    if (!victims.empty() &&
        (st = slora_adapters_evict(p, (int32_t)victims.size(), victims.data(), stream)) != SLORA_OK)
        return st;
    return p->pages.alloc(n, out_pages);
}

slora_status slora_pool_get_stats(slora_pool_t p, slora_pool_stats *out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "pool_get_stats");
    out->free_pages = p->pages.num_free();
    out->resident_adapters = (int64_t)p->lru.ents.size();
    out->pinned_adapters = (int64_t)(p->lru.ents.size() - p->lru.unpinned.size());
    out->adapters_loaded = p->n_loaded;
    out->adapters_evicted = p->n_evicted;
    return SLORA_OK;
}

slora_status slora_adapter_is_resident(slora_pool_t p, int32_t id, int32_t *out)
{
    if (!p || !valid_id(p, id) || !out)
        return fail(SLORA_ERR_INVALID_ARG, "adapter_is_resident: id=%d", id);
    *out = p->adapters[(size_t)id].resident ? 1 : 0;
    return SLORA_OK;
}

slora_status slora_adapter_rank(slora_pool_t p, int32_t id, int32_t *out)
{
    if (!p || !valid_id(p, id) || !out)
        return fail(SLORA_ERR_INVALID_ARG, "adapter_rank: id=%d", id);
    const AdapterRec &a = p->adapters[(size_t)id];
    if (!a.registered)
        return fail(SLORA_ERR_NOT_REGISTERED, "adapter_rank: id=%d", id);
    *out = a.rank;
    return SLORA_OK;
}

slora_status slora_adapter_pages(slora_pool_t p, int32_t id, int32_t proj, int32_t *out)
{
    if (!p || !valid_id(p, id) || !out || proj < 0 || proj >= (p ? p->n_proj : 0))
        return fail(SLORA_ERR_INVALID_ARG, "adapter_pages: id=%d proj=%d", id, proj);
    const AdapterRec &a = p->adapters[(size_t)id];
    if (!a.registered)
        return fail(SLORA_ERR_NOT_REGISTERED, "adapter_pages: id=%d", id);
    if (!a.resident)
        return fail(SLORA_ERR_NOT_RESIDENT, "adapter_pages: id=%d", id);
    memcpy(out, a.pt_host + (size_t)proj * 2 * a.rank, (size_t)2 * a.rank * 4);
    return SLORA_OK;
}

slora_status slora_page_read(slora_pool_t p, int32_t page, uint16_t *host_out)
{
    if (!p || page < 0 || page >= p->num_pages || !host_out)
        return fail(SLORA_ERR_INVALID_ARG, "page_read: page=%d", page);
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    CUDA_TRY(cudaDeviceSynchronize());
    CUDA_TRY(cudaMemcpy(host_out, p->pool_dev + (size_t)page * p->hidden, (size_t)p->hidden * 2,
                        cudaMemcpyDeviceToHost));
    return SLORA_OK;
}

slora_status slora_get_device_status(slora_pool_t p, int32_t *status)
{
    if (!p || !status)
        return fail(SLORA_ERR_INVALID_ARG, "get_device_status");
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    CUDA_TRY(cudaDeviceSynchronize());
    CUDA_TRY(cudaMemcpy(status, p->status_dev, 4, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemset(p->status_dev, 0, 4));
    CUDA_TRY(cudaDeviceSynchronize());
    return SLORA_OK;
}

static slora_status apply_list(slora_pool_t p, const char *fn, const ProjList &pl, int32_t T,
                               const int32_t *idx, const int32_t *seg_indptr, int32_t n_seg,
                               const float *scaling, slora_stream_t stream)
{
    if (T < 0 || T > (1 << 20))
        return fail(SLORA_ERR_INVALID_ARG, "%s: T=%d", fn, T);
    if (T == 0)
        return SLORA_OK;
    if (!idx)
        return fail(SLORA_ERR_INVALID_ARG, "%s: null token index pointer", fn);
    if (n_seg < 0 || (n_seg > 0 && !seg_indptr) || n_seg > T || n_seg > kMaxSegments)
        return fail(SLORA_ERR_INVALID_ARG, "%s: n_seg=%d (at most min(T, %d))", fn, n_seg, kMaxSegments);
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    const int32_t want_rank = std::max(p->max_rank, 1);
    if (T > p->plan.cap_tokens || want_rank > p->plan.max_rank || pl.n > p->plan.cap_proj) {
        int32_t cap = std::max(T, std::max(p->plan.cap_tokens, 256));
        const int32_t nproj = std::max(pl.n, p->plan.cap_proj);
        size_t bytes = plan_scratch_bytes(cap, want_rank, p->hidden, p->max_adapters, nproj);
        CUDA_TRY(cudaDeviceSynchronize());
        if (p->plan.base)
            cudaFree(p->plan.base);
        p->plan = PlanScratch();
        CUDA_TRY(cudaMalloc(&p->plan.base, bytes));
        CUDA_TRY(cudaMemset(p->plan.base, 0, bytes));
        p->plan.bytes = bytes;
        p->plan.cap_tokens = cap;
        p->plan.max_rank = want_rank;
        p->plan.cap_proj = nproj;
    }
    PoolView pv{p->pool_dev, p->pt_dev, p->dir_dev, p->num_pages, p->hidden, p->n_proj,
                p->max_adapters, p->status_dev};
    int launched = 0;
    cudaError_t e = launch_lora_apply(pv, pl, T, idx, seg_indptr, n_seg, scaling, p->plan, p->num_sms,
                                      (cudaStream_t)stream, &launched, p->stage_event);
    p->launches += launched;
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    return SLORA_OK;
}

slora_status slora_lora_apply(slora_pool_t p, int32_t proj, const void *x, void *y, int32_t T,
                              const int32_t *idx, const int32_t *seg_indptr, int32_t n_seg,
                              const float *scaling, slora_stream_t stream)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply: null pool");
    if (T == 0)
        return SLORA_OK;
    ProjList pl;
    void *ys[1] = {y};
    const void *xs[1] = {x};
    slora_status st = make_proj_list("lora_apply", p->n_proj, 1, &proj, xs, ys, &pl);
    if (st != SLORA_OK)
        return st;
    return apply_list(p, "lora_apply", pl, T, idx, seg_indptr, n_seg, scaling, stream);
}

slora_status slora_lora_apply_multi(slora_pool_t p, int32_t n, const int32_t *projs, const void *const *x,
                                    void *const *y, int32_t T, const int32_t *idx, const int32_t *seg_indptr,
                                    int32_t n_seg, const float *scaling, slora_stream_t stream)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_multi: null pool");
    ProjList pl;
    slora_status st = make_proj_list("lora_apply_multi", p->n_proj, n, projs, x, y, &pl);
    if (st != SLORA_OK)
        return st;
    return apply_list(p, "lora_apply_multi", pl, T, idx, seg_indptr, n_seg, scaling, stream);
}

// ---- batches planned once for several layers --------------------------------------------
struct slora_plan {
    slora_pool_t pool = nullptr;
    uint64_t residency_gen = 0;   // the pool's when planned: applies need the same directory
    int32_t n_slots = 0, T = 0, n_seg = 0;
    void *mem = nullptr;          // copies of the token map, segments and scaling; chunk scratch
    int32_t *idx = nullptr;
    int32_t *seg = nullptr;
    float *scale_mem = nullptr;   // room for a copy of the scaling override
    const float *scaling = nullptr;   // scale_mem when the plan has an override, else null
    std::vector<PlanScratch> chunks;
    int64_t applies = 0;          // applies since the plan was made or remade
};

// Copies the batch's token map, segments and scaling into the plan and runs the plan kernels.
static slora_status plan_batch(slora_plan *plan, const int32_t *idx, const int32_t *seg_indptr,
                               const float *scaling, cudaStream_t s, const char *fn)
{
    slora_pool_t p = plan->pool;
    cudaError_t e = cudaMemcpyAsync(plan->idx, idx, (size_t)plan->T * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && plan->n_seg > 0)
        e = cudaMemcpyAsync(plan->seg, seg_indptr, (size_t)(plan->n_seg + 1) * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && scaling)
        e = cudaMemcpyAsync(plan->scale_mem, scaling, (size_t)p->max_adapters * 4, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    plan->scaling = scaling ? plan->scale_mem : nullptr;
    PoolView pv{p->pool_dev, p->pt_dev, p->dir_dev, p->num_pages, p->hidden, p->n_proj, p->max_adapters,
                p->status_dev};
    int launched = 0;
    e = launch_plans(pv, plan->n_slots, plan->T, plan->idx, plan->n_seg > 0 ? plan->seg : nullptr, plan->n_seg,
                     plan->scaling, plan->chunks.data(), (int)plan->chunks.size(), p->num_sms, s, &launched);
    p->launches += launched;
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    plan->residency_gen = p->residency_gen;
    plan->applies = 0;
    return SLORA_OK;
}

slora_status slora_plan_create(slora_pool_t p, int32_t n_slots, int32_t T, const int32_t *idx,
                               const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                               slora_stream_t stream, slora_plan_t *out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "plan_create: null pool or out");
    *out = nullptr;
    if (n_slots < 1 || n_slots > kMaxApplyProj)
        return fail(SLORA_ERR_INVALID_ARG, "plan_create: n_slots=%d (1..%d)", n_slots, kMaxApplyProj);
    if (T < 1 || T > (1 << 20))
        return fail(SLORA_ERR_INVALID_ARG, "plan_create: T=%d (1..%d)", T, 1 << 20);
    if (!idx)
        return fail(SLORA_ERR_INVALID_ARG, "plan_create: null token index pointer");
    if (n_seg < 0 || (n_seg > 0 && !seg_indptr) || n_seg > T || n_seg > kMaxSegments)
        return fail(SLORA_ERR_INVALID_ARG, "plan_create: n_seg=%d (at most min(T, %d))", n_seg, kMaxSegments);
    DEVICE_SCOPE(p);
    slora_status st = SLORA_OK;
    const int32_t rank = std::max(p->max_rank, 1);
    const int32_t chunk = plan_chunk_tokens(p->max_adapters);
    const int n_chunks = (int)((T + (int64_t)chunk - 1) / chunk);
    const int32_t cap = std::min(T, chunk);
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t per_chunk = up(plan_scratch_bytes(cap, rank, p->hidden, p->max_adapters, n_slots));
    const size_t b_idx = up((size_t)T * 4), b_seg = up((size_t)(n_seg + 1) * 4);
    const size_t b_scale = up((size_t)p->max_adapters * 4);   // room for a scaling copy (create or remake)
    auto plan = std::make_unique<slora_plan>();
    plan->pool = p;
    plan->n_slots = n_slots;
    plan->T = T;
    plan->n_seg = n_seg;
    CUDA_TRY(cudaMalloc(&plan->mem, b_idx + b_seg + b_scale + per_chunk * n_chunks));
    uint8_t *m = static_cast<uint8_t *>(plan->mem);
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(m + b_idx + b_seg + b_scale, 0, per_chunk * n_chunks, s);
    if (e != cudaSuccess) {
        cudaFree(plan->mem);
        return fail(SLORA_ERR_CUDA, "plan_create: %s", cudaGetErrorString(e));
    }
    plan->idx = reinterpret_cast<int32_t *>(m);
    plan->seg = reinterpret_cast<int32_t *>(m + b_idx);
    plan->scale_mem = reinterpret_cast<float *>(m + b_idx + b_seg);
    plan->chunks.resize((size_t)n_chunks);
    for (int c = 0; c < n_chunks; ++c) {
        PlanScratch &sc = plan->chunks[(size_t)c];
        sc.base = m + b_idx + b_seg + b_scale + per_chunk * (size_t)c;
        sc.bytes = per_chunk;
        sc.cap_tokens = cap;
        sc.max_rank = rank;
        sc.cap_proj = n_slots;
    }
    st = plan_batch(plan.get(), idx, seg_indptr, scaling, s, "plan_create");
    if (st != SLORA_OK) {
        cudaStreamSynchronize(s);
        cudaFree(plan->mem);
        return st;
    }
    *out = plan.release();
    return SLORA_OK;
}

slora_status slora_plan_remake(slora_plan_t plan, const int32_t *idx, const int32_t *seg_indptr,
                               const float *scaling, slora_stream_t stream)
{
    if (!plan || !plan->pool)
        return fail(SLORA_ERR_INVALID_ARG, "plan_remake: null plan");
    if (!idx || (plan->n_seg > 0 && !seg_indptr))
        return fail(SLORA_ERR_INVALID_ARG, "plan_remake: null token index or segment pointer");
    DEVICE_SCOPE(plan->pool);
    slora_status st = plan_batch(plan, idx, seg_indptr, scaling, (cudaStream_t)stream, "plan_remake");
    return st;
}

slora_status slora_plan_apply(slora_plan_t plan, int32_t n, const int32_t *projs, const void *const *x,
                              void *const *y, slora_stream_t stream)
{
    if (!plan || !plan->pool)
        return fail(SLORA_ERR_INVALID_ARG, "plan_apply: null plan");
    slora_pool_t p = plan->pool;
    if (n != plan->n_slots)
        return fail(SLORA_ERR_INVALID_ARG, "plan_apply: n=%d, the plan was made for %d projections", n,
                    plan->n_slots);
    if (p->residency_gen != plan->residency_gen)
        return fail(SLORA_ERR_INVALID_ARG, "plan_apply: the pool's adapters were loaded or evicted since the "
                                           "plan was made");
    ProjList pl;
    slora_status st = make_proj_list("plan_apply", p->n_proj, n, projs, x, y, &pl);
    if (st != SLORA_OK)
        return st;
    DEVICE_SCOPE(p);
    PoolView pv{p->pool_dev, p->pt_dev, p->dir_dev, p->num_pages, p->hidden, p->n_proj, p->max_adapters,
                p->status_dev};
    int launched = 0;
    // after the first apply of a plan its plan kernels have completed before any later
    // apply starts (each decode launch waits for the kernel before it, back to the plan's)
    cudaError_t e = launch_planned(pv, pl, plan->T, plan->idx, plan->n_seg > 0 ? plan->seg : nullptr, plan->n_seg,
                                   plan->scaling, plan->chunks.data(), (int)plan->chunks.size(),
                                   plan->applies > 0, p->num_sms, (cudaStream_t)stream, &launched);
    p->launches += launched;
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "plan_apply: launch failed: %s", cudaGetErrorString(e));
    ++plan->applies;
    return SLORA_OK;
}

slora_status slora_plan_destroy(slora_plan_t plan)
{
    if (!plan)
        return SLORA_OK;
    slora_status st = SLORA_OK;
    if (plan->pool) {
        slora_pool_t p = plan->pool;
        DEVICE_SCOPE(p);
        // work still enqueued may read the plan: wait for the device, then free it
        CUDA_TRY(cudaDeviceSynchronize());
        CUDA_TRY(cudaFree(plan->mem));
    }
    delete plan;
    return st;
}

slora_status slora_pool_set_load_mode(slora_pool_t p, int32_t mode, int64_t staging_bytes)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "pool_set_load_mode: null pool");
    if ((mode != SLORA_LOAD_ZERO_COPY && mode != SLORA_LOAD_COPY_ENGINE) || staging_bytes < 0)
        return fail(SLORA_ERR_INVALID_ARG, "pool_set_load_mode: mode=%d staging_bytes=%lld", mode,
                    (long long)staging_bytes);
    DEVICE_SCOPE(p);
    const int64_t want = mode == SLORA_LOAD_COPY_ENGINE ? (staging_bytes > 0 ? staging_bytes : kDefaultStagingBytes) : 0;
    if (want != p->staging_bytes) {
        CUDA_TRY(cudaStreamSynchronize(p->side));   // no load still reads the old ring
        if (p->staging) cudaFree(p->staging);
        p->staging = nullptr;
        p->staging_bytes = 0;
        if (want > 0) {
            CUDA_TRY(cudaMalloc(&p->staging, (size_t)want));
            p->staging_bytes = want;
        }
    }
    p->load_mode = mode;
    return SLORA_OK;
}

slora_status slora_pool_get_load_mode(slora_pool_t p, int32_t *mode, int64_t *staging_bytes)
{
    if (!p || !mode || !staging_bytes)
        return fail(SLORA_ERR_INVALID_ARG, "pool_get_load_mode");
    *mode = p->load_mode;
    *staging_bytes = p->staging_bytes;
    return SLORA_OK;
}

slora_status slora_debug_inject_load_fault(int32_t kind, int32_t nth)
{
    if (kind < SLORA_FAULT_NONE || kind > SLORA_FAULT_ARENA || nth < 0)
        return fail(SLORA_ERR_INVALID_ARG, "debug_inject_load_fault: kind=%d nth=%d", kind, nth);
    std::lock_guard<std::mutex> lk(g_fault_mu);
    g_fault_kind = nth > 0 ? kind : SLORA_FAULT_NONE;
    g_fault_left = nth;
    return SLORA_OK;
}

slora_status slora_pool_set_load_start_event(slora_pool_t p, void *event)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "pool_set_load_start_event: null pool");
    p->load_start_event = (cudaEvent_t)event;
    return SLORA_OK;
}

slora_status slora_pool_set_stage_event(slora_pool_t p, void *event)
{
    if (!p)
        return fail(SLORA_ERR_INVALID_ARG, "pool_set_stage_event: null pool");
    p->stage_event = (cudaEvent_t)event;
    return SLORA_OK;
}

slora_status slora_pool_launch_count(slora_pool_t p, int64_t *out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "pool_launch_count");
    *out = p->launches;
    return SLORA_OK;
}

}  // extern "C"

slora_status slora::make_proj_list(const char *fn, int32_t pool_n_proj, int32_t n, const int32_t *projs,
                                   const void *const *x, void *const *y, ProjList *out)
{
    if (n < 1 || n > kMaxApplyProj)
        return fail(SLORA_ERR_INVALID_ARG, "%s: %d projections (1 to %d per call)", fn, n, kMaxApplyProj);
    if (!projs || !x || !y)
        return fail(SLORA_ERR_INVALID_ARG, "%s: null projection, x or y array", fn);
    out->n = n;
    for (int j = 0; j < n; ++j) {
        if (projs[j] < 0 || projs[j] >= pool_n_proj)
            return fail(SLORA_ERR_INVALID_ARG, "%s: proj=%d of %d", fn, projs[j], pool_n_proj);
        if (!x[j] || !y[j])
            return fail(SLORA_ERR_INVALID_ARG, "%s: null x / y pointer (entry %d)", fn, j);
        if (((uintptr_t)x[j] | (uintptr_t)y[j]) & 15)
            return fail(SLORA_ERR_INVALID_ARG, "%s: x and y must be 16-byte aligned (entry %d)", fn, j);
        for (int i = 0; i < n; ++i)
            if (y[j] == x[i] || (i != j && y[j] == y[i]))
                return fail(SLORA_ERR_INVALID_ARG, "%s: aliased x / y pointer (entries %d, %d)", fn, j, i);
        out->proj[j] = projs[j];
        out->x[j] = (const uint16_t *)x[j];
        out->y[j] = (uint16_t *)y[j];
    }
    return SLORA_OK;
}

slora_status slora::pool_hot_path(slora_pool_t p, PoolHotPath *out)
{
    if (!p || !out)
        return fail(SLORA_ERR_INVALID_ARG, "null pool");
    out->pv = PoolView{p->pool_dev, p->pt_dev, p->dir_dev, p->num_pages, p->hidden, p->n_proj,
                       p->max_adapters, p->status_dev};
    out->device = p->device;
    out->num_sms = p->num_sms;
    out->max_rank = p->max_rank;
    out->launches = &p->launches;
    return SLORA_OK;
}
