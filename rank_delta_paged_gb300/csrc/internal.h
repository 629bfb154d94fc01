// Internal declarations shared by the host code and the kernels of libslora.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "slora.h"

namespace slora {

// Makes `device` current for the lifetime of the object, then gives the calling thread
// back the device it had: every entry point leaves the caller's current device as it
// found it.
class DeviceScope {
public:
    explicit DeviceScope(int device)
    {
        have_prev_ = cudaGetDevice(&prev_) == cudaSuccess;
        err_ = (have_prev_ && prev_ == device) ? cudaSuccess : cudaSetDevice(device);
    }
    ~DeviceScope()
    {
        if (have_prev_ && err_ == cudaSuccess) cudaSetDevice(prev_);
    }
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;
    cudaError_t error() const { return err_; }

private:
    int prev_ = 0;
    bool have_prev_ = false;
    cudaError_t err_ = cudaSuccess;
};

// One adapter's directory entry on the device, indexed by adapter id.
// pt_off < 0 means "not resident".  The page table of projection p starts at
// pt_arena[pt_off + p * 2 * rank]: rank A^T pages, then rank B pages.
struct alignas(16) DirEntry {
    int32_t rank;
    float scaling;
    int64_t pt_off;
};
static_assert(sizeof(DirEntry) == 16, "DirEntry layout");

// A run of consecutive rows of an adapter's pinned host store that land on the pages of
// consecutive page-table entries; the kernel reads both the rows and the page ids from
// host memory and writes the pages and the page-table arena entries.
struct ScatterRun {
    const void *src;         // device view of the first pinned store row
    const int32_t *pt_src;   // device view of the rows' page ids (pinned)
    int64_t pt_index0;       // first page-table arena entry
    int64_t nrows;
};
static_assert(sizeof(ScatterRun) == 32, "ScatterRun layout");

// Directory update carried as a kernel argument.
struct DirUpdate {
    int32_t adapter_id;
    int32_t rank;
    float scaling;
    int32_t pad;
    int64_t pt_off;
};

constexpr int kMaxRunsPerLaunch = 512;     // 512 * 32 B fits the 32 KiB parameter space
constexpr int kMaxDirUpdatesPerLaunch = 512;

struct ScatterArgs {
    int32_t n_runs;
    ScatterRun runs[kMaxRunsPerLaunch];
};
struct DirArgs {
    int32_t n;
    DirUpdate upd[kMaxDirUpdatesPerLaunch];
};

// Kernel launchers (scatter.cu).
cudaError_t launch_scatter(int32_t *pt_arena, uint16_t *pool, int64_t num_pages, int32_t hidden,
                           const ScatterArgs &args, int32_t *status, int num_sms, cudaStream_t stream);
cudaError_t launch_dir_update(DirEntry *dir, const DirArgs &args, cudaStream_t stream);

// Everything the hot-path kernels read about the pool.
struct PoolView {
    const uint16_t *pool;      // [num_pages][hidden] fp16
    const int32_t *pt_arena;
    const DirEntry *dir;
    int64_t num_pages;
    int32_t hidden;
    int32_t n_proj;
    int32_t max_adapters;
    int32_t *status;           // device status word
};

// Device scratch of the token plan and the decode kernel's partial sums (decode.cu),
// owned by the pool.
struct PlanScratch {
    void *base = nullptr;
    size_t bytes = 0;
    int32_t cap_tokens = 0;   // tokens the layout was carved for
    int32_t max_rank = 0;     // largest adapter rank the layout was carved for
    int32_t cap_proj = 0;     // projections per call the layout was carved for
    int32_t max_chunk = 0;    // tokens per plan at most (0: the plan's own limit)
    // Tag of the decode kernel's partial sums: each delta launch uses the next value.  0 means
    // the partial region must be cleared first (fresh scratch, or the sequence wrapped), so a
    // stale word can never carry a live tag.
    uint32_t tag = 0;
};
size_t plan_scratch_bytes(int32_t T, int32_t max_rank, int32_t hidden, int32_t max_adapters, int32_t n_proj);

// Segments whose adapter rank is at most this run on the tensor cores (prefill.cu);
// larger ranks take the decode path.  At most kMaxSegments segments per call.
constexpr int kMaxPrefillRank = 128;
constexpr int kMaxSegments = 4096;

// The projections one apply call covers: the same tokens and adapters, each entry with
// its own projection index, input x and in/out y (fp16 [T][hidden] on the device).  The
// x of several entries may be one buffer; the y buffers are distinct.
constexpr int kMaxApplyProj = 8;
struct ProjList {
    int32_t n;
    int32_t proj[kMaxApplyProj];
    const uint16_t *x[kMaxApplyProj];
    uint16_t *y[kMaxApplyProj];
};

// Checks the projection entries of an apply call (fn names the call in the error text)
// and fills *out: 1 <= n <= kMaxApplyProj, every projection index in [0, pool_n_proj),
// x and y non-null and 16-byte aligned, no y equal to another entry's y or to any x.
slora_status make_proj_list(const char *fn, int32_t pool_n_proj, int32_t n, const int32_t *projs,
                            const void *const *x, void *const *y, ProjList *out);

cudaError_t launch_prefill(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                           const int32_t *seg_indptr, int32_t n_seg, const float *scaling, int num_sms,
                           cudaStream_t stream);

// The hot path (decode.cu / prefill.cu): one token plan, one decode launch and one segment
// launch for every projection of the list.
cudaError_t launch_lora_apply(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                              const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                              PlanScratch &scratch, int num_sms, cudaStream_t stream, int *launches,
                              cudaEvent_t after_plan = nullptr);

// A batch planned once and applied to several layers (decode.cu): the plans of every chunk of
// at most plan_chunk_tokens(max_adapters) tokens into chunks[c], then, per apply, the decode
// kernel over each chunk's plan and the segment kernel.
int32_t plan_chunk_tokens(int32_t max_adapters);
cudaError_t launch_plans(const PoolView &pv, int32_t n_slots, int32_t T, const int32_t *idx,
                         const int32_t *seg_indptr, int32_t n_seg, const float *scaling, PlanScratch *chunks,
                         int n_chunks, int num_sms, cudaStream_t stream, int *launches);
// plan_ready: the plans were complete before this launch (not the first apply after the
// plans were made), so the decode kernel may read them before its grid-dependency wait.
cudaError_t launch_planned(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                           const int32_t *seg_indptr, int32_t n_seg, const float *scaling, PlanScratch *chunks,
                           int n_chunks, bool plan_ready, int num_sms, cudaStream_t stream, int *launches);

// What the hot path needs to know about a pool, for entry points defined outside
// pool.cpp (pool.cpp).  *launches points at the pool's kernel-launch counter.
struct PoolHotPath {
    PoolView pv;
    int device;
    int num_sms;
    int32_t max_rank;
    int64_t *launches;
};
slora_status pool_hot_path(slora_pool_t pool, PoolHotPath *out);

}  // namespace slora
