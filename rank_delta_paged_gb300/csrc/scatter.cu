// Adapter load: rows of an adapter store go to their pool pages, bit for bit, and the
// page ids of those rows into the device page-table arena, in one kernel that reads the
// rows either from the pinned host store over the CPU-GPU link (zero-copy mode) or from a
// device staging ring the copy engines filled (copy-engine mode); plus the
// adapter-directory update that publishes a load.
// (S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "The mechanism":
// only the adapters the running batch needs are fetched into the paged pool; a block
// table maps each logical row to its physical page.)
#include <cuda_runtime.h>

#include "internal.h"

namespace slora {
namespace {

constexpr int kScatterThreads = 256;

// One warp moves one row (hidden * 2 bytes, a multiple of 128 bytes): its page id from the
// host page table into the arena, and the row itself with 16-byte loads from its source
// (host memory, or the staging ring in device memory).  The page id and up to 16 loads
// per lane (a whole row at hidden 4096) are in flight together, so a row costs about one
// round trip over the CPU-GPU link.  Rows are found by a binary search over the runs' row
// prefix.
__global__ void __launch_bounds__(kScatterThreads)
scatter_kernel(int32_t *__restrict__ pt_arena, uint4 *__restrict__ pool, int64_t num_pages, int32_t row_vecs,
               const __grid_constant__ ScatterArgs args, int32_t *status)
{
    constexpr int kPer = 16;   // 16-byte loads per lane in flight
    __shared__ int64_t prefix[kMaxRunsPerLaunch + 1];
    if (threadIdx.x == 0) {
        int64_t acc = 0;
        prefix[0] = 0;
        for (int i = 0; i < args.n_runs; ++i) {
            acc += args.runs[i].nrows;
            prefix[i + 1] = acc;
        }
    }
    __syncthreads();
    const int64_t total = prefix[args.n_runs];
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kScatterThreads / 32);
    for (int64_t row = (int64_t)blockIdx.x * (kScatterThreads / 32) + (threadIdx.x >> 5); row < total;
         row += warps) {
        int lo = 0, hi = args.n_runs - 1;
        while (lo < hi) {  // last run with prefix[run] <= row
            int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= row) lo = mid; else hi = mid - 1;
        }
        const ScatterRun &run = args.runs[lo];
        const int64_t k = row - prefix[lo];
        const uint4 *src = reinterpret_cast<const uint4 *>(run.src) + k * row_vecs;
        const int32_t page = run.pt_src[k];
        for (int v0 = 0; v0 < row_vecs; v0 += 32 * kPer) {
            uint4 buf[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int v = v0 + lane + 32 * i;
                if (v < row_vecs) buf[i] = src[v];
            }
            if (v0 == 0 && lane == 0) pt_arena[run.pt_index0 + k] = page;
            if (page < 0 || page >= num_pages) {
                if (v0 == 0 && lane == 0) atomicCAS(status, 0, SLORA_DEV_BAD_PAGE);
                continue;
            }
            uint4 *dst = pool + (int64_t)page * row_vecs;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int v = v0 + lane + 32 * i;
                if (v < row_vecs) dst[v] = buf[i];
            }
        }
    }
}

__global__ void dir_update_kernel(DirEntry *dir, const __grid_constant__ DirArgs args)
{
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < args.n) {
        const DirUpdate &u = args.upd[i];
        DirEntry e;
        e.rank = u.rank;
        e.scaling = u.scaling;
        e.pt_off = u.pt_off;
        dir[u.adapter_id] = e;
    }
}

}  // namespace

cudaError_t launch_scatter(int32_t *pt_arena, uint16_t *pool, int64_t num_pages, int32_t hidden,
                           const ScatterArgs &args, int32_t *status, int num_sms, cudaStream_t stream)
{
    if (args.n_runs <= 0)
        return cudaSuccess;
    int64_t rows = 0;
    for (int i = 0; i < args.n_runs; ++i)
        rows += args.runs[i].nrows;
    const int warps_per_block = kScatterThreads / 32;
    int64_t blocks = (rows + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    scatter_kernel<<<(unsigned)blocks, kScatterThreads, 0, stream>>>(pt_arena, reinterpret_cast<uint4 *>(pool),
                                                                     num_pages, hidden / 8, args, status);
    return cudaGetLastError();
}

cudaError_t launch_dir_update(DirEntry *dir, const DirArgs &args, cudaStream_t stream)
{
    if (args.n <= 0)
        return cudaSuccess;
    dir_update_kernel<<<(args.n + 127) / 128, 128, 0, stream>>>(dir, args);
    return cudaGetLastError();
}

}  // namespace slora
