// The batched heterogeneous-rank LoRA delta, first version: one CTA per token.
// Each CTA gathers its token's A^T pages, forms u = x A with warp reductions (u stays
// in shared memory), then streams B's pages and writes y = y0 + s * u B.
// (S-LoRA: Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU, sections 2
// and 3; S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "The
// mechanism": custom kernels that gather non-contiguous adapter pages and tolerate
// heterogeneous ranks.)
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace slora {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void set_status(int32_t *status, int32_t code)
{
    atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(kThreads)
decode_token_kernel(PoolView pv, int32_t proj, const __half *__restrict__ x, __half *__restrict__ y,
                    int32_t T, const int32_t *__restrict__ idx, const float *__restrict__ scaling)
{
    extern __shared__ float smem[];
    const int d = pv.hidden;
    float *xs = smem;       // [d]
    float *u = smem + d;    // [rank]
    const int t = blockIdx.x;
    const int a = idx[t];
    if (a == -1)
        return;
    if (a < -1 || a >= pv.max_adapters) {
        if (threadIdx.x == 0) set_status(pv.status, SLORA_DEV_BAD_ADAPTER);
        return;
    }
    const DirEntry e = pv.dir[a];
    if (e.pt_off < 0 || e.rank <= 0) {
        if (threadIdx.x == 0) set_status(pv.status, SLORA_DEV_NOT_RESIDENT);
        return;
    }
    const int r = e.rank;
    const float s = scaling ? scaling[a] : e.scaling;
    const int32_t *pt = pv.pt_arena + e.pt_off + (int64_t)proj * 2 * r;
    for (int j = threadIdx.x; j < 2 * r; j += kThreads) {
        int32_t pg = pt[j];
        if (pg < 0 || pg >= pv.num_pages) set_status(pv.status, SLORA_DEV_BAD_PAGE);
    }
    const __half *xt = x + (int64_t)t * d;
    for (int k = threadIdx.x; k < d; k += kThreads)
        xs[k] = __half2float(xt[k]);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __half *pool = reinterpret_cast<const __half *>(pv.pool);
    for (int j = warp; j < r; j += kWarps) {
        int32_t pg = pt[j];
        float acc = 0.f;
        if (pg >= 0 && pg < pv.num_pages) {
            const __half *row = pool + (int64_t)pg * d;
            for (int k = lane; k < d; k += 32)
                acc += xs[k] * __half2float(row[k]);
        }
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) u[j] = acc;
    }
    __syncthreads();
    __half *yt = y + (int64_t)t * d;
    for (int n = threadIdx.x; n < d; n += kThreads) {
        float acc = 0.f;
        for (int j = 0; j < r; ++j) {
            int32_t pg = pt[r + j];
            if (pg >= 0 && pg < pv.num_pages)
                acc += u[j] * __half2float(pool[(int64_t)pg * d + n]);
        }
        yt[n] = __float2half_rn(__half2float(yt[n]) + s * acc);
    }
}

}  // namespace

size_t plan_scratch_bytes(int32_t T, int32_t max_adapters)
{
    (void)max_adapters;
    return (size_t)T * 16 + 256;
}

cudaError_t launch_lora_apply(const PoolView &pv, int32_t proj, const uint16_t *x, uint16_t *y,
                              int32_t T, const int32_t *idx, const int32_t *seg_indptr,
                              int32_t n_seg, const float *scaling, const PlanScratch &scratch,
                              int num_sms, cudaStream_t stream, int *launches)
{
    (void)seg_indptr; (void)n_seg; (void)scratch; (void)num_sms;
    size_t smem = (size_t)(pv.hidden + 1024) * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)((16384 + 1024) * sizeof(float)));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    decode_token_kernel<<<T, kThreads, smem, stream>>>(pv, proj, reinterpret_cast<const __half *>(x),
                                                       reinterpret_cast<__half *>(y), T, idx, scaling);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace slora
