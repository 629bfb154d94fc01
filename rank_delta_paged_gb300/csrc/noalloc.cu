// slora_lora_apply_noalloc: the batched LoRA delta without any device allocation.
//
// slora_lora_apply keeps its scratch (the token plan, the decode kernel's work list, and
// the tagged fp32 partial sums of x A that its units exchange) in memory the pool allocates on
// first use and re-allocates (after a device synchronisation) when a larger batch, more
// projections per call or a larger adapter rank arrives.  Some callers cannot allow that: code that runs under a host
// framework whose allocator must own and account for every device byte, or a serving
// step with a fixed latency budget in which a cudaMalloc / cudaFree (and the device-wide
// synchronisation around them) is not acceptable.  This entry point serves them: its
// scratch is one file-scope device array of a fixed size, kNoAllocScratchBytes, which
// every GPU that loads this library holds until the process exits.  The caller passes
// the pool, inputs and outputs exactly as for slora_lora_apply.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "host_common.h"
#include "internal.h"
#include "slora.h"

namespace slora {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
constexpr int32_t kMinNoAllocChunk = 64;              // tokens per plan at least
constexpr int kMaxDevices = 64;

// Shared by every call of the entry point on a device; holds the last call's plan and
// partial sums.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};
// Per device: the tag sequence of the partial sums in the array (0: clear the array's
// partial region before the next launch).
uint32_t g_tag[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `device` (which must be current).  The name of
// the array in host code is only a host-side stand-in, so the address is fetched once per
// device with cudaGetSymbolAddress and cached.
slora_status scratch_for_device(int device, void **out)
{
    if (device < 0 || device >= kMaxDevices)
        return fail(SLORA_ERR_UNSUPPORTED, "lora_apply_noalloc: device %d beyond %d", device, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[device]) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return fail(SLORA_ERR_CUDA, "lora_apply_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_ptr[device] = ptr;
    }
    *out = g_scratch_ptr[device];
    return SLORA_OK;
}

}  // namespace
}  // namespace slora

using namespace slora;

extern "C" slora_status slora_lora_apply_noalloc(slora_pool_t pool, int32_t proj, const void *x, void *y,
                                                 int32_t T, const int32_t *token_adapter_idx,
                                                 const int32_t *seg_indptr, int32_t n_seg,
                                                 const float *scaling, slora_stream_t stream)
{
    PoolHotPath hp;
    slora_status st = pool_hot_path(pool, &hp);
    if (st != SLORA_OK)
        return st;
    if (T < 0 || T > (1 << 20))
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_noalloc: T=%d", T);
    if (T == 0)
        return SLORA_OK;
    ProjList pl;
    const void *xs[1] = {x};
    void *ys[1] = {y};
    if ((st = make_proj_list("lora_apply_noalloc", hp.pv.n_proj, 1, &proj, xs, ys, &pl)) != SLORA_OK)
        return st;
    if (!token_adapter_idx)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_noalloc: null token index pointer");
    if (n_seg < 0 || (n_seg > 0 && !seg_indptr) || n_seg > T || n_seg > kMaxSegments)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_noalloc: n_seg=%d (at most min(T, %d))", n_seg,
                    kMaxSegments);
    const int32_t max_rank = hp.max_rank > 0 ? hp.max_rank : 1;
    // The batch runs as plans of at most `chunk` tokens: the plan's own limit, halved until
    // one plan's scratch fits the array (every token's arithmetic is the same whatever
    // plan it is in); below kMinNoAllocChunk tokens the call is refused.
    int32_t chunk = T;
    while (chunk > kMinNoAllocChunk &&
           plan_scratch_bytes(chunk, max_rank, hp.pv.hidden, hp.pv.max_adapters, 1) > kNoAllocScratchBytes)
        chunk = (chunk + 1) / 2;
    const size_t need = plan_scratch_bytes(chunk, max_rank, hp.pv.hidden, hp.pv.max_adapters, 1);
    if (need > kNoAllocScratchBytes)
        return fail(SLORA_ERR_UNSUPPORTED,
                    "lora_apply_noalloc: a plan of %d tokens needs %zu bytes of scratch (largest registered "
                    "rank %d, hidden %d) but the static scratch holds %zu; use slora_lora_apply",
                    chunk, need, max_rank, hp.pv.hidden, kNoAllocScratchBytes);
    DeviceScope dev_scope(hp.device);   // the caller's current device comes back on return
    cudaError_t e = dev_scope.error();
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "lora_apply_noalloc: cudaSetDevice: %s", cudaGetErrorString(e));
    void *scratch = nullptr;
    if ((st = scratch_for_device(hp.device, &scratch)) != SLORA_OK)
        return st;
    // The plan kernel writes every scratch field the delta kernel reads (the header and its
    // unit counter, the work list) before the delta kernel starts, and a partial word is
    // read only once it carries the launch's tag, which no earlier launch used (the
    // partial region is cleared when the tag sequence starts or wraps; that is a memset on
    // the stream, not an allocation), so nothing else needs clearing here.
    PlanScratch ps;
    ps.base = scratch;
    ps.bytes = kNoAllocScratchBytes;
    ps.cap_tokens = chunk;
    ps.max_rank = max_rank;
    ps.cap_proj = 1;
    ps.max_chunk = chunk;
    int launched = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ps.tag = g_tag[hp.device];
        e = launch_lora_apply(hp.pv, pl, T, token_adapter_idx, seg_indptr, n_seg, scaling, ps, hp.num_sms,
                              (cudaStream_t)stream, &launched);
        g_tag[hp.device] = ps.tag;
    }
    *hp.launches += launched;
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "lora_apply_noalloc: launch failed: %s", cudaGetErrorString(e));
    return SLORA_OK;
}
