// The padded batched-GEMM path: the comparison the S-LoRA ablation calls the slower BMM
// path (S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "Results and
// evidence", Figure 5 narrative: replacing the custom kernels with a slower BMM path hurts
// throughput and latency; same page, "Prior limits": per-adapter weights copied into
// contiguous, padded tensors).
//
// Each decode token gets its own dense copy of its adapter's factors, zero-padded to the
// pool's largest registered rank R: a gather kernel copies the token's A^T rows and its B
// rows (multiplied by the scaling s, a power of two for the ranks the pages use, so the
// product is exact) from the pool pages into W_A[t][R][hidden] and W_B[t][R][hidden];
// then two strided batched GEMMs of the cuBLAS library (fp16 in, fp32 accumulation) form
// u_t = W_A[t] x_t (rounded to fp16 once) and y_t = y0_t + W_B[t]^T u_t, one GEMM of the
// batch per token.  cuBLAS is loaded on first use (dlopen), so the rest of the library
// does not depend on it.  This path exists to be measured against the custom kernels;
// it moves every token's padded weights through HBM twice.
#include <dlfcn.h>

#include <cstring>
#include <mutex>

#include <cublas_api.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "host_common.h"
#include "internal.h"
#include "ptx.h"
#include "slora.h"

namespace slora {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kMaxDevices = 64;

// One warp per (token, row): rows 0..R-1 of W_A then rows 0..R-1 of W_B; rows past the
// adapter's rank, and every row of a token without a (resident, valid) adapter, are zero.
__global__ void __launch_bounds__(kGatherThreads)
bmm_gather_kernel(PoolView pv, int32_t proj, const int32_t *__restrict__ idx, int32_t T, int32_t R,
                  const float *__restrict__ scaling, uint4 *__restrict__ wa, uint4 *__restrict__ wb)
{
    const int lane = threadIdx.x & 31;
    const int64_t vecs = pv.hidden / 8;
    const int64_t total = (int64_t)T * 2 * R;
    const int64_t warps = (int64_t)gridDim.x * (kGatherThreads / 32);
    for (int64_t w = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); w < total; w += warps) {
        const int t = (int)(w / (2 * R));
        const int j2 = (int)(w - (int64_t)t * 2 * R);
        const bool is_b = j2 >= R;
        const int j = is_b ? j2 - R : j2;
        uint4 *dst = (is_b ? wb : wa) + ((int64_t)t * R + j) * vecs;
        const int ad = idx[t];
        int32_t page = -1;
        float s = 1.f;
        if (ad >= 0 && ad < pv.max_adapters) {
            const DirEntry e = pv.dir[ad];
            if (e.pt_off >= 0 && e.rank > 0) {
                if (j < e.rank) {
                    page = pv.pt_arena[e.pt_off + (int64_t)proj * 2 * e.rank + (is_b ? e.rank : 0) + j];
                    if (page < 0 || page >= pv.num_pages) {
                        if (lane == 0) set_status(pv.status, SLORA_DEV_BAD_PAGE);
                        page = -1;
                    }
                }
                s = scaling ? scaling[ad] : e.scaling;
            } else if (lane == 0 && j2 == 0) {
                set_status(pv.status, SLORA_DEV_NOT_RESIDENT);
            }
        } else if (ad != -1 && lane == 0 && j2 == 0) {
            set_status(pv.status, SLORA_DEV_BAD_ADAPTER);
        }
        const uint4 *src = page >= 0 ? reinterpret_cast<const uint4 *>(pv.pool) + (int64_t)page * vecs : nullptr;
        for (int64_t v = lane; v < vecs; v += 32) {
            uint4 q = make_uint4(0, 0, 0, 0);
            if (src) {
                q = src[v];
                if (is_b) {   // W_B = s * B, exact for a power-of-two s
                    __half2 *h = reinterpret_cast<__half2 *>(&q);
                    const __half2 s2 = __float2half2_rn(s);
#pragma unroll
                    for (int i = 0; i < 4; ++i) h[i] = __hmul2(h[i], s2);
                }
            }
            dst[v] = q;
        }
    }
}

// ---- cuBLAS, loaded on first use ------------------------------------------------------
using CreateFn = cublasStatus_t (*)(cublasHandle_t *);
using SetStreamFn = cublasStatus_t (*)(cublasHandle_t, cudaStream_t);
using GemmSBFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int,
                                    const void *, const void *, cudaDataType, int, long long int, const void *,
                                    cudaDataType, int, long long int, const void *, void *, cudaDataType, int,
                                    long long int, int, cublasComputeType_t, cublasGemmAlgo_t);
struct Cublas {
    CreateFn create = nullptr;
    SetStreamFn set_stream = nullptr;
    GemmSBFn gemm = nullptr;
    cublasHandle_t handle[kMaxDevices] = {};
};
std::mutex g_mu;
Cublas g_cb;
bool g_cb_tried = false;

slora_status cublas_for(int device, cudaStream_t stream, cublasHandle_t *out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_cb_tried) {
        g_cb_tried = true;
        void *h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL);
        if (!h) h = dlopen("libcublas.so", RTLD_NOW | RTLD_LOCAL);
        if (h) {
            g_cb.create = reinterpret_cast<CreateFn>(dlsym(h, "cublasCreate_v2"));
            g_cb.set_stream = reinterpret_cast<SetStreamFn>(dlsym(h, "cublasSetStream_v2"));
            g_cb.gemm = reinterpret_cast<GemmSBFn>(dlsym(h, "cublasGemmStridedBatchedEx"));
        }
    }
    if (!g_cb.create || !g_cb.set_stream || !g_cb.gemm)
        return fail(SLORA_ERR_UNSUPPORTED, "lora_apply_bmm: libcublas could not be loaded");
    if (device < 0 || device >= kMaxDevices)
        return fail(SLORA_ERR_UNSUPPORTED, "lora_apply_bmm: device %d", device);
    if (!g_cb.handle[device] && g_cb.create(&g_cb.handle[device]) != CUBLAS_STATUS_SUCCESS) {
        g_cb.handle[device] = nullptr;
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: cublasCreate failed");
    }
    if (g_cb.set_stream(g_cb.handle[device], stream) != CUBLAS_STATUS_SUCCESS)
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: cublasSetStream failed");
    *out = g_cb.handle[device];
    return SLORA_OK;
}

inline int32_t padded_rank(int32_t max_rank) { return max_rank < 1 ? 8 : (max_rank + 7) / 8 * 8; }

size_t workspace_bytes(int32_t T, int32_t R, int32_t hidden)
{
    const size_t w = (size_t)T * (size_t)R * (size_t)hidden * 2;   // one of W_A, W_B
    const size_t u = ((size_t)T * (size_t)R * 2 + 255) / 256 * 256;
    return 2 * w + u;
}

}  // namespace
}  // namespace slora

using namespace slora;

extern "C" slora_status slora_bmm_workspace_bytes(slora_pool_t pool, int32_t T, size_t *out)
{
    PoolHotPath hp;
    slora_status st = pool_hot_path(pool, &hp);
    if (st != SLORA_OK)
        return st;
    if (T < 0 || !out)
        return fail(SLORA_ERR_INVALID_ARG, "bmm_workspace_bytes: T=%d", T);
    *out = workspace_bytes(T, padded_rank(hp.max_rank), hp.pv.hidden);
    return SLORA_OK;
}

extern "C" slora_status slora_lora_apply_bmm(slora_pool_t pool, int32_t proj, const void *x, void *y, int32_t T,
                                             const int32_t *token_adapter_idx, const float *scaling,
                                             void *workspace, size_t workspace_bytes_, slora_stream_t stream)
{
    PoolHotPath hp;
    slora_status st = pool_hot_path(pool, &hp);
    if (st != SLORA_OK)
        return st;
    if (proj < 0 || proj >= hp.pv.n_proj)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_bmm: proj=%d of %d", proj, hp.pv.n_proj);
    if (T < 0 || T > (1 << 20))
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_bmm: T=%d", T);
    if (T == 0)
        return SLORA_OK;
    if (!x || !y || !token_adapter_idx || x == y || !workspace)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_bmm: null or aliased pointer");
    if (((uintptr_t)x | (uintptr_t)y | (uintptr_t)workspace) & 15)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_bmm: x, y and the workspace must be 16-byte aligned");
    const int32_t R = padded_rank(hp.max_rank), d = hp.pv.hidden;
    const size_t need = workspace_bytes(T, R, d);
    if (workspace_bytes_ < need)
        return fail(SLORA_ERR_INVALID_ARG, "lora_apply_bmm: workspace of %zu bytes, %zu needed", workspace_bytes_,
                    need);
    DeviceScope dev_scope(hp.device);   // the caller's current device comes back on return
    cudaError_t e = dev_scope.error();
    if (e != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: cudaSetDevice: %s", cudaGetErrorString(e));
    cublasHandle_t h;
    if ((st = cublas_for(hp.device, (cudaStream_t)stream, &h)) != SLORA_OK)
        return st;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t wbytes = (size_t)T * R * d * 2;
    __half *wa = reinterpret_cast<__half *>(ws), *wb = reinterpret_cast<__half *>(ws + wbytes);
    __half *u = reinterpret_cast<__half *>(ws + 2 * wbytes);
    const int64_t rows = (int64_t)T * 2 * R;
    int64_t blocks = (rows + kGatherThreads / 32 - 1) / (kGatherThreads / 32);
    const int64_t cap = (int64_t)(hp.num_sms > 0 ? hp.num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    bmm_gather_kernel<<<(unsigned)blocks, kGatherThreads, 0, (cudaStream_t)stream>>>(
        hp.pv, proj, token_adapter_idx, T, R, scaling, reinterpret_cast<uint4 *>(wa), reinterpret_cast<uint4 *>(wb));
    if ((e = cudaGetLastError()) != cudaSuccess)
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: gather launch: %s", cudaGetErrorString(e));
    *hp.launches += 1;
    const float one = 1.f, zero = 0.f;
    // u_t (R x 1) = W_A[t] (R x d, row-major = column-major d x R, transposed) x_t (d x 1)
    cublasStatus_t cs = g_cb.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, R, 1, d, &one, wa, CUDA_R_16F, d, (long long)R * d, x,
                                  CUDA_R_16F, d, d, &zero, u, CUDA_R_16F, R, R, T, CUBLAS_COMPUTE_32F,
                                  CUBLAS_GEMM_DEFAULT);
    if (cs != CUBLAS_STATUS_SUCCESS)
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: shrink GEMM failed (%d)", (int)cs);
    // y_t (d x 1) = W_B[t]^T (column-major d x R) u_t + y0_t
    cs = g_cb.gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, 1, R, &one, wb, CUDA_R_16F, d, (long long)R * d, u, CUDA_R_16F, R,
                   R, &one, y, CUDA_R_16F, d, d, T, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (cs != CUBLAS_STATUS_SUCCESS)
        return fail(SLORA_ERR_CUDA, "lora_apply_bmm: expand GEMM failed (%d)", (int)cs);
    return SLORA_OK;
}
