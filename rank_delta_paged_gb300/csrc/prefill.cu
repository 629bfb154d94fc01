// Prefill path of the LoRA delta: contiguous segments of tokens that share one adapter,
// computed as two dense contractions on the tcgen05 tensor cores with fp32 accumulators
// in tensor memory.
//
// S-LoRA: Serving Thousands of Concurrent LoRA Adapters (research note): the
// heterogeneous-batching kernels let a batch with different adapters' requests still run
// as efficient GEMMs; S-LoRA: Multiplexing Thousands of Fine-Tuned Adapters on a Single
// GPU, section 3: batched matrix multiplications for heterogeneous-rank adapters in one
// kernel invocation, with memory laid out so the tensor cores run near peak.  A prefill
// segment is the one place where the delta is a real GEMM: U = X_s A (T_s x r), then
// Y_s = Y0_s + s * U B.
//
// One persistent CTA per SM walks units (segment, 128-token M tile, column part):
//   shrink   K loop over hidden in 64-element blocks, 4-stage cp.async pipeline into
//            128-byte-swizzled K-major shared memory (X rows and the adapter's A^T page
//            rows, gathered through the page table), tcgen05.mma M=128, N=r (padded to a
//            multiple of 16 with zero rows in shared memory, never in the pool), K=16 per
//            instruction, accumulating in TMEM.
//   U        TMEM -> registers -> fp16 -> K-major swizzled shared memory (the A operand
//            of the expand).  This rounding of x A to fp16 is the only extra rounding.
//   expand   256-column tiles of B's page rows as the MN-major operand, double-buffered,
//            tcgen05.mma M=128, N=256, K=r; epilogue y = y0 + s * acc, one fp16 rounding.
// Every mbarrier wait is bounded; a unit whose tokens disagree on their adapter, or whose
// adapter is not resident, is skipped with a device status code.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"
#include "tcgen05.h"

namespace slora {
namespace {

constexpr int kPThreads = 256;
constexpr int MT = 128;            // tokens per M tile
constexpr int KBLK = 64;           // K elements per stage (one 128-byte swizzle atom row)
constexpr int NSTG = 4;
constexpr int NT = 256;            // expand N tile
constexpr int kXBytes = MT * 128;                  // 16 KiB
constexpr int kABytes = kMaxPrefillRank * 128;     // 16 KiB
constexpr int kStage = kXBytes + kABytes;          // 32 KiB
constexpr int kUBytes = (kMaxPrefillRank / 64) * MT * 128;   // 32 KiB
constexpr int kBBuf = kMaxPrefillRank * NT * 2;    // 64 KiB (two fit in the stage area)
constexpr uint32_t kTmemCols = 512;
constexpr int kSegSmem = (kMaxSegments + 1) * 4;
constexpr int kSmemBytes = 1024 /*align slack*/ + NSTG * kStage + kUBytes + kSegSmem + 2 * kMaxPrefillRank * 4;

static_assert(2 * kBBuf <= NSTG * kStage, "B double buffer reuses the shrink stages");

struct PrefillArgs {
    PoolView pv;
    int32_t proj;
    const __half *x;
    __half *y;
    int32_t T;
    const int32_t *idx;
    const int32_t *seg_indptr;
    int32_t n_seg;
    const float *scaling;
};

__device__ __forceinline__ uint4 pack_h8(const uint32_t *v)
{
    uint4 r;
    __half2 *h = reinterpret_cast<__half2 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        h[i] = __floats2half2_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    return r;
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;                                  // NSTG x (X 16K | A 16K)
    uint8_t *Us = smem + NSTG * kStage;                      // 2 K blocks x 16K
    int32_t *segp = reinterpret_cast<int32_t *>(Us + kUBytes);   // [n_seg + 1] tile prefix
    int32_t *pa = segp + (kMaxSegments + 1);                 // A^T pages of the unit
    int32_t *pb = pa + kMaxPrefillRank;                      // B pages
    __shared__ __align__(8) uint64_t mma_bar[NSTG];
    __shared__ __align__(8) uint64_t acc_bar[2];
    __shared__ uint32_t s_tmem;
    __shared__ int warp_sum[kPThreads / 32 + 1];
    __shared__ int s_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.pv.hidden;
    const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);

    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < NSTG; ++i) mbar_init(&mma_bar[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&acc_bar[i], 1);
        fence_mbar_init();
        s_flag = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    // segment tile prefix: segp[i] = M tiles before segment i
    {
        const int ns = a.n_seg;
        const int per = (ns + kPThreads - 1) / kPThreads;
        const int i0 = tid * per;
        int my = 0;
        for (int i = i0; i < i0 + per && i < ns; ++i) {
            const int lo = a.seg_indptr[i], hi = a.seg_indptr[i + 1];
            if (lo < 0 || hi < lo || hi > a.T) s_flag = 1;
            else my += (hi - lo + MT - 1) / MT;
        }
        int incl = my;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int w = 0; w < kPThreads / 32; ++w) {
                int v = warp_sum[w];
                warp_sum[w] = acc;
                acc += v;
            }
            warp_sum[kPThreads / 32] = acc;
        }
        __syncthreads();
        int base = warp_sum[warp] + incl - my;
        for (int i = i0; i < i0 + per && i < ns; ++i) {
            segp[i] = base;
            const int lo = a.seg_indptr[i], hi = a.seg_indptr[i + 1];
            if (!(lo < 0 || hi < lo || hi > a.T)) base += (hi - lo + MT - 1) / MT;
        }
        if (tid == 0) segp[ns] = warp_sum[kPThreads / 32];
        __syncthreads();
    }
    if (s_flag) {
        if (tid == 0) set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
    } else {
        const int total_mt = segp[a.n_seg];
        int S = (int)gridDim.x / (total_mt > 0 ? total_mt : 1);
        S = S < 1 ? 1 : (S > 4 ? 4 : S);
        const int cols_per = ((d + S - 1) / S + 63) / 64 * 64;
        const int S_eff = (d + cols_per - 1) / cols_per;
        const int units = total_mt * S_eff;
        uint32_t g_kb = 0;   // global K-block sequence (stage / phase bookkeeping)
        uint32_t g_nt = 0;   // global expand-tile sequence
        bool alive = true;

        for (int u = blockIdx.x; u < units && alive; u += gridDim.x) {
            const int mt = u / S_eff, part = u % S_eff;
            int lo_s = 0, hi_s = a.n_seg - 1;      // last segment with segp[i] <= mt
            while (lo_s < hi_s) {
                const int mid = (lo_s + hi_s + 1) >> 1;
                if (segp[mid] <= mt) lo_s = mid; else hi_s = mid - 1;
            }
            const int sg = lo_s;
            const int seg_lo = a.seg_indptr[sg], seg_hi = a.seg_indptr[sg + 1];
            const int m0 = seg_lo + (mt - segp[sg]) * MT;
            const int mlen = min(MT, seg_hi - m0);
            const int c_lo = part * cols_per;
            const int c_hi = min(d, c_lo + cols_per);

            // ---- adapter of the unit, checks ----
            const int ad = a.idx[m0];
            if (tid == 0) s_flag = 0;
            __syncthreads();
            for (int i = tid; i < mlen; i += kPThreads)
                if (a.idx[m0 + i] != ad) s_flag = 1;
            __syncthreads();
            if (s_flag) {
                if (tid == 0) set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
                continue;
            }
            if (ad == -1)
                continue;   // base only
            if (ad < -1 || ad >= a.pv.max_adapters) {
                if (tid == 0) set_status(a.pv.status, SLORA_DEV_BAD_ADAPTER);
                continue;
            }
            const DirEntry e = a.pv.dir[ad];
            if (e.pt_off < 0 || e.rank <= 0) {
                if (tid == 0) set_status(a.pv.status, SLORA_DEV_NOT_RESIDENT);
                continue;
            }
            const int r = e.rank;
            if (r > kMaxPrefillRank)
                continue;   // such segments take the decode path (the plan routes them there)
            const int r_pad = (r + 15) / 16 * 16;
            const float sc = a.scaling ? a.scaling[ad] : e.scaling;
            const int32_t *pt = a.pv.pt_arena + e.pt_off + (int64_t)a.proj * 2 * r;
            if (tid == 0) s_flag = 0;
            __syncthreads();
            for (int j = tid; j < r; j += kPThreads) {
                const int32_t p0 = pt[j], p1 = pt[r + j];
                if (p0 < 0 || p0 >= a.pv.num_pages || p1 < 0 || p1 >= a.pv.num_pages) s_flag = 1;
                pa[j] = p0;
                pb[j] = p1;
            }
            __syncthreads();
            if (s_flag) {
                if (tid == 0) set_status(a.pv.status, SLORA_DEV_BAD_PAGE);
                continue;
            }

            // ---- shrink: U = X A over K = d ----
            const int nkb = d / KBLK;
            auto issue = [&](int kb) {
                uint8_t *st = stages + ((g_kb + kb) % NSTG) * kStage;
                uint8_t *Xs = st, *As = st + kXBytes;
                for (int q = tid; q < MT * 8; q += kPThreads) {
                    const int m = q >> 3, ch = q & 7;
                    void *dst = Xs + m * 128 + ((ch ^ (m & 7)) << 4);
                    if (m < mlen)
                        cp_async16(dst, a.x + (int64_t)(m0 + m) * d + kb * KBLK + ch * 8, 16);
                    else
                        cp_async16(dst, a.x, 0);
                }
                for (int q = tid; q < r_pad * 8; q += kPThreads) {
                    const int j = q >> 3, ch = q & 7;
                    void *dst = As + j * 128 + ((ch ^ (j & 7)) << 4);
                    if (j < r)
                        cp_async16(dst, pool + (int64_t)pa[j] * d + kb * KBLK + ch * 8, 16);
                    else
                        cp_async16(dst, a.x, 0);
                }
                cp_async_commit();
            };
            for (int kb = 0; kb < NSTG - 1; ++kb) {
                if (kb < nkb) issue(kb);
                else cp_async_commit();
            }
            const uint32_t idesc_s = tc::idesc_f16_f32(MT, r_pad, 0, 0);
            for (int kb = 0; kb < nkb; ++kb) {
                const int nxt = kb + NSTG - 1;
                bool ok = true;
                if (nxt < nkb) {
                    if (kb >= 1) {   // the stage of block nxt was read by the MMAs of block kb-1
                        const uint32_t gq = g_kb + kb - 1;
                        ok = mbar_wait_bounded(&mma_bar[gq % NSTG], (gq / NSTG) & 1u, a.pv.status);
                    }
                    if (ok) issue(nxt);
                    else cp_async_commit();
                } else {
                    cp_async_commit();
                }
                cp_async_wait<NSTG - 1>();
                tc::fence_proxy_async_smem();
                if (__syncthreads_or(!ok)) { alive = false; break; }
                if (tid == 0) {
                    tc::fence_after_sync();
                    const uint32_t gq = g_kb + kb;
                    const uint8_t *st = stages + (gq % NSTG) * kStage;
                    const uint32_t xa = smem_u32(st), aa = smem_u32(st + kXBytes);
#pragma unroll
                    for (int kk = 0; kk < KBLK / 16; ++kk) {
                        tc::mma_f16(tmem, tc::smem_desc_sw128(xa + kk * 32, 16, 1024),
                                    tc::smem_desc_sw128(aa + kk * 32, 16, 1024), idesc_s,
                                    (kb | kk) != 0);
                    }
                    tc::commit(&mma_bar[gq % NSTG]);
                }
            }
            cp_async_wait<0>();
            if (!alive) break;
            {
                const uint32_t gq = g_kb + nkb - 1;
                const bool ok = mbar_wait_bounded(&mma_bar[gq % NSTG], (gq / NSTG) & 1u, a.pv.status);
                g_kb += nkb;
                if (__syncthreads_or(!ok)) { alive = false; break; }
            }
            tc::fence_after_sync();

            // ---- U: TMEM -> fp16 K-major swizzled shared memory ----
            if (warp < 4) {
                const int m = 32 * warp + lane;
                for (int cb = 0; cb < r_pad / 16; ++cb) {
                    uint32_t v[16];
                    tc::ld_32x32b_x16(tmem + ((uint32_t)(32 * warp) << 16) + cb * 16, v);
                    tc::ld_wait();
                    const int k = cb * 16;
                    uint8_t *row = Us + (k / 64) * (MT * 128) + m * 128;
                    const int ch0 = (k % 64) / 8;
                    *reinterpret_cast<uint4 *>(row + ((ch0 ^ (m & 7)) << 4)) = pack_h8(v);
                    *reinterpret_cast<uint4 *>(row + (((ch0 + 1) ^ (m & 7)) << 4)) = pack_h8(v + 8);
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();

            // ---- expand: Y = Y0 + s * U B over this unit's columns ----
            const int ntiles = (c_hi - c_lo + NT - 1) / NT;
            auto load_b = [&](int n, int buf) {
                const int n0 = c_lo + n * NT;
                const int nt = min(NT, c_hi - n0);
                const int cpr = nt / 8;   // 16-byte chunks per row
                uint8_t *Bs = stages + buf * kBBuf;
                for (int q = tid; q < r_pad * cpr; q += kPThreads) {
                    const int j = q / cpr, c = q % cpr;
                    const int col = c * 8;
                    void *dst = Bs + (j >> 3) * (4 * 1024) + (col >> 6) * 1024 + (j & 7) * 128 +
                                ((((col & 63) >> 3) ^ (j & 7)) << 4);
                    if (j < r)
                        cp_async16(dst, pool + (int64_t)pb[j] * d + n0 + col, 16);
                    else
                        cp_async16(dst, a.x, 0);
                }
                cp_async_commit();
            };
            load_b(0, 0);
            for (int n = 0; n < ntiles; ++n) {
                if (n + 1 < ntiles) load_b(n + 1, (n + 1) & 1);
                else cp_async_commit();
                cp_async_wait<1>();
                tc::fence_proxy_async_smem();
                __syncthreads();
                const int n0 = c_lo + n * NT;
                const int nt = min(NT, c_hi - n0);
                const uint32_t tb = g_nt & 1u;
                if (tid == 0) {
                    tc::fence_after_sync();
                    const uint32_t idesc_e = tc::idesc_f16_f32(MT, nt, 0, 1);
                    const uint32_t ua = smem_u32(Us);
                    const uint32_t ba = smem_u32(stages + (n & 1) * kBBuf);
                    for (int ks = 0; ks < r_pad / 16; ++ks) {
                        const int k = ks * 16;
                        const uint32_t a_addr = ua + (k / 64) * (MT * 128) + ((k % 64) / 16) * 32;
                        const uint32_t b_addr = ba + ks * 2 * (4 * 1024);
                        tc::mma_f16(tmem + tb * NT, tc::smem_desc_sw128(a_addr, 16, 1024),
                                    tc::smem_desc_sw128(b_addr, 1024, 4 * 1024), idesc_e, ks != 0);
                    }
                    tc::commit(&acc_bar[tb]);
                }
                const bool ok = mbar_wait_bounded(&acc_bar[tb], (g_nt >> 1) & 1u, a.pv.status);
                ++g_nt;
                if (__syncthreads_or(!ok)) { alive = false; break; }
                tc::fence_after_sync();
                // epilogue: warps w and w+4 share TMEM lanes 32*(w%4).. and split the columns
                const int sub = warp & 3, half = warp >> 2;
                const int m = 32 * sub + lane;
                const bool valid = m < mlen;
                const int64_t yrow = (int64_t)(m0 + m) * d;
                const int cols_half = nt / 2;
                for (int cc = 0; cc < cols_half; cc += 16) {
                    const int col = half * cols_half + cc;
                    uint32_t v[16];
                    tc::ld_32x32b_x16(tmem + tb * NT + ((uint32_t)(32 * sub) << 16) + col, v);
                    tc::ld_wait();
                    if (valid) {
                        uint4 *yp = reinterpret_cast<uint4 *>(a.y + yrow + n0 + col);
                        uint4 y0a = yp[0], y0b = yp[1];
                        const __half2 *ha = reinterpret_cast<const __half2 *>(&y0a);
                        const __half2 *hb = reinterpret_cast<const __half2 *>(&y0b);
                        uint32_t o[16];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float2 f = __half22float2(ha[i]);
                            o[2 * i] = __float_as_uint(fmaf(sc, __uint_as_float(v[2 * i]), f.x));
                            o[2 * i + 1] = __float_as_uint(fmaf(sc, __uint_as_float(v[2 * i + 1]), f.y));
                            float2 g = __half22float2(hb[i]);
                            o[8 + 2 * i] = __float_as_uint(fmaf(sc, __uint_as_float(v[8 + 2 * i]), g.x));
                            o[8 + 2 * i + 1] = __float_as_uint(fmaf(sc, __uint_as_float(v[8 + 2 * i + 1]), g.y));
                        }
                        yp[0] = pack_h8(o);
                        yp[1] = pack_h8(o + 8);
                    }
                }
                tc::fence_before_sync();
                __syncthreads();
            }
            cp_async_wait<0>();
            __syncthreads();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill(const PoolView &pv, int32_t proj, const uint16_t *x, uint16_t *y, int32_t T,
                           const int32_t *idx, const int32_t *seg_indptr, int32_t n_seg,
                           const float *scaling, int num_sms, cudaStream_t stream)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    PrefillArgs pa{pv, proj, reinterpret_cast<const __half *>(x), reinterpret_cast<__half *>(y), T, idx,
                   seg_indptr, n_seg, scaling};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel, pa);
}

}  // namespace slora
