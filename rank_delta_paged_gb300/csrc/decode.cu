// Decode path of the heterogeneous-rank batched LoRA delta over the paged pool.
//
// S-LoRA: Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU, section 3: one
// kernel invocation for a batch whose requests use different adapters of different
// ranks; it gathers the tokens' hidden states and matches them against their adapters'
// pages through the paging table.  S-LoRA: Serving Thousands of Concurrent LoRA
// Adapters (explainer), "The mechanism": custom kernels that gather non-contiguous pages
// and tolerate heterogeneous ranks; "What to notice when reading": a batch mixing ranks
// needs kernels that do not assume one contiguous packing.
//
// Two kernels per batch (chained with programmatic dependent launch):
//
//   plan_kernel (one CTA): groups the decode tokens by adapter in a shared-memory hash
//     table and writes the work list: shrink items (adapter, 8 rank rows, <= 4 tokens)
//     first, then expand items (adapter, 1024 output columns, <= 4 tokens), each list in
//     descending rank.  Each item carries its group's fields.
//
//   delta_kernel (persistent, 128 threads, two CTAs per SM when ranks are at most 128):
//     each CTA takes a fixed subset of the items (rounds over the list in alternating
//     direction), loads their descriptors, page indices and token ids into shared memory,
//     then streams their page rows with cp.async: every thread copies its own 16-byte piece
//     of each row segment into a 4-deep per-thread ring, 3 tiles ahead of its arithmetic,
//     so no barrier guards the ring.  The threads compute
//       shrink  u[t][j] = sum_k x[t][k] * At[j][k]     (A^T rows + x rows per 1024-element
//               K tile; fp32 partials per thread, one butterfly reduce-scatter per warp,
//               written to a small fp32 scratch, published with release increments of the
//               group's counter)
//       expand  y[t][c] = y0[t][c] + s * sum_j u[t][j] * B[j][c]
//               (8 B row segments per tile; waits, with a time limit, until every shrink
//               item of its group has been published)
//     Each used adapter page row is read from HBM once per token chunk of its group (the
//     repeats of hot adapters hit L2).  Ranks 1..1024 run in the same launch: the last
//     rank chunk of an adapter simply has fewer rows; nothing in the pool is padded.
//
// Per-token arithmetic is fixed by the thread layout (which K elements a thread sums,
// the butterfly order, the row order of the expand), never by how tokens are grouped,
// so results do not depend on the batch, its order, or the physical pages.
#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"

namespace slora {
namespace {

constexpr int kDT = 128;                 // threads of the delta kernel
constexpr int kDW = kDT / 32;            // its warps
constexpr int RS = 8;       // A^T rows per shrink item
constexpr int TS = 4;       // tokens per shrink item
constexpr int TE = 4;       // tokens per expand item
constexpr int RB = 8;       // B rows per expand tile
constexpr int VC = 8 * kDT; // elements of a row segment: K per shrink tile, columns per expand item
constexpr int NST = 4;      // depth of each thread's cp.async ring (tiles)
constexpr int kMaxRank = 1024;
constexpr int kBatchItems = 32;          // item metadata a CTA holds at once
constexpr int kBatchPages = 2048;        // page indices a CTA holds at once

constexpr int kPlanThreads = 1024;
constexpr int kMaxPlanTokens = 16384;   // token-index range per plan when groups fit
constexpr int kMaxPlanGroups = 2048;    // distinct adapters per plan
constexpr int kMaxHash = 2 * kMaxPlanGroups;

static_assert(RS * TS == 32, "shrink item partials = one value per lane after the butterfly");
static_assert(RB <= RS + TS, "expand rows fit the tile slots");
static_assert(kBatchPages >= kMaxRank, "one expand item's pages always fit a batch");

struct PlanHeader {
    int32_t n_groups, n_shrink, n_expand, claim;
    int32_t seg_lo, seg_hi, pad0, pad1;
};
// One work item, with the fields of its group copied in.
struct alignas(16) Item {
    int32_t g, a, t0, nt;           // group, first rank row (shrink) or column chunk (expand), tokens
    int32_t rank, tok_begin, u_off, adapter;
    int32_t n_tok;
    float scaling;
    int64_t pt_base;                // arena index of this projection's page table
};
static_assert(sizeof(Item) == 48, "Item layout");

struct PlanLayout {
    PlanHeader *hdr;
    int32_t *tok_order;
    int32_t *done;
    Item *items;
    float *u;
    int64_t cap_items;
    int64_t cap_u;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Number of column chunks of the expand.
__host__ __device__ inline int n_col_chunks(int d) { return ceil_div(d, VC); }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tokens one plan covers: the whole range up to kMaxPlanTokens when every adapter id fits
// the plan's group tables, otherwise chunks of kMaxPlanGroups tokens.
inline int32_t plan_chunk(int32_t max_adapters)
{
    return max_adapters <= kMaxPlanGroups ? kMaxPlanTokens : kMaxPlanGroups;
}

PlanLayout carve(void *base, int32_t cap_tokens, int32_t max_rank, int32_t hidden, size_t *total)
{
    PlanLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return (char *)base + o;
    };
    const int64_t cap = cap_tokens;
    L.cap_items = cap * (ceil_div(max_rank, RS) + n_col_chunks(hidden));
    L.cap_u = cap * ((int64_t)max_rank + 4) + 16;   // per-group offsets padded to 4 floats
    L.hdr = (PlanHeader *)take(sizeof(PlanHeader));
    L.tok_order = (int32_t *)take(cap * 4);
    L.done = (int32_t *)take(cap * 4);
    L.items = (Item *)take(L.cap_items * sizeof(Item));
    L.u = (float *)take(L.cap_u * 4);
    if (total)
        *total = off;
    return L;
}

// ---- block-wide exclusive scan of one int per thread --------------------------------
// warp_tot: shared int[33]; every thread gets the block total in *total.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_tot[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - v;
    *total = warp_tot[32];
    __syncthreads();
    return r;
}

// Four exclusive scans at once (one set of barriers).  wt: shared int4[33].
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int4 *wt, int4 *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4 incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int nx = __shfl_up_sync(0xffffffffu, incl.x, o), ny = __shfl_up_sync(0xffffffffu, incl.y, o);
        const int nz = __shfl_up_sync(0xffffffffu, incl.z, o), nw = __shfl_up_sync(0xffffffffu, incl.w, o);
        if (lane >= o) { incl.x += nx; incl.y += ny; incl.z += nz; incl.w += nw; }
    }
    if (lane == 31) wt[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int4 w = (lane < (int)(blockDim.x >> 5)) ? wt[lane] : make_int4(0, 0, 0, 0);
        int4 wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nx = __shfl_up_sync(0xffffffffu, wi.x, o), ny = __shfl_up_sync(0xffffffffu, wi.y, o);
            const int nz = __shfl_up_sync(0xffffffffu, wi.z, o), nw = __shfl_up_sync(0xffffffffu, wi.w, o);
            if (lane >= o) { wi.x += nx; wi.y += ny; wi.z += nz; wi.w += nw; }
        }
        wt[lane] = make_int4(wi.x - w.x, wi.y - w.y, wi.z - w.z, wi.w - w.w);
        if (lane == 31) wt[32] = wi;
    }
    __syncthreads();
    const int4 b = wt[warp];
    *total = wt[32];
    __syncthreads();
    return make_int4(b.x + incl.x - v.x, b.y + incl.y - v.y, b.z + incl.z - v.z, b.w + incl.w - v.w);
}

struct PlanArgs {
    PoolView pv;
    int32_t proj;
    const int32_t *idx;
    int32_t T;
    const int32_t *seg_indptr;
    int32_t n_seg;
    int32_t t_begin, t_end;
    int32_t hash_size;  // power of two >= 2 * min(t_end - t_begin, max_adapters), <= kMaxHash
    PlanLayout L;
};

constexpr int kRankBuckets = 11;        // floor(log2(rank)) for ranks 1..1024

constexpr size_t plan_smem_bytes(int hs)
{
    return (size_t)hs * 4 + (size_t)kMaxPlanTokens * 2 + (size_t)13 * kMaxPlanGroups * 4;
}

__device__ __forceinline__ void plan_refuse(const PlanArgs &a)
{
    set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
    a.L.hdr->n_groups = 0;
    a.L.hdr->n_shrink = 0;
    a.L.hdr->n_expand = 0;
    a.L.hdr->claim = 0;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const __grid_constant__ PlanArgs a)
{
    extern __shared__ int plan_smem[];
    const int HS = a.hash_size;
    const int Tc = a.t_end - a.t_begin;
    int *keys = plan_smem;                                  // [HS] adapter id / -1, then group id
    short *tslot = reinterpret_cast<short *>(keys + HS);     // [Tc] hash slot, then group id
    int *gad = reinterpret_cast<int *>(tslot + kMaxPlanTokens);  // [G] adapter
    int *gn = gad + kMaxPlanGroups;                         // [G] tokens
    int *gtok = gn + kMaxPlanGroups;                        // [G] first token position
    int *gsh = gtok + kMaxPlanGroups;                       // [G] token placement cursor
    int *psh = gsh + kMaxPlanGroups;                        // [position] first shrink item
    int *pex = psh + kMaxPlanGroups;                        // [position] first expand item
    int *gu = pex + kMaxPlanGroups;                         // [G] first u float (multiple of 4)
    int *grank = gu + kMaxPlanGroups;                       // [G] rank
    float *gscale = reinterpret_cast<float *>(grank + kMaxPlanGroups);   // [G] scaling
    int *gperm = reinterpret_cast<int *>(gscale + kMaxPlanGroups);       // [position] group, by rank descending
    long long *gpt = reinterpret_cast<long long *>(gperm + kMaxPlanGroups);  // [G] page-table offset
    __shared__ int warp_tot[33];
    __shared__ int4 warp_tot4[33];
    __shared__ int s_lo, s_hi, s_G, s_nsh, s_nex, s_bad;
    __shared__ int s_bucket[kRankBuckets + 1];
    const int tid = threadIdx.x;
    const int d = a.pv.hidden;
    const int nch = n_col_chunks(d);

    griddep_launch_dependents();
    griddep_wait();

    if (tid == 0) {
        int lo = 0, hi = 0;
        if (a.n_seg > 0) {
            lo = a.seg_indptr[0];
            hi = a.seg_indptr[a.n_seg];
            if (lo < 0 || hi < lo || hi > a.T) {
                set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
                lo = hi = 0;
            }
        }
        s_lo = lo;
        s_hi = hi;
        s_bad = 0;
    }
    if (tid <= kRankBuckets)
        s_bucket[tid] = 0;
    for (int h = tid; h < HS; h += kPlanThreads)
        keys[h] = -1;
    for (int g = tid; g < kMaxPlanGroups; g += kPlanThreads)
        gn[g] = 0;
    __syncthreads();
    const int lo = s_lo, hi = s_hi;

    // 1. hash the decode tokens of [t_begin, t_end) by adapter
    for (int i = tid; i < Tc; i += kPlanThreads) {
        const int t = a.t_begin + i;
        int slot = -1;
        const bool in_seg = t >= lo && t < hi;
        const int ad = a.idx[t];
        if (ad >= 0 && ad < a.pv.max_adapters) {
            const DirEntry e = a.pv.dir[ad];
            const bool resident = e.pt_off >= 0 && e.rank > 0 && e.rank <= kMaxRank;
            // segment tokens run on the tensor cores unless their adapter's rank is too
            // large for that path; errors of segment tokens are reported there
            const bool mine = !in_seg || (resident && e.rank > kMaxPrefillRank);
            if (mine) {
                if (resident) {
                    int h = (int)(((uint32_t)ad * 2654435761u) & (uint32_t)(HS - 1));
                    for (int probe = 0; probe < HS; ++probe) {
                        const int k = atomicCAS(&keys[h], -1, ad);
                        if (k == -1 || k == ad) { slot = h; break; }
                        h = (h + 1) & (HS - 1);
                    }
                    if (slot < 0) s_bad = 1;   // more distinct adapters than the table holds
                } else {
                    set_status(a.pv.status, SLORA_DEV_NOT_RESIDENT);
                }
            }
        } else if (ad != -1 && !in_seg) {
            set_status(a.pv.status, SLORA_DEV_BAD_ADAPTER);
        }
        tslot[i] = (short)slot;
    }
    __syncthreads();

    // 2. groups = occupied slots, numbered in slot order; keys[h] becomes the group id;
    //    each group's directory entry is cached and its rank bucket counted
    {
        const int per = HS / kPlanThreads;
        const int h0 = tid * per;
        int c = 0;
        for (int h = h0; h < h0 + per; ++h)
            c += keys[h] != -1;
        int total;
        int base = block_excl_scan(c, warp_tot, &total);
        for (int h = h0; h < h0 + per; ++h) {
            const int k = keys[h];
            if (k != -1) {
                if (base < kMaxPlanGroups) {
                    const DirEntry e = a.pv.dir[k];
                    gad[base] = k;
                    grank[base] = e.rank;
                    gscale[base] = e.scaling;
                    gpt[base] = e.pt_off + (long long)a.proj * 2 * e.rank;
                    atomicAdd(&s_bucket[31 - __clz(e.rank)], 1);
                }
                keys[h] = base;
                ++base;
            }
        }
        if (tid == 0 && total > kMaxPlanGroups) s_bad = 1;
        if (tid == 0) s_G = total;
    }
    __syncthreads();
    if (s_bad) {
        // cannot happen with the host's chunking; refuse the batch rather than overrun
        if (tid == 0) plan_refuse(a);
        return;
    }
    const int G = s_G;
    if (tid == 0) {   // bucket starts, largest ranks first
        int acc = 0;
        for (int b = kRankBuckets - 1; b >= 0; --b) {
            const int n = s_bucket[b];
            s_bucket[b] = acc;
            acc += n;
        }
    }
    for (int i = tid; i < Tc; i += kPlanThreads) {
        const int h = tslot[i];
        if (h >= 0) {
            const int g = keys[h];
            tslot[i] = (short)g;
            atomicAdd(&gn[g], 1);
        }
    }
    __syncthreads();
    for (int g = tid; g < G; g += kPlanThreads)
        gperm[atomicAdd(&s_bucket[31 - __clz(grank[g])], 1)] = g;
    __syncthreads();

    // 3. per-group offsets (tokens, shrink items, expand items, u floats), laid out in
    //    descending-rank order so the costliest items are claimed first
    const int per_g = ceil_div(G > 0 ? G : 1, kPlanThreads);   // <= 2
    const int p0 = tid * per_g;
    int my_tok = 0, my_sh = 0, my_ex = 0, my_u = 0;
    for (int q = 0; q < per_g && p0 + q < G; ++q) {
        const int g = gperm[p0 + q];
        const int r = grank[g], n = gn[g];
        my_tok += n;
        my_sh += ceil_div(r, RS) * ceil_div(n, TS);
        my_ex += nch * ceil_div(n, TE);
        my_u += (n * r + 3) & ~3;
    }
    int4 tot4;
    const int4 off4 = block_excl_scan4(make_int4(my_tok, my_sh, my_ex, my_u), warp_tot4, &tot4);
    int off_tok = off4.x, off_sh = off4.y, off_ex = off4.z, off_u = off4.w;
    const int tot_sh = tot4.y, tot_ex = tot4.z, tot_u = tot4.w;
    for (int q = 0; q < per_g && p0 + q < G; ++q) {
        const int g = gperm[p0 + q];
        const int r = grank[g], n = gn[g];
        gtok[g] = off_tok;
        gu[g] = off_u;
        psh[p0 + q] = off_sh;
        pex[p0 + q] = off_ex;
        off_tok += n;
        off_sh += ceil_div(r, RS) * ceil_div(n, TS);
        off_ex += nch * ceil_div(n, TE);
        off_u += (n * r + 3) & ~3;
    }
    if (tid == 0) {
        s_nsh = tot_sh;
        s_nex = tot_ex;
    }
    __syncthreads();
    if ((int64_t)tot_sh + tot_ex > a.L.cap_items || (int64_t)tot_u + 4 > a.L.cap_u) {
        if (tid == 0) plan_refuse(a);
        return;
    }

    // 4. items, in parallel over items: each finds its group position by binary search over
    //    the (strictly increasing) first-item offsets
    for (int i = tid; i < tot_sh + tot_ex; i += kPlanThreads) {
        const bool sh = i < tot_sh;
        const int rel = sh ? i : i - tot_sh;
        const int *off = sh ? psh : pex;
        int lo_p = 0, hi_p = G - 1;
        while (lo_p < hi_p) {
            const int mid = (lo_p + hi_p + 1) >> 1;
            if (off[mid] <= rel) lo_p = mid; else hi_p = mid - 1;
        }
        const int g = gperm[lo_p];
        const int local = rel - off[lo_p];
        const int r = grank[g], n = gn[g];
        Item it;
        it.g = g;
        it.rank = r;
        it.tok_begin = gtok[g];
        it.u_off = gu[g];
        it.adapter = gad[g];
        it.n_tok = n;
        it.scaling = gscale[g];
        it.pt_base = gpt[g];
        if (sh) {
            const int ntc = ceil_div(n, TS), jc = local / ntc, tc = local - jc * ntc;
            it.a = jc * RS;
            it.t0 = tc * TS;
            it.nt = min(TS, n - tc * TS);
        } else {
            const int ntc = ceil_div(n, TE), c = local / ntc, tc = local - c * ntc;
            it.a = c;
            it.t0 = tc * TE;
            it.nt = min(TE, n - tc * TE);
        }
        const uint4 *src4 = reinterpret_cast<const uint4 *>(&it);
        uint4 *dst4 = reinterpret_cast<uint4 *>(a.L.items + i);
        dst4[0] = src4[0];
        dst4[1] = src4[1];
        dst4[2] = src4[2];
    }
    for (int g = tid; g < G; g += kPlanThreads)
        a.L.done[g] = 0;
    __syncthreads();
    // 5. token placement: gsh becomes the cursor
    for (int g = tid; g < G; g += kPlanThreads)
        gsh[g] = 0;
    __syncthreads();
    for (int i = tid; i < Tc; i += kPlanThreads) {
        const int g = tslot[i];
        if (g >= 0) {
            const int pos = gtok[g] + atomicAdd(&gsh[g], 1);
            a.L.tok_order[pos] = a.t_begin + i;
        }
    }
    if (tid == 0) {
        a.L.hdr->n_groups = G;
        a.L.hdr->n_shrink = s_nsh;
        a.L.hdr->n_expand = s_nex;
        a.L.hdr->claim = 0;
        a.L.hdr->seg_lo = lo;
        a.L.hdr->seg_hi = hi;
    }
}

struct DeltaArgs {
    PoolView pv;
    const __half *x;
    __half *y;
    const float *scaling;   // optional override [max_adapters]
    PlanLayout L;
    int32_t ustride;        // u row stride in shared memory: the largest rank rounded up to 8
};

__device__ __forceinline__ void h8_to_f(const uint4 &raw, float *f)
{
    const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 v = __half22float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

__device__ __forceinline__ uint4 f_to_h8(const float *f)
{
    uint4 raw;
    __half2 *h = reinterpret_cast<__half2 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return raw;
}

// Butterfly reduce-scatter of 32 per-lane values: afterwards lane L holds the warp sum
// of value L.
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            float send = upper ? v[i] : v[i + n / 2];
            float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// acc += x.lo * a.lo, then acc += x.hi * a.hi: fp16 operands, exact widening, one fp32
// rounding per product-add (the same value as widening both and using fmaf).
__device__ __forceinline__ float fma_h2(uint32_t x, uint32_t a, float acc)
{
    asm("{\n\t.reg .f16 xl, xh, al, ah;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, xl, al, %0;\n\tfma.rn.f32.f16 %0, xh, ah, %0;\n\t}"
        : "+f"(acc)
        : "r"(x), "r"(a));
    return acc;
}

// A tile is up to kSlots row segments of VC elements; every thread owns the same 16-byte
// piece (8 elements) of each segment.  Shrink tiles: 8 A^T rows then 4 token rows;
// expand tiles: 8 B rows.
constexpr int kSlots = RS + TS;

// acc[t][j] += x[t] . At[j] over the thread's 8 elements.  Rows past the adapter's rank
// are never loaded; their accumulators are never published.
template <int NT>
__device__ __forceinline__ void shrink_tile(const uint4 (&v)[kSlots], float (&acc)[TS][RS])
{
#pragma unroll
    for (int j = 0; j < RS; ++j) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float s = acc[t][j];
            s = fma_h2(v[RS + t].x, v[j].x, s);
            s = fma_h2(v[RS + t].y, v[j].y, s);
            s = fma_h2(v[RS + t].z, v[j].z, s);
            s = fma_h2(v[RS + t].w, v[j].w, s);
            acc[t][j] = s;
        }
    }
}

// acc[t][0..7] += u[t][j] * B[j][the thread's 8 columns], rows in order.  FULL: all 8 rows
// exist; otherwise rows past the rank contribute exactly zero.
template <int NT, bool FULL>
__device__ __forceinline__ void expand_tile(const uint4 (&v)[kSlots], const float *u_s, int ustride, int j0,
                                            int nrows, float (&acc)[TS][RS])
{
    float uu[NT][RB];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (FULL) {
            const float4 u0 = *reinterpret_cast<const float4 *>(u_s + t * ustride + j0);
            const float4 u1 = *reinterpret_cast<const float4 *>(u_s + t * ustride + j0 + 4);
            uu[t][0] = u0.x; uu[t][1] = u0.y; uu[t][2] = u0.z; uu[t][3] = u0.w;
            uu[t][4] = u1.x; uu[t][5] = u1.y; uu[t][6] = u1.z; uu[t][7] = u1.w;
        } else {
#pragma unroll
            for (int j = 0; j < RB; ++j)
                uu[t][j] = j < nrows ? u_s[t * ustride + j0 + j] : 0.f;
        }
    }
#pragma unroll
    for (int j = 0; j < RB; ++j) {
        float bf[8];
        h8_to_f((FULL || j < nrows) ? v[j] : make_uint4(0, 0, 0, 0), bf);
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[t][e] = fmaf(uu[t][j], bf[e], acc[t][e]);
    }
}

// Item index of this CTA's k-th item: rounds of gridDim.x items, walked in alternating
// direction so that the costliest items (the list is ordered by rank, descending) spread
// evenly over the CTAs.  Every CTA's items are increasing, so all its shrink items (which
// never wait) come before its expand items (which wait only on shrink items).
__device__ __forceinline__ int my_item(int k)
{
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    return k * G + ((k & 1) ? (G - 1 - b) : b);
}

__device__ __forceinline__ int item_pages(const Item &it, bool shrink)
{
    return shrink ? min(RS, it.rank - it.a) : it.rank;
}

template <bool V>
using bool_c = std::integral_constant<bool, V>;
template <int V>
using int_c = std::integral_constant<int, V>;

__global__ void __launch_bounds__(kDT, 2) delta_kernel(const __grid_constant__ DeltaArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint4 *stg = reinterpret_cast<uint4 *>(smem);                                   // [NST][kSlots][kDT]
    float *u_s = reinterpret_cast<float *>(smem + NST * kSlots * kDT * 16);       // [TE][ustride]
    float *red = u_s + TE * a.ustride;                                             // [2][kDW][32]
    Item *mit = reinterpret_cast<Item *>(red + 2 * kDW * 32);                      // [kBatchItems]
    int *mpo = reinterpret_cast<int *>(mit + kBatchItems);                         // [kBatchItems + 1]
    int *mpg = mpo + kBatchItems + 1;                                              // [kBatchPages]
    int *mtk = mpg + kBatchPages;                                                  // [kBatchItems][TE]
    __shared__ int s_nb, s_flag;

    constexpr uint32_t kSlotB = kDT * 16;          // one row segment of the CTA
    constexpr uint32_t kStageB = kSlots * kSlotB;  // one tile
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.pv.hidden;
    const int nkt = ceil_div(d, VC);               // K tiles of a shrink item
    const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);
    const uint32_t sbase = smem_u32(stg) + (uint32_t)tid * 16;

    griddep_wait();   // the plan of this batch is complete and visible
    griddep_launch_dependents();
    const int n_sh = a.L.hdr->n_shrink;
    const int n_tot = n_sh + a.L.hdr->n_expand;

    float acc[TS][RS];
    int n_red = 0;
    for (int k0 = 0;;) {
        // ---- metadata of the next batch of this CTA's items, into shared memory ----
        if (tid < kBatchItems) {
            const int i = my_item(k0 + tid);
            if (i < n_tot)
                mit[tid] = a.L.items[i];
        }
        __syncthreads();
        if (tid == 0) {
            int nb = 0, np = 0;
            while (nb < kBatchItems && my_item(k0 + nb) < n_tot) {
                const int need = item_pages(mit[nb], my_item(k0 + nb) < n_sh);
                if (np + need > kBatchPages) break;
                mpo[nb] = np;
                np += need;
                ++nb;
            }
            mpo[nb] = np;
            s_nb = nb;
        }
        __syncthreads();
        const int nb = s_nb;
        if (nb == 0)
            break;
        for (int q = 0; q < nb; ++q) {
            const bool sh = my_item(k0 + q) < n_sh;
            const Item &it = mit[q];
            const int np = mpo[q + 1] - mpo[q];
            const int64_t base = it.pt_base + (sh ? it.a : it.rank);
            for (int j = tid; j < np; j += kDT) {
                int32_t pg = a.pv.pt_arena[base + j];
                if (pg < 0 || pg >= a.pv.num_pages) {
                    set_status(a.pv.status, SLORA_DEV_BAD_PAGE);
                    pg = -1;
                }
                mpg[mpo[q] + j] = pg;
            }
        }
        for (int e = tid; e < nb * TE; e += kDT) {
            const int q = e / TE, t = e - q * TE;
            const Item &it = mit[q];
            mtk[e] = t < it.nt ? a.L.tok_order[it.tok_begin + it.t0 + t] : -1;
        }
        __syncthreads();

        // ---- copy stream: every thread copies its own 16-byte piece of each row segment
        //      into an NST-deep ring, NST-1 tiles ahead of its arithmetic ----
        int is_q = 0, is_sub = 0, is_ntiles = 0, is_rank = 0, is_col = 0;
        bool is_sh = true;
        const int *is_pg = mpg;
        const __half *is_src[kSlots];
        auto load_issue_item = [&]() {
            if (is_q >= nb)
                return;
            const Item &it = mit[is_q];
            is_sh = my_item(k0 + is_q) < n_sh;
            is_pg = mpg + mpo[is_q];
            if (is_sh) {
                is_ntiles = nkt;
                const int nrows = min(RS, it.rank - it.a);
#pragma unroll
                for (int j = 0; j < RS; ++j)
                    is_src[j] = (j < nrows && is_pg[j] >= 0) ? pool + (int64_t)is_pg[j] * d + 8 * tid : nullptr;
#pragma unroll
                for (int t = 0; t < TS; ++t)
                    is_src[RS + t] = t < it.nt ? a.x + (int64_t)mtk[is_q * TE + t] * d + 8 * tid : nullptr;
            } else {
                is_ntiles = ceil_div(it.rank, RB);
                is_rank = it.rank;
                is_col = it.a * VC + 8 * tid;
            }
        };
        auto issue_tile = [&](int stage) {
            if (is_q < nb) {
                const uint32_t sd = sbase + (uint32_t)stage * kStageB;
                if (is_sh) {
                    const int off = is_sub * VC;
                    if (off + 8 * tid < d) {
#pragma unroll
                        for (int j = 0; j < kSlots; ++j)
                            if (is_src[j])
                                cp_async16_s(sd + j * kSlotB, is_src[j] + off);
                    }
                } else if (is_col < d) {
                    const int j0 = is_sub * RB;
#pragma unroll
                    for (int j = 0; j < RB; ++j)
                        if (j0 + j < is_rank && is_pg[j0 + j] >= 0)
                            cp_async16_s(sd + j * kSlotB, pool + (int64_t)is_pg[j0 + j] * d + is_col);
                }
                if (++is_sub == is_ntiles) {
                    is_sub = 0;
                    ++is_q;
                    load_issue_item();
                }
            }
            cp_async_commit();   // one group per tile, possibly empty
        };
        load_issue_item();
#pragma unroll 1
        for (int p = 0; p < NST - 1; ++p)
            issue_tile(p);

        int ct = 0;   // tiles consumed in this batch
        // One item's tiles, with the item kind and token count fixed at compile time.
        auto run_item = [&](int q, auto sh_c, auto nt_c) {
            constexpr bool SH = decltype(sh_c)::value;
            constexpr int NT = decltype(nt_c)::value;
            const Item it = mit[q];
            const int ntiles = SH ? nkt : ceil_div(it.rank, RB);
            const int col = it.a * VC + 8 * tid;
#pragma unroll
            for (int t = 0; t < TS; ++t)
#pragma unroll
                for (int j = 0; j < RS; ++j)
                    acc[t][j] = 0.f;
            uint4 yv[NT];
            bool ok = true;
            if (!SH) {
                if (col < d) {
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        yv[t] = *reinterpret_cast<const uint4 *>(a.y + (int64_t)mtk[q * TE + t] * d + col);
                }
                __syncthreads();   // every thread is done with the previous item's u_s
                if (tid == 0) {
                    // every shrink item of the group has published its u values?
                    const int need = 32 * ceil_div(it.rank, RS) * ceil_div(it.n_tok, TS);
                    int flag = 1;
                    if (ld_acquire_gpu(&a.L.done[it.g]) < need) {
                        const uint64_t t0 = global_timer_ns();
                        for (;;) {
                            __nanosleep(32);
                            if (ld_acquire_gpu(&a.L.done[it.g]) >= need) break;
                            if (global_timer_ns() - t0 > kWaitLimitNs) {
                                set_status(a.pv.status, SLORA_DEV_TIMEOUT);
                                flag = 0;
                                break;
                            }
                        }
                    }
                    s_flag = flag;
                }
                __syncthreads();
                ok = s_flag != 0;
                const int r = it.rank;
                const float *ug = a.L.u + it.u_off + (int64_t)it.t0 * r;
                for (int e = tid; e < NT * r; e += kDT) {
                    const int t = e / r, j = e - t * r;
                    u_s[t * a.ustride + j] = __ldcg(ug + e);
                }
                __syncthreads();
            }
#pragma unroll 1
            for (int sub = 0; sub < ntiles; ++sub) {
                issue_tile((ct + NST - 1) % NST);
                cp_async_wait<NST - 1>();   // this thread's copies of tile ct have landed
                const uint4 *slot = stg + (ct % NST) * (kSlots * kDT) + tid;
                if (SH) {
                    if (sub * VC + 8 * tid < d) {
                        uint4 v[kSlots];
#pragma unroll
                        for (int i = 0; i < RS + NT; ++i)
                            v[i] = slot[i * kDT];
                        shrink_tile<NT>(v, acc);
                    }
                } else if (col < d) {
                    const int j0 = sub * RB;
                    const int nrows = min(RB, it.rank - j0);
                    uint4 v[kSlots];
                    if (nrows == RB) {
#pragma unroll
                        for (int i = 0; i < RB; ++i)
                            v[i] = slot[i * kDT];
                        expand_tile<NT, true>(v, u_s, a.ustride, j0, nrows, acc);
                    } else {
#pragma unroll
                        for (int i = 0; i < RB; ++i)
                            v[i] = i < nrows ? slot[i * kDT] : make_uint4(0, 0, 0, 0);
                        expand_tile<NT, false>(v, u_s, a.ustride, j0, nrows, acc);
                    }
                }
                ++ct;
            }
            if (SH) {
                // ---- reduce the 32 partials over the CTA, publish u ----
                float vv[32];
#pragma unroll
                for (int t = 0; t < TS; ++t)
#pragma unroll
                    for (int j = 0; j < RS; ++j)
                        vv[t * RS + j] = acc[t][j];
                const float ws = warp_reduce_scatter32(vv);
                float *rb = red + (n_red & 1) * (kDW * 32);
                ++n_red;
                rb[warp * 32 + lane] = ws;
                __syncthreads();
                if (tid < 32) {
                    float tot = 0.f;
#pragma unroll
                    for (int w = 0; w < kDW; ++w)
                        tot += rb[w * 32 + tid];
                    const int t = tid / RS, j = tid % RS;
                    if (t < it.nt && it.a + j < it.rank)
                        __stcg(a.L.u + it.u_off + (int64_t)(it.t0 + t) * it.rank + it.a + j, tot);
                    red_release_add1(&a.L.done[it.g]);   // 32 per shrink item
                }
            } else if (ok && col < d) {
                const float sc = a.scaling ? a.scaling[it.adapter] : it.scaling;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float y0f[8], out[8];
                    h8_to_f(yv[t], y0f);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        out[e] = fmaf(sc, acc[t][e], y0f[e]);
                    *reinterpret_cast<uint4 *>(a.y + (int64_t)mtk[q * TE + t] * d + col) = f_to_h8(out);
                }
            }
        };
        for (int q = 0; q < nb; ++q) {
            const bool sh = my_item(k0 + q) < n_sh;
            const int nt = mit[q].nt;
            if (sh) {
                switch (nt) {
                case 1: run_item(q, bool_c<true>(), int_c<1>()); break;
                case 2: run_item(q, bool_c<true>(), int_c<2>()); break;
                case 3: run_item(q, bool_c<true>(), int_c<3>()); break;
                default: run_item(q, bool_c<true>(), int_c<4>()); break;
                }
            } else {
                switch (nt) {
                case 1: run_item(q, bool_c<false>(), int_c<1>()); break;
                case 2: run_item(q, bool_c<false>(), int_c<2>()); break;
                case 3: run_item(q, bool_c<false>(), int_c<3>()); break;
                default: run_item(q, bool_c<false>(), int_c<4>()); break;
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();   // the batch's metadata is about to be replaced
        k0 += nb;
    }
}

}  // namespace

size_t plan_scratch_bytes(int32_t T, int32_t max_rank, int32_t hidden, int32_t max_adapters)
{
    size_t total = 0;
    const int32_t chunk = plan_chunk(max_adapters);
    const int32_t cap = T < chunk ? T : chunk;
    carve(nullptr, cap, max_rank, hidden, &total);
    return total;
}

inline size_t delta_smem_bytes(int ustride)
{
    return (size_t)NST * kSlots * kDT * 16 + (size_t)TE * ustride * 4 + 2 * kDW * 32 * 4 +
           kBatchItems * sizeof(Item) + (kBatchItems + 1) * 4 + kBatchPages * 4 + kBatchItems * TE * 4;
}

cudaError_t launch_lora_apply(const PoolView &pv, int32_t proj, const uint16_t *x, uint16_t *y,
                              int32_t T, const int32_t *idx, const int32_t *seg_indptr,
                              int32_t n_seg, const float *scaling, const PlanScratch &scratch,
                              int num_sms, cudaStream_t stream, int *launches)
{
    static bool attrs_set = false;
    static int occ_ustride = -1, occ_blocks = 1;
    if (!attrs_set) {
        cudaError_t e = cudaFuncSetAttribute(delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)delta_smem_bytes(kMaxRank));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)plan_smem_bytes(kMaxHash));
        if (e != cudaSuccess) return e;
        attrs_set = true;
    }
    const int ustride = (scratch.max_rank + 7) & ~7;
    const size_t dsmem = delta_smem_bytes(ustride);
    if (ustride != occ_ustride) {
        int nb = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, delta_kernel, kDT, dsmem);
        if (e != cudaSuccess) return e;
        occ_blocks = nb > 0 ? nb : 1;
        occ_ustride = ustride;
    }
    const int32_t chunk = plan_chunk(pv.max_adapters);
    const int32_t cap = scratch.cap_tokens < chunk ? scratch.cap_tokens : chunk;
    PlanLayout L = carve(scratch.base, cap, scratch.max_rank, pv.hidden, nullptr);

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    for (int32_t tb = 0; tb < T; tb += chunk) {
        const int32_t te = tb + chunk < T ? tb + chunk : T;
        const int32_t groups = (te - tb) < pv.max_adapters ? (te - tb) : pv.max_adapters;
        int hs = 1024;
        while (hs < 2 * groups && hs < kMaxHash) hs <<= 1;
        PlanArgs pa{pv, proj, idx, T, seg_indptr, n_seg, tb, te, hs, L};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPlanThreads);
        cfg.dynamicSmemBytes = plan_smem_bytes(hs);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, plan_kernel, pa);
        if (e != cudaSuccess) return e;
        *launches += 1;

        DeltaArgs da{pv, reinterpret_cast<const __half *>(x), reinterpret_cast<__half *>(y), scaling, L, ustride};
        cudaLaunchConfig_t cfg2 = {};
        cfg2.gridDim = dim3(num_sms * occ_blocks);
        cfg2.blockDim = dim3(kDT);
        cfg2.dynamicSmemBytes = dsmem;
        cfg2.stream = stream;
        cfg2.attrs = attr;
        cfg2.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg2, delta_kernel, da);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (n_seg > 0) {
        cudaError_t e = launch_prefill(pv, proj, x, y, T, idx, seg_indptr, n_seg, scaling, num_sms, stream);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaSuccess;
}

}  // namespace slora
