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
//     table (caching each adapter's directory entry in its slot) and writes the work
//     list: one item per adapter and chunk of up to 16 of its tokens, in descending rank.
//
//   delta_kernel: persistent clusters of C = ceil(hidden / 1024) CTAs; a cluster takes
//     whole items, and CTA c of the cluster owns slice c of the hidden dimension (at most
//     1024 elements): the K range of the shrink and the output columns of the expand.
//     An item runs in units of 64 rank rows:
//       shrink  partial u[t][j] = sum over the CTA's K slice of x[t][k] * At[j][k]
//       reduce  every CTA sums the C partials (read from the cluster's shared memory, in
//               CTA order) and rounds u to fp16 once
//       expand  acc[t][c] += sum_j u[t][j] * B[j][c] over the CTA's columns
//     then y[t][c] = y0[t][c] + s * acc[t][c].  A producer warp streams the row slices
//     (the tokens' x rows, A^T rows, y0 rows, B rows) with 1-D bulk copies into a ring of
//     16-row stages; eight consumer warps contract them on the tensor cores with
//     warp-level mma.sync m16n8k16 (fp16 operands, fp32 accumulators; tokens on M),
//     running the shrink of unit u before the expand of unit u-1 so that the wait for the
//     cluster's partials overlaps useful work; a signal warp relays the "partials
//     written / read" events to the cluster.  Each page row is read once per item; the
//     cluster exchanges only the small fp32 partials.  Every wait is bounded in time.
//
// One call may cover several projections of a layer (q, k, v, o: the same tokens and
// adapters, each projection with its own pages, x and y).  The plan is made once; the
// delta kernel's work list is every (item, projection) pair, item-major, so the pairs
// keep the plan's descending-cost order and the clusters share them out as they would
// the items of one projection.
//
// A token's arithmetic is fixed by the fragment layout, the slice boundaries and the CTA
// order of the partial sum, never by the other tokens of its item or the other
// projections of the call, so results do not depend on the batch, its order, the
// physical pages, or how the projections are grouped into calls.
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"
#include "tcgen05.h"

namespace slora {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;   // consumer threads
constexpr int kThreads = kConsumers + 64;         // plus a producer warp and a signal warp
constexpr int kTok = 16;                          // tokens per item: the MMA's M
constexpr int kMaxSlice = 1024;                   // elements of hidden per CTA
constexpr int kMaxCluster = 8;
constexpr int kRC = 64;                           // rank rows per rank chunk (unit)
constexpr int NST = 4;                            // ring depth (16-row stages)
constexpr int kUPitch = kRC + 8;                  // halves per token row of the u buffer
constexpr int kMaxRank = 1024;

constexpr int kPlanThreads = 1024;       // threads of the plan kernel (256 for batches of <= 256 tokens)
constexpr int kPlanThreadsSmall = 256;
constexpr int kMaxPlanTokens = 16384;   // token-index range per plan when groups fit
constexpr int kMaxPlanGroups = 2048;    // distinct adapters per plan
constexpr int kMaxHash = 2 * kMaxPlanGroups;

static_assert(kRC / 16 <= kConsumerWarps, "one shrink block per consumer warp and rank chunk");
// per-warp K-split partials of a unit's shrink: ksplit = warps / nb parts of 16 x 16 nb,
// at most 16 x 16 x (number of warps) floats whatever the unit's size
constexpr int kPtmpFloats = kTok * 16 * kConsumerWarps;

struct PlanHeader {
    int32_t n_groups, n_items, pad0, pad1;
    int32_t seg_lo, seg_hi, pad2, pad3;
};
// One work item: an adapter and up to kTok of its tokens, with the group's fields.
struct alignas(16) Item {
    int32_t t0, nt;     // first token (position within the group), tokens (<= kTok)
    int32_t rank;
    int32_t tok_begin;  // the group's first position in tok_order
    int32_t adapter;
    float scaling;
    int64_t pt_base;    // arena index of the adapter's page tables (projection 0's)
};
static_assert(sizeof(Item) == 32, "Item layout");

struct PlanLayout {
    PlanHeader *hdr;
    int32_t *tok_order;
    Item *items;
    int64_t cap_items;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tokens one plan covers: the whole range up to kMaxPlanTokens when every adapter id fits
// the plan's group tables, otherwise chunks of kMaxPlanGroups tokens.
inline int32_t plan_chunk(int32_t max_adapters)
{
    return max_adapters <= kMaxPlanGroups ? kMaxPlanTokens : kMaxPlanGroups;
}

PlanLayout carve(void *base, int32_t cap_tokens, size_t *total)
{
    PlanLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return (char *)base + o;
    };
    const int64_t cap = cap_tokens;
    L.cap_items = cap;
    L.hdr = (PlanHeader *)take(sizeof(PlanHeader));
    L.tok_order = (int32_t *)take(cap * 4);
    L.items = (Item *)take(L.cap_items * sizeof(Item));
    if (total)
        *total = off;
    return L;
}

// ---- block-wide exclusive scans -------------------------------------------------------
// N exclusive scans of one int per thread at once; wt: shared int[33][N]; every thread
// gets the block totals.
template <int N>
__device__ __forceinline__ void block_excl_scan(const int (&v)[N], int (*wt)[N], int (&excl)[N], int (&total)[N])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        incl[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int n = __shfl_up_sync(0xffffffffu, incl[i], o);
            if (lane >= o) incl[i] += n;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            wt[warp][i] = incl[i];
    }
    __syncthreads();
    if (warp == 0) {
        const bool have = lane < (int)(blockDim.x >> 5);
        int w[N], wi[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            wi[i] = w[i] = have ? wt[lane][i] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int n = __shfl_up_sync(0xffffffffu, wi[i], o);
                if (lane >= o) wi[i] += n;
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i) {
            wt[lane][i] = wi[i] - w[i];   // exclusive prefix of warp totals
            if (lane == 31) wt[32][i] = wi[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        excl[i] = wt[warp][i] + incl[i] - v[i];
        total[i] = wt[32][i];
    }
    __syncthreads();
}

struct PlanArgs {
    PoolView pv;
    const int32_t *idx;
    int32_t T;
    const int32_t *seg_indptr;
    int32_t n_seg;
    int32_t t_begin, t_end;
    int32_t hash_size;  // power of two >= 2 * min(t_end - t_begin, max_adapters), <= kMaxHash
    int32_t dir_cache;  // the directory (max_adapters entries) is copied into shared memory
    PlanLayout L;
};

constexpr int kRankBuckets = 11;        // floor(log2(rank)) for ranks 1..1024

// group page-table bases + three int hash tables + seven int group tables + two short
// token tables
constexpr size_t plan_smem_bytes(int hs)
{
    return (size_t)kMaxPlanGroups * 8 + (size_t)hs * 12 + (size_t)7 * kMaxPlanGroups * 4 + (size_t)kMaxPlanTokens * 4;
}
// directories of at most this many adapters are copied into the plan's shared memory
constexpr int kPlanDirCache = 2048;

__device__ __forceinline__ void plan_refuse(const PlanArgs &a)
{
    set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
    a.L.hdr->n_groups = 0;
    a.L.hdr->n_items = 0;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) plan_kernel(const __grid_constant__ PlanArgs a)
{
    extern __shared__ __align__(16) int plan_smem[];
    const int HS = a.hash_size;
    const int Tc = a.t_end - a.t_begin;
    long long *gpt = reinterpret_cast<long long *>(plan_smem);              // [G] page-table base
    int *keys = reinterpret_cast<int *>(gpt + kMaxPlanGroups);             // [HS] adapter id / -1
    int *hgrp = keys + HS;                                                 // [HS] group of the slot
    int *hcnt = hgrp + HS;                                                 // [HS] tokens of the slot
    int *gad = hcnt + HS;                                                  // [G] adapter
    int *grank = gad + kMaxPlanGroups;                                     // [G] rank
    float *gscale = reinterpret_cast<float *>(grank + kMaxPlanGroups);     // [G] scaling
    int *gslot = reinterpret_cast<int *>(gscale + kMaxPlanGroups);         // [G] hash slot
    int *gtok = gslot + kMaxPlanGroups;                                    // [G] first token position
    int *pit = gtok + kMaxPlanGroups;                                      // [position] first item
    int *gperm = pit + kMaxPlanGroups;                                     // [position] group, by rank descending
    short *tslot = reinterpret_cast<short *>(gperm + kMaxPlanGroups);      // [Tc] hash slot of the token (-1: none)
    short *tpos = tslot + kMaxPlanTokens;                                  // [Tc] the token's place within its group
    DirEntry *sdir = reinterpret_cast<DirEntry *>(tpos + kMaxPlanTokens);  // [max_adapters] when dir_cache
    __shared__ int warp_tot2[33][2];
    __shared__ int s_lo, s_hi, s_G, s_nit;
    __shared__ int s_bucket[kRankBuckets + 1], s_bcur[kRankBuckets + 1];
    const int tid = threadIdx.x, lane = tid & 31;

    griddep_launch_dependents();
    griddep_wait();

    // the first NT tokens' adapter ids and (small) directories are fetched at once, beside
    // the segment bounds, so the hash below waits for one round trip instead of three
    const int ad_first = tid < Tc ? a.idx[a.t_begin + tid] : -1;
    if (a.dir_cache) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.pv.dir);
        uint4 *dst = reinterpret_cast<uint4 *>(sdir);
        for (int i = tid; i < a.pv.max_adapters; i += NT) dst[i] = src[i];
    }
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
        s_G = 0;
    }
    if (tid <= kRankBuckets) {
        s_bucket[tid] = 0;
        s_bcur[tid] = 0;
    }
    for (int h = tid; h < HS; h += NT) {
        keys[h] = -1;
        hcnt[h] = 0;
    }
    __syncthreads();
    const int lo = s_lo, hi = s_hi;

    // 1. hash the decode tokens of [t_begin, t_end) by adapter.  The thread that claims a
    //    slot numbers the group and fills its fields from the adapter's directory entry;
    //    every token learns its place within its group (one atomic per warp and group).
    for (int i0 = 0; i0 < Tc; i0 += NT) {
        const int i = i0 + tid;
        int slot = -1;
        if (i < Tc) {
            const int t = a.t_begin + i;
            const bool in_seg = t >= lo && t < hi;
            const int ad = i0 == 0 ? ad_first : a.idx[t];
            if (ad >= 0 && ad < a.pv.max_adapters) {
                const DirEntry e = a.dir_cache ? sdir[ad] : a.pv.dir[ad];
                const bool resident = e.pt_off >= 0 && e.rank > 0 && e.rank <= kMaxRank;
                // segment tokens run on the tensor-core prefill path unless their adapter's
                // rank is too large for it; errors of segment tokens are reported there
                const bool mine = !in_seg || (resident && e.rank > kMaxPrefillRank);
                if (mine) {
                    if (resident) {
                        int h = (int)(((uint32_t)ad * 2654435761u) & (uint32_t)(HS - 1));
                        for (int probe = 0; probe < HS; ++probe) {
                            const int k = atomicCAS(&keys[h], -1, ad);
                            if (k == -1) {
                                const int g = atomicAdd(&s_G, 1);
                                hgrp[h] = g;
                                if (g < kMaxPlanGroups) {
                                    gad[g] = ad;
                                    grank[g] = e.rank;
                                    gscale[g] = e.scaling;
                                    gpt[g] = e.pt_off;
                                    gslot[g] = h;
                                    atomicAdd(&s_bucket[31 - __clz(e.rank)], 1);
                                }
                            }
                            if (k == -1 || k == ad) { slot = h; break; }
                            h = (h + 1) & (HS - 1);
                        }
                        // a full table cannot happen with the host's chunking (HS >= 2 x groups)
                    } else {
                        set_status(a.pv.status, SLORA_DEV_NOT_RESIDENT);
                    }
                }
            } else if (ad != -1 && !in_seg) {
                set_status(a.pv.status, SLORA_DEV_BAD_ADAPTER);
            }
        }
        // the token's place within its group: lanes with the same slot share one atomic
        const uint32_t same = __match_any_sync(0xffffffffu, slot);
        const int leader = __ffs(same) - 1;
        int base = 0;
        if (slot >= 0 && lane == leader) base = atomicAdd(&hcnt[slot], __popc(same));
        base = __shfl_sync(0xffffffffu, base, leader);
        if (i < Tc) {
            tslot[i] = (short)slot;
            tpos[i] = (short)(base + __popc(same & ((1u << lane) - 1u)));
        }
    }
    __syncthreads();
    const int G = s_G;
    if (G > kMaxPlanGroups) {
        // cannot happen with the host's chunking; refuse the batch rather than overrun
        if (tid == 0) plan_refuse(a);
        return;
    }

    // 2. groups in descending-rank order (a counting sort on floor(log2(rank)))
    {
        int start[kRankBuckets];
        int acc = 0;
#pragma unroll
        for (int b = kRankBuckets - 1; b >= 0; --b) {
            start[b] = acc;
            acc += s_bucket[b];
        }
        for (int g = tid; g < G; g += NT) {
            const int b = 31 - __clz(grank[g]);
            int st = 0;
#pragma unroll
            for (int bb = 0; bb < kRankBuckets; ++bb)
                if (bb == b) st = start[bb];
            gperm[st + atomicAdd(&s_bcur[b], 1)] = g;
        }
    }
    __syncthreads();

    // 3. per-group offsets (tokens, items) in that order
    const int per_g = ceil_div(G > 0 ? G : 1, NT);
    const int p0 = tid * per_g;
    int mine[2] = {0, 0};
    for (int q = 0; q < per_g && p0 + q < G; ++q) {
        const int n = hcnt[gslot[gperm[p0 + q]]];
        mine[0] += n;
        mine[1] += ceil_div(n, kTok);
    }
    int off[2], tot[2];
    block_excl_scan<2>(mine, warp_tot2, off, tot);
    for (int q = 0; q < per_g && p0 + q < G; ++q) {
        const int g = gperm[p0 + q];
        const int n = hcnt[gslot[g]];
        gtok[g] = off[0];
        pit[p0 + q] = off[1];
        off[0] += n;
        off[1] += ceil_div(n, kTok);
    }
    if (tid == 0) s_nit = tot[1];
    __syncthreads();
    const int n_items = s_nit;
    if ((int64_t)n_items > a.L.cap_items) {
        if (tid == 0) plan_refuse(a);
        return;
    }

    // 4. items, in parallel over items (each finds its group position by binary search over
    //    the strictly increasing first-item offsets), and the token order
    for (int i = tid; i < n_items; i += NT) {
        int lo_p = 0, hi_p = G - 1;
        while (lo_p < hi_p) {
            const int mid = (lo_p + hi_p + 1) >> 1;
            if (pit[mid] <= i) lo_p = mid; else hi_p = mid - 1;
        }
        const int g = gperm[lo_p];
        const int tc = i - pit[lo_p];
        Item it;
        it.t0 = tc * kTok;
        it.nt = min(kTok, hcnt[gslot[g]] - it.t0);
        it.rank = grank[g];
        it.tok_begin = gtok[g];
        it.adapter = gad[g];
        it.scaling = gscale[g];
        it.pt_base = gpt[g];
        const uint4 *src4 = reinterpret_cast<const uint4 *>(&it);
        uint4 *dst4 = reinterpret_cast<uint4 *>(a.L.items + i);
        dst4[0] = src4[0];
        dst4[1] = src4[1];
    }
    for (int i = tid; i < Tc; i += NT) {
        const int h = tslot[i];
        if (h >= 0)
            a.L.tok_order[gtok[hgrp[h]] + tpos[i]] = a.t_begin + i;
    }
    if (tid == 0) {
        a.L.hdr->n_groups = G;
        a.L.hdr->n_items = n_items;
        a.L.hdr->seg_lo = lo;
        a.L.hdr->seg_hi = hi;
    }
}

// ---------------------------------------------------------------------------------------
// delta kernel

struct DeltaArgs {
    PoolView pv;
    const __half *x[kMaxApplyProj];   // per projection of the call
    __half *y[kMaxApplyProj];
    int32_t proj[kMaxApplyProj];
    int32_t n_proj;                   // projections of the call
    const float *scaling;   // optional override [max_adapters]
    PlanLayout L;
    int32_t pitch;          // bytes per row of a stage / x / y0 buffer: 2 * largest slice + 16
};

// ---- decode-specific helpers (inline PTX) ---------------------------------------------
__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += a * b for one 16x8x16 tile: fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The k-th item of this cluster: rounds of ncl items, walked in alternating direction so
// that the costliest items (the list is ordered by rank, descending) spread evenly over
// the clusters.
__device__ __forceinline__ int cluster_item(int k, int cl, int ncl)
{
    return k * ncl + ((k & 1) ? (ncl - 1 - cl) : cl);
}

// Balanced item order for batches of at most kBalRounds rounds of items over at most 64
// clusters: round 0 gives item c to cluster c; every later round gives its costliest item
// to the least loaded cluster, the next to the next least loaded, and so on (cost: the
// rows of A^T, B, x, y0 and y the item moves).  Every CTA of the grid computes the same
// order, so each item is still processed by exactly one cluster.
constexpr int kBalRounds = 4;
constexpr int kBalClusters = 64;

// Ascending bitonic sort of 64 keys held two per lane (element lane and lane + 32).
__device__ __forceinline__ void warp_sort64(int &a, int &b, int lane)
{
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j == 32) {
                const int lo = min(a, b), hi = max(a, b);
                a = lo;
                b = hi;
            } else {
                const int pa = __shfl_xor_sync(0xffffffffu, a, j), pb = __shfl_xor_sync(0xffffffffu, b, j);
                const bool low = (lane & j) == 0;
                const bool upa = (lane & k) == 0, upb = ((lane + 32) & k) == 0;
                a = (low == upa) ? min(a, pa) : max(a, pa);
                b = (low == upb) ? min(b, pb) : max(b, pb);
            }
        }
    }
}

// One warp: this cluster's work entries of rounds 1 .. kBalRounds-1 into seq[] (n_items =
// none).  Entry i is item i / np of the plan for projection slot i % np.
__device__ void balance_items(const Item *items, int n_items, int np, int ncl, int cl, int lane, int *seq,
                              int *cost, int *load)
{
    for (int i = lane; i < kBalRounds * kBalClusters; i += 32) {
        int c = 0;
        if (i < n_items) c = 4 * __ldcg(&items[i / np].rank) + 3 * __ldcg(&items[i / np].nt);
        cost[i] = c;
    }
    for (int r = lane; r < kBalRounds; r += 32) seq[r] = n_items;
    __syncwarp();
    for (int c = lane; c < kBalClusters; c += 32) load[c] = c < ncl && c < n_items ? cost[c] : 0;
    __syncwarp();
    for (int r = 1; r < kBalRounds; ++r) {
        const int base = r * ncl;
        if (base >= n_items) break;
        const int nb = min(ncl, n_items - base);
        // items of the round, costliest first (ties: lower position first)
        int ia = lane < nb ? -(cost[base + lane] * 1024 + (1023 - lane)) : INT_MAX;
        int ib = lane + 32 < nb ? -(cost[base + lane + 32] * 1024 + (1023 - lane - 32)) : INT_MAX;
        warp_sort64(ia, ib, lane);
        // clusters, least loaded first (ties: lower cluster first)
        int ca = lane < ncl ? load[lane] * 256 + lane : INT_MAX;
        int cb = lane + 32 < ncl ? load[lane + 32] * 256 + lane + 32 : INT_MAX;
        warp_sort64(ca, cb, lane);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int pos = lane + 32 * h;
            const int ik = h ? ib : ia, ck = h ? cb : ca;
            if (pos < nb) {
                const int key = -ik, c = ck & 255;
                load[c] += key / 1024;
                if (c == cl) seq[r] = base + (1023 - key % 1024);
            }
        }
        __syncwarp();
    }
}

__device__ __forceinline__ Item load_item(const Item *p)
{
    const uint4 *s = reinterpret_cast<const uint4 *>(p);
    const uint4 w0 = __ldcg(s), w1 = __ldcg(s + 1);
    Item it;
    it.t0 = (int32_t)w0.x;
    it.nt = (int32_t)w0.y;
    it.rank = (int32_t)w0.z;
    it.tok_begin = (int32_t)w0.w;
    it.adapter = (int32_t)w1.x;
    it.scaling = __uint_as_float(w1.y);
    it.pt_base = (int64_t)(((uint64_t)w1.w << 32) | w1.z);
    return it;
}

__global__ void __launch_bounds__(kThreads, 1) delta_kernel(const __grid_constant__ DeltaArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int P = a.pitch;
    const int stageB = kTok * P;                                                 // one 16-row stage
    uint8_t *ring = smem;                                                        // [NST][16][P]
    uint8_t *xbuf = ring + NST * stageB;                                         // [2][16][P] x rows, by item parity
    float *part = reinterpret_cast<float *>(xbuf + 2 * stageB);                  // [2][16][kRC] partial u, by unit parity
    float *ptmp = part + 2 * kTok * kRC;                                         // [ksplit][16][16 nb] per-warp partials
    __half *ubuf = reinterpret_cast<__half *>(ptmp + kPtmpFloats);               // [16][kUPitch] u (fp16)
    Item *rec_it = reinterpret_cast<Item *>(ubuf + kTok * kUPitch);              // [2] item, by item parity
    int32_t *rec_tok = reinterpret_cast<int32_t *>(rec_it + 2);                 // [2][kTok] token ids
    int32_t *rec_pj = rec_tok + 2 * kTok;                                        // [2] projection slot
    uint64_t *bars = reinterpret_cast<uint64_t *>(rec_pj + 2);
    uint64_t *full = bars, *empty = bars + NST;
    uint64_t *full_x = bars + 2 * NST;   // [2] an item's x rows (and record) landed
    uint64_t *xfree = full_x + 2;        // [2] an item's shrink no longer reads its x rows
    uint64_t *ready = full_x + 4;        // [2] every CTA of the cluster wrote its partials of a unit
    uint64_t *consumed = full_x + 6;     // [2] every CTA of the cluster has read the partials of a unit
    uint64_t *done = full_x + 8;         // every CTA of the cluster is finished with the others' memory
    uint64_t *pwrit = full_x + 9;        // [2] this CTA's partials of a unit are written (local)
    uint64_t *rdone = full_x + 11;       // [2] this CTA has read the cluster's partials of a unit (local)
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.pv.hidden;
    const uint32_t crank = cluster_ctarank(), C = cluster_nctarank();
    const int cl = (int)cluster_id_x(), ncl = (int)ncluster_x();
    __shared__ int s_seq[kBalRounds], s_cost[kBalRounds * kBalClusters], s_load[kBalClusters];
    __shared__ __align__(8) uint64_t seq_bar;
    // this CTA's slice of the hidden dimension, in whole 16-element steps
    const int nk16 = d / 16;
    const int kb = 16 * (int)((crank * (uint32_t)nk16) / C);
    const int KS = 16 * (int)(((crank + 1) * (uint32_t)nk16) / C) - kb;
    const uint32_t sliceB = (uint32_t)KS * 2;
    int32_t *status = a.pv.status;
    volatile int *abort = &s_abort;
    const uint32_t ring_s = smem_u32(ring), xbuf_s = smem_u32(xbuf);
    const uint32_t ubuf_s = smem_u32(ubuf);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&full_x[b], 1);
            mbar_init(&xfree[b], 1);
            mbar_init(&ready[b], C);
            mbar_init(&consumed[b], C);
        }
        mbar_init(done, C);
        mbar_init(&seq_bar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pwrit[b], 1);
            mbar_init(&rdone[b], 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    cluster_sync_all();   // every CTA's barriers exist before any remote arrival
    griddep_wait();       // the plan of this batch is complete and visible
    griddep_launch_dependents();
    const int NP = a.n_proj;
    const int n_items = a.L.hdr->n_items * NP;   // (item, projection) entries
    const bool bal = n_items <= kBalRounds * ncl && ncl <= kBalClusters;
    // the index of this cluster's k-th item (n_items or more: no more items)
    auto item_of = [&](int k) -> int {
        if (!bal) return cluster_item(k, cl, ncl);
        if (k == 0) return cl;
        if (k >= kBalRounds || k * ncl >= n_items) return n_items;
        wait_phase<false>(&seq_bar, 0, abort, status);
        return s_seq[k];
    };

    // Work runs in units: one chunk of at most kRC rank rows of an item.  Both sides walk
    // the units in the same order and interleave them one unit apart (the shrink of unit
    // u, then the expand of unit u-1), so the wait for the cluster's partials of a unit
    // overlaps the next unit's shrink.

    if (warp == kConsumerWarps + 1) {
        // ================================ signal warp ================================
        // Relays this CTA's "partials written" and "partials read" events of every unit to
        // the cluster (lane c arrives, release at cluster scope, on CTA c's barrier).  The
        // warp writes no global memory, so its releases only order the shared-memory
        // writes it has observed through the local barriers.
        int k = -1, c = 0, nch = 0;
        uint32_t u = 0;
        for (;;) {
            bool have = true;
            if (c == nch) {
                ++k;
                const int i = item_of(k);
                if (i >= n_items) {
                    have = false;
                } else {
                    c = 0;
                    nch = ceil_div(__ldcg(&a.L.items[i / NP].rank), kRC);
                }
            }
            if (have) {
                wait_phase<false>(&pwrit[u & 1], (u >> 1) & 1, abort, status);
                if (lane < (int)C) mbar_arrive_remote(mapa(smem_u32(&ready[u & 1]), lane));
            }
            if (u >= 1) {
                const uint32_t pu = u - 1;
                wait_phase<false>(&rdone[pu & 1], (pu >> 1) & 1, abort, status);
                if (lane < (int)C) mbar_arrive_remote(mapa(smem_u32(&consumed[pu & 1]), lane));
            }
            if (!have) break;
            ++c;
            ++u;
        }
        // the CTA is done reading the others' partials once its last unit was reduced
        if (lane < (int)C) mbar_arrive_remote(mapa(smem_u32(done), lane));
        if (lane == 0) wait_phase<true>(done, 0, abort, status);
        return;
    }

    if (warp == kConsumerWarps) {
        // ===================================== producer =====================================
        const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);
        uint32_t sc = 0;   // stages issued
        // Lane r < 16 copies the CTA's slice of row r from src_r (when ok_r) into a 16-row
        // buffer at dst; rows not copied are zero-filled when zero_rest.  Completion on *bar.
        auto fill16 = [&](uint32_t dst, uint64_t *bar, const __half *src_r, bool ok_r, bool zero_rest) {
            const bool mine = ok_r && lane < 16;
            const uint32_t m = __ballot_sync(0xffffffffu, mine);
            if (mine && !*abort)
                bulk_g2s_s(dst + lane * P, src_r + kb, sliceB, bar);
            if (zero_rest && m != 0xffffu) {
                for (int r = 0; r < 16; ++r) {
                    if ((m >> r) & 1u) continue;
                    for (uint32_t o = lane * 16; o < sliceB; o += 32 * 16)
                        *reinterpret_cast<uint4 *>(smem + (dst - ring_s) + r * P + o) = make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();   // before later bulk copies land in the same rows
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(bar, *abort ? 0u : (uint32_t)__popc(m) * sliceB);
        };
        auto next_slot = [&]() -> uint32_t {
            const uint32_t slot = sc % NST;
            if (sc >= NST) wait_phase<false>(&empty[slot], ((sc / NST) - 1) & 1, abort, status);
            return slot;
        };
        auto page_ok = [&](int32_t pg) -> bool {
            if (pg >= 0 && pg < a.pv.num_pages) return true;
            set_status(status, SLORA_DEV_BAD_PAGE);
            return false;
        };
        // the 16-row blocks of a unit: rows rc0 .. rc0+rows-1 of A^T (ab 0) or B (ab 1);
        // lane l holds the page indices of the unit's rows l + 32m in pg4[m]
        auto emit_blocks = [&](int rows, const int32_t (&pg4)[4], bool zero_rest) {
            const int nb = ceil_div(rows, 16);
            for (int b = 0; b < nb; ++b) {
                const uint32_t slot = next_slot();
                const int src_lane = 16 * (b & 1) + (lane & 15);   // rows 16b+l live in lane 16(b&1)+l, word b/2
                int32_t pg = -1;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int v = __shfl_sync(0xffffffffu, pg4[m], src_lane);
                    if (m == (b >> 1)) pg = v;
                }
                const bool ok = 16 * b + (lane & 15) < rows && pg >= 0 && page_ok(pg);
                fill16(ring_s + slot * stageB, &full[slot], pool + (int64_t)(ok ? pg : 0) * d, ok, zero_rest);
                ++sc;
            }
        };
        int k = -1, c = 0, nch = 0;      // current unit: item ordinal, rank chunk, chunks of the item
        Item it{};
        int ipj = 0;                     // projection slot of the current item
        int tl = 0;                      // lane l: token id of the item's token l & 15
        bool tv = false;
        bool have_prev = false;          // previous unit, whose expand data follows
        Item pit{};
        int pc = 0, ptl = 0, ppj = 0;
        bool ptv = false;
        int32_t ppb[4] = {-1, -1, -1, -1};
        // The next item's metadata is fetched ahead in two steps, its record while the
        // current item's A^T rows go out, then its tokens and the page-table entries of its
        // first unit after the previous unit's B rows, so an item boundary waits for no load.
        bool nvalid = false;
        Item nit{};
        int ntok = 0, npj = 0;
        int32_t npa[4] = {-1, -1, -1, -1}, npb[4] = {-1, -1, -1, -1};
        auto fetch_record = [&](int kk) {
            const int i = item_of(kk);
            nvalid = i < n_items;
            if (nvalid) {
                nit = load_item(a.L.items + i / NP);   // not used before fetch_rest: no wait here
                npj = i % NP;
            }
        };
        auto fetch_rest = [&]() {
            if (!nvalid) return;
            nit.pt_base += (int64_t)a.proj[npj] * 2 * nit.rank;   // this projection's page table
            ntok = lane < nit.nt ? __ldcg(a.L.tok_order + nit.tok_begin + nit.t0 + lane) : 0;
            const int rows = min(kRC, nit.rank);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = lane + 32 * m;
                npa[m] = -1;
                npb[m] = -1;
                if (r < rows) {
                    npa[m] = __ldcg(a.pv.pt_arena + nit.pt_base + r);
                    npb[m] = __ldcg(a.pv.pt_arena + nit.pt_base + nit.rank + r);
                }
            }
        };
        fetch_record(0);
        fetch_rest();
        for (;;) {
            bool have = true;
            bool fresh = false;          // the unit is its item's first: its entries came ahead
            if (c == nch) {
                ++k;
                if (!nvalid) {
                    have = false;
                } else {
                    it = nit;
                    ipj = npj;
                    const int tok = ntok;
                    tl = __shfl_sync(0xffffffffu, tok, lane & 15);
                    tv = (lane & 15) < it.nt;
                    c = 0;
                    nch = ceil_div(it.rank, kRC);
                    fresh = true;
                    // the item's record and x rows, once item k-2's shrink is done with buffer k&1
                    if (k >= 2) wait_phase<false>(&xfree[k & 1], ((k >> 1) - 1) & 1, abort, status);
                    if (lane == 0) {
                        rec_it[k & 1] = it;
                        rec_pj[k & 1] = ipj;
                    }
                    if (lane < kTok) rec_tok[(k & 1) * kTok + lane] = tok;
                    fill16(xbuf_s + (k & 1) * stageB, &full_x[k & 1], a.x[ipj] + (int64_t)tl * d, tv, false);
                }
            }
            int32_t pb[4] = {-1, -1, -1, -1};
            if (have) {
                // shrink data of the unit: its A^T rows
                const int rc0 = c * kRC, rows = min(kRC, it.rank - rc0);
                int32_t pa[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int r = lane + 32 * m;
                    if (fresh) {
                        pa[m] = npa[m];
                        pb[m] = npb[m];
                    } else {
                        pa[m] = -1;
                        if (r < rows) {
                            pa[m] = __ldcg(a.pv.pt_arena + it.pt_base + rc0 + r);
                            pb[m] = __ldcg(a.pv.pt_arena + it.pt_base + it.rank + rc0 + r);
                        }
                    }
                }
                emit_blocks(rows, pa, false);
                if (fresh) fetch_record(k + 1);
            }
            if (have_prev) {
                // expand data of the previous unit: the item's y0 rows (first unit) and B rows
                if (pc == 0) {
                    const uint32_t slot = next_slot();
                    fill16(ring_s + slot * stageB, &full[slot], a.y[ppj] + (int64_t)ptl * d, ptv, false);
                    ++sc;
                }
                emit_blocks(min(kRC, pit.rank - pc * kRC), ppb, true);
            }
            if (have && fresh) fetch_rest();
            if (!have) break;
            have_prev = true;
            pit = it;
            pc = c;
            ptl = tl;
            ptv = tv;
            ppj = ipj;
#pragma unroll
            for (int m = 0; m < 4; ++m) ppb[m] = pb[m];
            ++c;
        }
        return;
    }

    // ===================================== consumers =====================================
    const int w = warp;
    if (w == 0 && bal && n_items > ncl) {
        // while the first data is in flight
        balance_items(a.L.items, n_items, NP, ncl, cl, lane, s_seq, s_cost, s_load);
        __syncwarp();
        if (lane == 0) mbar_arrive(&seq_bar);
    }
    const int q = lane >> 3, rr = lane & 7, gid = lane >> 2, tig = lane & 3;
    // this warp's output columns in the expand: column pairs [pp0, pp1) of 16 columns
    const int npair = KS / 16;
    const int pp0 = (w * npair) / kConsumerWarps, pp1 = ((w + 1) * npair) / kConsumerWarps;
    uint32_t sc = 0;    // stages consumed
    uint32_t un = 0;    // units shrunk
    int k = -1, c = 0, nch = 0;
    Item it{};
    int ipj = 0;                        // projection slot of the current item
    int tk[2] = {0, 0};                 // token ids of rows gid, gid+8 of the current item
    bool have_prev = false;
    Item pit{};
    int pc = 0, ppj = 0, ptk[2] = {0, 0};
    float acc[16][4];
    uint32_t yv[2][16];                 // y0 of the item being expanded: [token half][n-block], half2 bits
#pragma unroll
    for (int n8 = 0; n8 < 16; ++n8)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[n8][e] = 0.f;
    for (;;) {
        bool have = true;
        if (c == nch) {
            ++k;
            const int i = item_of(k);
            if (i >= n_items) {
                have = false;
            } else {
                wait_phase<false>(&full_x[k & 1], (k >> 1) & 1, abort, status);
                it = rec_it[k & 1];
                ipj = rec_pj[k & 1];
                tk[0] = rec_tok[(k & 1) * kTok + gid];
                tk[1] = rec_tok[(k & 1) * kTok + gid + 8];
                c = 0;
                nch = ceil_div(it.rank, kRC);
            }
        }
        if (have) {
            // ---- shrink of unit un: block b (16 rank rows) of the unit goes to warps
            //      b + nb*g, which split the CTA's K slice into ksplit = 8/nb parts ----
            const uint32_t par = un & 1;
            if (un >= 2) wait_phase<true>(&consumed[par], ((un >> 1) - 1) & 1, abort, status);
            float *mypart = part + par * (kTok * kRC);
            const uint32_t xs = xbuf_s + (k & 1) * stageB;
            const int rows = min(kRC, it.rank - c * kRC), nb = ceil_div(rows, 16);
            const int ksplit = kConsumerWarps / nb, wb = w % nb, wg = w / nb;
            const int nsteps = KS / 16;
            const int ks0 = (wg * nsteps) / ksplit, ks1 = ((wg + 1) * nsteps) / ksplit;
            for (int b = 0; b < nb; ++b) {
                const uint32_t s = sc + b, slot = s % NST;
                wait_phase<false>(&full[slot], (s / NST) & 1, abort, status);
                if (b == wb && wg < ksplit) {
                    // two accumulators per n-block (even / odd K steps) halve the MMA chains
                    float pacc[2][2][4] = {};
                    const uint32_t sb = ring_s + slot * stageB;
                    for (int st = ks0; st < ks1; st += 2) {
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            if (st + h2 < ks1) {
                                const int k16 = 16 * (st + h2);
                                uint32_t af[4], bf[4];
                                ldsm_x4(xs + (rr + 8 * (q & 1)) * P + (k16 + 8 * (q >> 1)) * 2, af);   // token rows
                                ldsm_x4(sb + (rr + 8 * (q >> 1)) * P + (k16 + 8 * (q & 1)) * 2, bf);   // A^T rows
                                mma16816(pacc[h2][0], af, bf[0], bf[1]);
                                mma16816(pacc[h2][1], af, bf[2], bf[3]);
                            }
                        }
                    }
                    const int ld = 16 * nb;
#pragma unroll
                    for (int nb8 = 0; nb8 < 2; ++nb8)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            *reinterpret_cast<float2 *>(ptmp + (wg * kTok + gid + 8 * h) * ld + 16 * b + 8 * nb8 + 2 * tig) =
                                make_float2(pacc[0][nb8][2 * h] + pacc[1][nb8][2 * h],
                                            pacc[0][nb8][2 * h + 1] + pacc[1][nb8][2 * h + 1]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            sc += nb;
            consumers_sync();   // every warp's partials are written
            {
                // this CTA's partial: the ksplit parts summed in order
                const int ld = 16 * nb;
                for (int e = tid; e < kTok * ld; e += kConsumers) {
                    const int t = e / ld, j = e - t * ld;
                    float v = 0.f;
                    for (int g = 0; g < ksplit; ++g)
                        v += ptmp[(g * kTok + t) * ld + j];
                    mypart[t * kRC + j] = v;
                }
            }
            consumers_sync();   // this CTA's partials of the unit are written
            if (tid == 0) {
                if (c == nch - 1) mbar_arrive(&xfree[k & 1]);   // the item's x rows are no longer read
                mbar_arrive(&pwrit[par]);                       // relayed to the cluster by the signal warp
            }
        }
        if (have_prev) {
            // ---- expand of unit un-1 ----
            const uint32_t pu = un - 1, ppar = pu & 1;
            const int rows = min(kRC, pit.rank - pc * kRC), nb = ceil_div(rows, 16);
            wait_phase<true>(&ready[ppar], (pu >> 1) & 1, abort, status);
            consumers_sync();   // the previous expand is done reading u
            {
                // u = sum of the C partials in CTA order, rounded to fp16 once.  A thread
                // takes up to two 4-element vectors of the unit and issues the 16-byte
                // remote loads of four CTAs at once (a second round only for clusters of
                // more than four), so the exchange costs one or two remote round trips.
                const uint32_t pbase = smem_u32(part + ppar * (kTok * kRC));
                const int vpr = 4 * nb;                 // vectors per token row
                const int nv = kTok * vpr;
                static_assert(kTok * kRC / 4 <= 2 * kConsumers, "two vectors per thread");
                float4 sum[2];
                int vt[2], vj[2];
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int e = tid + m * kConsumers;
                    vt[m] = e / vpr;
                    vj[m] = e - vt[m] * vpr;
                    sum[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int c0 = 0; c0 < kMaxCluster; c0 += 4) {
                    if (c0 >= (int)C) break;
                    float4 v[2][4];
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const bool ok = tid + m * kConsumers < nv;
                        const uint32_t off = (uint32_t)(vt[m] * kRC + vj[m] * 4) * 4;
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            v[m][cc] = (ok && c0 + cc < (int)C) ? ld_cluster_v4(mapa(pbase + off, c0 + cc))
                                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {   // CTA order; absent CTAs add zero
                            sum[m].x += v[m][cc].x;
                            sum[m].y += v[m][cc].y;
                            sum[m].z += v[m][cc].z;
                            sum[m].w += v[m][cc].w;
                        }
                }
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    if (tid + m * kConsumers < nv) {
                        const int j = vj[m] * 4;
                        __half2 h[2];
                        h[0] = __floats2half2_rn(j < rows ? sum[m].x : 0.f, j + 1 < rows ? sum[m].y : 0.f);
                        h[1] = __floats2half2_rn(j + 2 < rows ? sum[m].z : 0.f, j + 3 < rows ? sum[m].w : 0.f);
                        *reinterpret_cast<uint2 *>(ubuf + vt[m] * kUPitch + j) = *reinterpret_cast<const uint2 *>(h);
                    }
                }
            }
            consumers_sync();   // u of the unit is in place; the partials have been read
            if (tid == 0) mbar_arrive(&rdone[ppar]);   // relayed to the cluster by the signal warp
            if (pc == 0) {
                // the item's y0 rows: into registers, and a fresh accumulator
                const uint32_t slot = sc % NST;
                wait_phase<false>(&full[slot], (sc / NST) & 1, abort, status);
                const uint8_t *st = ring + slot * stageB;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int p = 0; p < 8; ++p)
#pragma unroll
                        for (int n2 = 0; n2 < 2; ++n2)
                            yv[h][2 * p + n2] = pp0 + p < pp1 ? *reinterpret_cast<const uint32_t *>(
                                                                    st + (gid + 8 * h) * P + (16 * (pp0 + p) + 8 * n2 + 2 * tig) * 2)
                                                              : 0u;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                ++sc;
#pragma unroll
                for (int n8 = 0; n8 < 16; ++n8)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[n8][e] = 0.f;
            }
            // every warp its column pairs, over the unit's B blocks
            for (int b = 0; b < nb; ++b) {
                const uint32_t s = sc + b, slot = s % NST;
                wait_phase<false>(&full[slot], (s / NST) & 1, abort, status);
                const uint32_t sb = ring_s + slot * stageB;
                uint32_t af[4];
                ldsm_x4(ubuf_s + ((rr + 8 * (q & 1)) * kUPitch + 16 * b + 8 * (q >> 1)) * 2, af);   // u rows
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    if (pp0 + p < pp1) {
                        uint32_t bf[4];
                        ldsm_x4_t(sb + (rr + 8 * (q & 1)) * P + (16 * (pp0 + p) + 8 * (q >> 1)) * 2, bf);   // B rows
                        mma16816(acc[2 * p], af, bf[0], bf[1]);
                        mma16816(acc[2 * p + 1], af, bf[2], bf[3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            sc += nb;
            if (pc == ceil_div(pit.rank, kRC) - 1 && !*abort) {
                // ---- epilogue of the item: y = y0 + s * acc over this CTA's columns ----
                const float scl = a.scaling ? a.scaling[pit.adapter] : pit.scaling;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = gid + 8 * h;
                    if (t < pit.nt) {
                        __half *yrow = a.y[ppj] + (int64_t)ptk[h] * d + kb;
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            if (pp0 + p < pp1) {
#pragma unroll
                                for (int n2 = 0; n2 < 2; ++n2) {
                                    const int col = 16 * (pp0 + p) + 8 * n2 + 2 * tig;
                                    const float2 y0 = __half22float2(*reinterpret_cast<const __half2 *>(&yv[h][2 * p + n2]));
                                    const float *ac = acc[2 * p + n2];
                                    *reinterpret_cast<__half2 *>(yrow + col) =
                                        __floats2half2_rn(fmaf(scl, ac[2 * h], y0.x), fmaf(scl, ac[2 * h + 1], y0.y));
                                }
                            }
                        }
                    }
                }
            }
        }
        if (!have) break;
        have_prev = true;
        pit = it;
        pc = c;
        ppj = ipj;
        ptk[0] = tk[0];
        ptk[1] = tk[1];
        ++c;
        ++un;
    }
    // the signal warp keeps the CTA alive until no other CTA may still read its partials
}

}  // namespace

size_t plan_scratch_bytes(int32_t T, int32_t max_rank, int32_t hidden, int32_t max_adapters)
{
    (void)max_rank;
    (void)hidden;
    size_t total = 0;
    const int32_t chunk = plan_chunk(max_adapters);
    const int32_t cap = T < chunk ? T : chunk;
    carve(nullptr, cap, &total);
    return total;
}

// CTAs per cluster for a hidden size: slices of at most kMaxSlice elements.
inline int delta_cluster(int hidden) { return ceil_div(hidden, kMaxSlice); }
inline int delta_pitch(int hidden)
{
    const int C = delta_cluster(hidden);
    return 2 * 16 * ceil_div(hidden / 16, C) + 16;
}
inline size_t delta_smem_bytes(int hidden)
{
    const size_t stage = (size_t)kTok * delta_pitch(hidden);
    return (NST + 2) * stage + 2 * (size_t)kTok * kRC * 4 + (size_t)kPtmpFloats * 4 + (size_t)kTok * kUPitch * 2 + 2 * sizeof(Item) +
           2 * kTok * 4 + 2 * 4 + (2 * NST + 13) * 8;
}

// Kernel attributes and the delta grid's resident clusters, per device (the attributes
// are per-device state; calls may come from several threads).
struct DeltaLaunchState {
    bool attrs = false;
    int occ_hidden = -1;
    int occ_clusters = 1;
};
constexpr int kMaxLaunchDevices = 64;
std::mutex g_delta_mu;
DeltaLaunchState g_delta_state[kMaxLaunchDevices];

cudaError_t launch_lora_apply(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                              const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                              const PlanScratch &scratch, int num_sms, cudaStream_t stream, int *launches,
                              cudaEvent_t after_plan)
{
    if (pv.hidden > kMaxCluster * kMaxSlice || pl.n < 1 || pl.n > kMaxApplyProj) return cudaErrorInvalidValue;
    int device = 0;
    cudaError_t de = cudaGetDevice(&device);
    if (de != cudaSuccess) return de;
    if (device < 0 || device >= kMaxLaunchDevices) return cudaErrorInvalidDevice;
    std::unique_lock<std::mutex> lk(g_delta_mu);
    DeltaLaunchState &ls = g_delta_state[device];
    if (!ls.attrs) {
        cudaError_t e = cudaFuncSetAttribute(delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)delta_smem_bytes(kMaxSlice));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(plan_kernel<kPlanThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(plan_smem_bytes(kMaxHash) + kPlanDirCache * sizeof(DirEntry)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(plan_kernel<kPlanThreadsSmall>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(plan_smem_bytes(kMaxHash) + kPlanDirCache * sizeof(DirEntry)));
        if (e != cudaSuccess) return e;
        ls.attrs = true;
    }
    const int C = delta_cluster(pv.hidden);
    const size_t dsmem = delta_smem_bytes(pv.hidden);

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;

    cudaLaunchConfig_t cfg2 = {};
    cfg2.blockDim = dim3(kThreads);
    cfg2.dynamicSmemBytes = dsmem;
    cfg2.stream = stream;
    cfg2.attrs = attr;
    cfg2.numAttrs = 2;
    if (pv.hidden != ls.occ_hidden) {
        cfg2.gridDim = dim3(C * num_sms);
        int ncl = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&ncl, delta_kernel, &cfg2);
        if (e != cudaSuccess) return e;
        ls.occ_clusters = ncl > 0 ? ncl : 1;
        ls.occ_hidden = pv.hidden;
    }
    const int occ_clusters = ls.occ_clusters;
    lk.unlock();
    cfg2.gridDim = dim3(C * occ_clusters);

    const int32_t chunk = plan_chunk(pv.max_adapters);
    const int32_t cap = scratch.cap_tokens < chunk ? scratch.cap_tokens : chunk;
    PlanLayout L = carve(scratch.base, cap, nullptr);

    for (int32_t tb = 0; tb < T; tb += chunk) {
        const int32_t te = tb + chunk < T ? tb + chunk : T;
        const int32_t groups = (te - tb) < pv.max_adapters ? (te - tb) : pv.max_adapters;
        int hs = 1024;
        while (hs < 2 * groups && hs < kMaxHash) hs <<= 1;
        const int dcache = pv.max_adapters <= kPlanDirCache ? 1 : 0;
        PlanArgs pa{pv, idx, T, seg_indptr, n_seg, tb, te, hs, dcache, L};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        const bool small = te - tb <= kPlanThreadsSmall;
        cfg.blockDim = dim3(small ? kPlanThreadsSmall : kPlanThreads);
        cfg.dynamicSmemBytes = plan_smem_bytes(hs) + (dcache ? (size_t)pv.max_adapters * sizeof(DirEntry) : 0);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = small ? cudaLaunchKernelEx(&cfg, plan_kernel<kPlanThreadsSmall>, pa)
                              : cudaLaunchKernelEx(&cfg, plan_kernel<kPlanThreads>, pa);
        if (e != cudaSuccess) return e;
        *launches += 1;

        if (after_plan && tb == 0) {
            e = cudaEventRecord(after_plan, stream);
            if (e != cudaSuccess) return e;
        }
        DeltaArgs da{};
        da.pv = pv;
        for (int j = 0; j < pl.n; ++j) {
            da.x[j] = reinterpret_cast<const __half *>(pl.x[j]);
            da.y[j] = reinterpret_cast<__half *>(pl.y[j]);
            da.proj[j] = pl.proj[j];
        }
        da.n_proj = pl.n;
        da.scaling = scaling;
        da.L = L;
        da.pitch = delta_pitch(pv.hidden);
        e = cudaLaunchKernelEx(&cfg2, delta_kernel, da);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (n_seg > 0) {
        cudaError_t e = launch_prefill(pv, pl, T, idx, seg_indptr, n_seg, scaling, num_sms, stream);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaSuccess;
}

}  // namespace slora
