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
//     table (caching each adapter's directory entry in its slot), cuts every group into
//     items of up to 8 tokens, packs small items into shared work groups, and writes the
//     work list of the delta kernel: for every work group and projection of the call, one
//     shrink unit per (hidden block, 64-row rank chunk) and one expand unit per hidden
//     block; all shrink units come first, items in descending rank.
//
//   delta_kernel: one persistent CTA per SM takes units in list order (its first by its
//     index, then from a counter in the plan), so every SM stays busy until the list ends:
//       shrink  (item, block b, chunk c): partial u[t][j] = sum over the K slice b of
//               x[t][k] * At[j][k] for the chunk's rank rows -> fp32 partials in global
//               scratch (L2), each written as one 64-bit word {value, launch tag}
//       expand  (item, block b): once every partial word of the item carries this
//               launch's tag, u = sum of the partials over the hidden blocks in block
//               order, rounded to fp16 once; acc[t][c] = sum_j u[t][j] * B[j][c] over the
//               block's columns; y[t][c] = y0[t][c] + s * acc[t][c]
//     Warp roles: a lead warp fetches the units and publishes each with its token ids and
//     first page ids; four copy warps stream the row slices (the item's token rows, then
//     A^T or B rows) into a ring of 8-row stages with 1-D bulk copies; eight consumer
//     warps contract them on the tensor cores with warp-level mma.sync m16n8k16 (fp16
//     operands, fp32 accumulators; a shrink puts rank rows on M and tokens on N, an
//     expand tokens on M and columns on N); a reduce warp sums the consumers' shrink
//     partials and writes them as tagged words; a gather warp polls and sums the partials
//     of the expand units ahead of the consumers, so no consumer waits on a global round
//     trip.  Every page row is read once per item (small items share units); the only
//     cross-SM traffic is the small tagged partials.  Every wait is bounded in time.
//
// A plan may also be made once and used by several decode launches (the layers of an
// iteration, slora_plan_apply): the last lead warp of a launch resets the unit counter, each
// launch tags its partial sums anew, and from the second launch on the lead publishes its
// CTA's first unit, and the copy warps start that unit's page rows, before the grid-dependency
// wait.
//
// Expand units only wait for shrink units that precede them in the list, and shrink
// units never wait on another SM, so the list drains whatever number of CTAs is resident.
//
// One call may cover several projections of a layer (q, k, v, o: the same tokens and
// adapters, each projection with its own pages, x and y): the plan is made once and
// lists the units of every (item, projection) pair.
//
// A token's arithmetic is fixed by the fragment layout, the hidden-block boundaries, the
// fixed split of a block's K steps over the eight consumer warps (summed in warp order)
// and the block order of the partial sum, never by the other tokens of its item, the other projections of the call
// or the SM that runs a unit, so results do not depend on the batch, its order, the
// physical pages, or how the projections are grouped into calls.
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"
#include "tcgen05.h"

namespace slora {
namespace {

constexpr int kConsumerWarps = 8;                 // warps doing the contractions
constexpr int kCopyWarps = 4;                     // warps issuing the bulk copies
constexpr int kWarpLead = kConsumerWarps;         // fetches and publishes the units
constexpr int kWarpCopy0 = kConsumerWarps + 1;    // first copy warp
constexpr int kWarpReduce = kWarpCopy0 + kCopyWarps;   // sums the consumers' shrink partials
constexpr int kWarpGather = kWarpReduce + 1;            // sums the shrink partials of the expand units ahead
constexpr int kThreads = 32 * (kWarpGather + 1);
constexpr int kRecReaders = kConsumerWarps + kCopyWarps + 2;   // warps that read every unit record
constexpr int kTok = 8;                           // tokens per item: one MMA n-tile / one ring stage
constexpr int kMaxSlice = 1024;                   // elements of a hidden block
constexpr int kMaxBlocks = 8;                     // hidden blocks (hidden <= 8192)
constexpr int kRC = 64;                           // rank rows per rank chunk
constexpr int NST = 12;                           // ring depth (8-row stages)
constexpr int QD = 8;                             // unit records in flight
constexpr int QU = 4;                             // u buffers (gather warp -> consumers)
#ifndef SLORA_CLAIM_AHEAD
#define SLORA_CLAIM_AHEAD 5
#endif
constexpr int kClaimAhead = SLORA_CLAIM_AHEAD;    // units a CTA holds beyond those it has finished
static_assert(kClaimAhead >= 2, "the consumers read the record after the one they work on");
constexpr int kUPitch = kRC + 8;                  // halves per token row of a u buffer
constexpr int kMaxRank = 1024;

constexpr int kPlanThreads = 1024;       // threads of the plan kernel (256 for batches of <= 256 tokens)
constexpr int kPlanThreadsSmall = 256;
constexpr int kMaxPlanTokens = 16384;   // token-index range per plan when groups fit
constexpr int kMaxPlanGroups = 2048;    // distinct adapters per plan
constexpr int kMaxHash = 2 * kMaxPlanGroups;

static_assert(kTok == 8, "one ring stage of token rows, one MMA n-tile of tokens");
// Copy warp g % kCopyWarps fills stage g; with NST a multiple of kCopyWarps every ring slot
// is always filled by the same warp, which saw the release of stage g - 2 NST before it
// issued stage g - NST, so the parity it waits on for stage g is never one phase behind,
// whatever order the consumers release stages in (an expand holds its token stage).
static_assert(NST % kCopyWarps == 0, "each ring slot always filled by the same copy warp");
// Per consumer warp: K steps of a shrink block, 16-column pairs of an expand block at most.
constexpr int kXs = kMaxSlice / 16 / kConsumerWarps;
constexpr int kPairs = kMaxSlice / 16 / kConsumerWarps;
// A consumer warp's scratch region: a shrink unit's partial (8 tokens x 64 rank rows), summed
// by the reduce warp, or the y0 values of an expand unit of more than 64 rank rows (2 kPairs
// n-tiles x 32 lanes, half2 each).
constexpr int kRegionFloats = kTok * kRC;
static_assert(2 * kPairs * 32 <= kRegionFloats, "y0 values fit a region");
constexpr int kPtmpFloats = kRegionFloats * kConsumerWarps;

struct PlanHeader {
    int32_t n_groups, n_wg, n_units, n_shrink;   // n_wg: work groups (own items and packs)
    int32_t seg_lo, seg_hi;
    int32_t grab;    // the delta kernel's unit counter (0 before a launch)
    int32_t exits;   // lead warps of the running delta launch that have taken their last unit
};

// Items (an adapter and up to kTok of its tokens) share a unit when they are small: the
// last item of a group, of at most kPackTokens tokens and rank at most 2 kSlot, is
// packable; packable items of rank <= kSlot fill kPackItems 16-row slots of one unit,
// those of rank kSlot+1 .. 2 kSlot two 32-row slots.  Every item starts on a multiple of
// 16 rows, so its K steps in the expand line up as in a unit of its own, and rows of
// other items only add exact zeros to its sums.
constexpr int kPackItems = 4;
constexpr int kPackTokens = 2;
constexpr int kSlot = 16;
static_assert(kPackItems * kPackTokens <= kTok && kPackItems * kSlot == kRC, "a full pack fits one unit");

// One item of a unit.
struct PackItem {
    int64_t pt_base;    // arena index of the projection's page table (A^T rows, then B rows)
    int32_t tok_start;  // first position of the item's tokens in tok_order
    uint32_t geo;       // bits 0-6 first row in the unit, 7-17 rank, 18-20 first token in the
                        // unit, 21-23 tokens - 1
    float scaling;      // the adapter's scaling (the call's override applied)
    int32_t uoff;       // first word of the (item, projection)'s partials
};
static_assert(sizeof(PackItem) == 24, "PackItem layout");

__host__ __device__ inline uint32_t geo_pack(int row0, int rank, int t0, int nt)
{
    return (uint32_t)row0 | ((uint32_t)rank << 7) | ((uint32_t)t0 << 18) | ((uint32_t)(nt - 1) << 21);
}
__host__ __device__ inline int geo_row0(uint32_t g) { return (int)(g & 127u); }
__host__ __device__ inline int geo_rank(uint32_t g) { return (int)((g >> 7) & 2047u); }
__host__ __device__ inline int geo_t0(uint32_t g) { return (int)((g >> 18) & 7u); }
__host__ __device__ inline int geo_nt(uint32_t g) { return (int)((g >> 21) & 7u) + 1; }

// A unit as the delta kernel's warps see it: a shrink or an expand unit of one work group
// (an item of its own, or a pack of items) and one projection of the call.  The plan writes
// the work groups in this form for projection slot 0 with no unit fields (page-table bases
// and partial offsets of slot 0, packed = tokens and items only); the lead warp adds the
// unit's fields and the slot's offsets.
//   packed: bits 0-4 tokens - 1 (all items), bit 5 expand, bits 6-8 projection slot,
//           bits 9-11 hidden block, bits 12-15 rank chunk (shrink units), bits 16-17 items - 1
//   rows:   rank rows: the item's rank (one item; chunks of kRC), or the last item's first
//           row + its rank (a pack: one chunk)
struct alignas(16) Unit {
    uint32_t packed;
    int32_t rows;
    int32_t pad[2];
    PackItem item[kPackItems];
};
static_assert(sizeof(Unit) == 112, "Unit layout");

__host__ __device__ inline uint32_t unit_pack(int nt, int expand, int pj, int b, int c, int ni)
{
    return (uint32_t)(nt - 1) | ((uint32_t)expand << 5) | ((uint32_t)pj << 6) | ((uint32_t)b << 9) |
           ((uint32_t)c << 12) | ((uint32_t)(ni - 1) << 16);
}

// One entry of the work list: the work group and the unit's bits of `packed` (expand,
// projection slot, hidden block, rank chunk).
struct alignas(8) ListUnit {
    int32_t wg;
    uint32_t packed;
};

// The shrink units' partial sums: one 64-bit word per value, the fp32 bits in the low half
// and the launch's tag in the high half, written with one relaxed store, so a reader that
// sees the tag sees the value (no fence, no counter).
struct PlanLayout {
    PlanHeader *hdr;
    int32_t *tok_order;
    Unit *wgs;              // work groups (projection slot 0, no unit fields)
    ListUnit *units;        // the work list
    unsigned long long *upart;
    int64_t cap_wg, cap_units, cap_words;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tokens one plan covers: the whole range up to kMaxPlanTokens when every adapter id fits
// the plan's group tables, otherwise chunks of kMaxPlanGroups tokens.
inline int32_t plan_chunk(int32_t max_adapters)
{
    return max_adapters <= kMaxPlanGroups ? kMaxPlanTokens : kMaxPlanGroups;
}

// Hidden blocks: the K slices of the shrink and the column blocks of the expand.
inline int n_blocks(int hidden) { return ceil_div(hidden, kMaxSlice); }

// Scratch of one plan: header, token order, units, tagged partials.  Items are at most one
// per token, so every count is bounded by the tokens of the plan.
PlanLayout carve(void *base, int32_t cap_tokens, int32_t n_proj, int32_t nblk, int32_t max_rank, size_t *total)
{
    PlanLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return (char *)base + o;
    };
    const int64_t cap = cap_tokens;
    const int64_t nch = ceil_div(max_rank < 1 ? 1 : max_rank, kRC);
    L.cap_wg = cap;
    L.cap_units = cap * n_proj * nblk * (nch + 1);
    L.cap_words = cap * n_proj * nblk * nch * kRC;
    L.hdr = (PlanHeader *)take(sizeof(PlanHeader));
    L.tok_order = (int32_t *)take(cap * 4);
    L.wgs = (Unit *)take(L.cap_wg * sizeof(Unit));
    L.units = (ListUnit *)take(L.cap_units * sizeof(ListUnit));
    L.upart = (unsigned long long *)take(L.cap_words * 8);
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
    int32_t n_proj;     // projections of the call
    int32_t nblk;       // hidden blocks
    int32_t proj[kMaxApplyProj];
    const float *scaling;   // optional override [max_adapters]
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
    a.L.hdr->n_wg = 0;
    a.L.hdr->n_units = 0;
    a.L.hdr->n_shrink = 0;
    a.L.hdr->grab = 0;
    a.L.hdr->exits = 0;
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
    __shared__ int warp_tot8[33][8];
    __shared__ int s_lo, s_hi, s_G;
    __shared__ int s_bucket[kRankBuckets + 1], s_bcur[kRankBuckets + 1];
    __shared__ int s_proj[kMaxApplyProj];   // the call's projection slots (indexed per unit)
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
    if (tid < kMaxApplyProj) s_proj[tid] = a.proj[tid];
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

    // 3. per-group offsets in that order.  A group's items hold kTok tokens each but the
    //    last.  Its last item is packable when it has at most kPackTokens tokens and the
    //    rank is at most 2 kSlot (class 1: rank <= kSlot, class 2: above); every other item
    //    is a work group of its own.  Scanned per group: tokens, own items, their shrink
    //    units, partial words, and per class the packable items and their tokens.
    const int NP = a.n_proj, NB = a.nblk;
    // the hash keys are not read after step 1; HS >= 2 G, so they hold both tables
    int *pus = keys;        // [position] first shrink unit of the group's own items
    int *puw = keys + G;    // [position] first partial word
    int *psolo = pit;       // [position] first own item (its work group)
    auto pk_class = [](int rank, int lnt) {
        return lnt <= kPackTokens && rank <= 2 * kSlot ? (rank <= kSlot ? 1 : 2) : 0;
    };
    const int per_g = ceil_div(G > 0 ? G : 1, NT);
    const int p0 = tid * per_g;
    int mine[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    auto group_counts = [&](int pos, int (&v)[8]) {
        const int g = gperm[pos];
        const int n = hcnt[gslot[g]], r = grank[g], nch = ceil_div(r, kRC);
        const int m = ceil_div(n, kTok), lnt = n - kTok * (m - 1), cl = pk_class(r, lnt);
        const int solo = m - (cl ? 1 : 0);
        v[0] = n;
        v[1] = solo;
        v[2] = NP * NB * nch * solo;
        v[3] = NP * NB * nch * kRC * n;
        v[4] = cl == 1;
        v[5] = cl == 1 ? lnt : 0;
        v[6] = cl == 2;
        v[7] = cl == 2 ? lnt : 0;
        return cl;
    };
    for (int q = 0; q < per_g && p0 + q < G; ++q) {
        int v[8];
        group_counts(p0 + q, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) mine[i] += v[i];
    }
    int off0[8], tot[8];
    block_excl_scan<8>(mine, warp_tot8, off0, tot);
    {
        int off[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) off[i] = off0[i];
        for (int q = 0; q < per_g && p0 + q < G; ++q) {
            const int pos = p0 + q;
            int v[8];
            group_counts(pos, v);
            gtok[gperm[pos]] = off[0];
            psolo[pos] = off[1];
            pus[pos] = off[2];
            puw[pos] = off[3];
#pragma unroll
            for (int i = 0; i < 8; ++i) off[i] += v[i];
        }
    }
    const int n_solo = tot[1], s_solo = tot[2], n_c1 = tot[4], n_c2 = tot[6];
    const int n_p2 = ceil_div(n_c2, 2), n_p1 = ceil_div(n_c1, kPackItems);
    const int n_wg = n_solo + n_p2 + n_p1;
    const int n_shrink = s_solo + (n_p2 + n_p1) * NP * NB;
    const int64_t n_units = (int64_t)n_shrink + (int64_t)n_wg * NP * NB;
    if (n_units > a.L.cap_units || n_wg > a.L.cap_wg || (int64_t)tot[3] > a.L.cap_words) {
        if (tid == 0) plan_refuse(a);
        return;
    }
    __syncthreads();

    // the token order first: the hash-slot table is free afterwards
    for (int i = tid; i < Tc; i += NT) {
        const int h = tslot[i];
        if (h >= 0)
            a.L.tok_order[gtok[hgrp[h]] + tpos[i]] = a.t_begin + i;
    }
    __syncthreads();
    // packable items by class, in group order: their group position and the tokens of the
    // class before them (class 1 at [0, n_c1), class 2 at [n_c1, n_c1 + n_c2))
    int *cpos = hgrp, *ctp = hgrp + G;
    {
        int off[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) off[i] = off0[i];
        for (int q = 0; q < per_g && p0 + q < G; ++q) {
            const int pos = p0 + q;
            int v[8];
            const int cl = group_counts(pos, v);
            if (cl == 1) {
                cpos[off[4]] = pos;
                ctp[off[4]] = off[5];
            } else if (cl == 2) {
                cpos[n_c1 + off[6]] = pos;
                ctp[n_c1 + off[6]] = off[7];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) off[i] += v[i];
        }
    }
    __shared__ unsigned long long s_mag[kMaxRank / kRC + 1];   // ceil(2^32 / (NP NB nch)), per nch
    __shared__ unsigned long long s_mag_e, s_mag_nb;
    auto magic = [](uint32_t d) { return (unsigned long long)(0xffffffffu / d) + 1ull; };
    if (tid <= kMaxRank / kRC) s_mag[tid] = magic((uint32_t)(NP * NB) * (uint32_t)(tid < 1 ? 1 : tid));
    if (tid == 0) {
        s_mag_e = magic((uint32_t)(NP * NB));
        s_mag_nb = magic((uint32_t)NB);
    }
    __syncthreads();

    // 4. the units, one per thread in list order (consecutive threads write consecutive
    //    units): the shrink units of the own items (groups in order, items in order), then
    //    those of the packs (class 2, then class 1), then one expand unit per work group,
    //    projection slot and hidden block in the same work-group order.  An own item finds
    //    its group by binary search over the group offsets; divisions by the per-call
    //    divisors use exact reciprocal multiplies (x d < 2^32 here).
    auto div = [](uint32_t x, unsigned long long m) { return (int)((x * m) >> 32); };
    auto last_le = [&](const int *arr, int key) {
        int lo_p = 0, hi_p = G - 1;
        while (lo_p < hi_p) {
            const int mid = (lo_p + hi_p + 1) >> 1;
            if (arr[mid] <= key) lo_p = mid; else hi_p = mid - 1;
        }
        return lo_p;
    };
    // the work groups, one per thread: an own item (group found by binary search over the
    // own-item offsets) or a pack
    for (int w = tid; w < n_wg; w += NT) {
        Unit u;
        u.pad[0] = u.pad[1] = 0;
        auto fill = [&](PackItem &it, int g, int item_in_group, int row0, int t0, int nt, int p) {
            const int rank = grank[g], nch = ceil_div(rank, kRC);
            it.pt_base = gpt[g];
            it.tok_start = gtok[g] + kTok * item_in_group;
            it.geo = geo_pack(row0, rank, t0, nt);
            it.scaling = a.scaling ? a.scaling[gad[g]] : gscale[g];
            it.uoff = puw[p] + item_in_group * NP * NB * nch * kRC * kTok;
        };
        int ni, nt_all;
        if (w < n_solo) {
            const int pos = last_le(psolo, w), ig = w - psolo[pos];
            const int g = gperm[pos];
            const int nt = min(kTok, hcnt[gslot[g]] - kTok * ig);
            fill(u.item[0], g, ig, 0, 0, nt, pos);
            ni = 1;
            nt_all = nt;
            u.rows = grank[g];
        } else {
            const int pack = w - n_solo;
            const bool c2 = pack < n_p2;
            const int cap = c2 ? 2 : kPackItems, slot = c2 ? 2 * kSlot : kSlot;
            const int cbase = c2 ? n_c1 : 0, cnt = c2 ? n_c2 : n_c1;
            const int ci0 = (c2 ? pack : pack - n_p2) * cap;
            ni = min(cap, cnt - ci0);
            const int tp0 = ctp[cbase + ci0];
            int rows = 0;
            nt_all = 0;
#pragma unroll
            for (int j = 0; j < kPackItems; ++j) {   // unrolled: the items stay in registers
                if (j < ni) {
                    const int p = cpos[cbase + ci0 + j], g = gperm[p];
                    const int n = hcnt[gslot[g]], m = ceil_div(n, kTok), lnt = n - kTok * (m - 1);
                    fill(u.item[j], g, m - 1, slot * j, ctp[cbase + ci0 + j] - tp0, lnt, p);
                    rows = slot * j + grank[g];
                    nt_all = ctp[cbase + ci0 + j] - tp0 + lnt;
                }
            }
            u.rows = rows;
        }
#pragma unroll
        for (int j = 1; j < kPackItems; ++j) {
            if (j >= ni) {
                u.item[j].pt_base = 0;
                u.item[j].tok_start = 0;
                u.item[j].geo = 0;
                u.item[j].scaling = 0.f;
                u.item[j].uoff = 0;
            }
        }
        u.packed = unit_pack(nt_all, 0, 0, 0, 0, ni);
        a.L.wgs[w] = u;
    }
    // the work list, one entry per thread
    for (int k = tid; k < n_units; k += NT) {
        const bool expand = k >= n_shrink;
        int pj, b, c = 0, wg;
        if (!expand && k < s_solo) {
            const int pos = last_le(pus, k);
            const int nch = ceil_div(grank[gperm[pos]], kRC);
            const int r = k - pus[pos];
            const int ig = div((uint32_t)r, s_mag[nch]);
            const int l = r - ig * NP * NB * nch;
            pj = l / (NB * nch);
            const int rem = l - pj * NB * nch;
            b = rem / nch;
            c = rem - b * nch;
            wg = psolo[pos] + ig;
        } else {
            const int e = expand ? k - n_shrink : k - s_solo;
            const int q = div((uint32_t)e, s_mag_e);
            const int l = e - q * NP * NB;
            pj = div((uint32_t)l, s_mag_nb);
            b = l - pj * NB;
            wg = expand ? q : n_solo + q;
        }
        ListUnit lu;
        lu.wg = wg;
        lu.packed = ((uint32_t)(expand ? 1 : 0) << 5) | ((uint32_t)pj << 6) | ((uint32_t)b << 9) | ((uint32_t)c << 12);
        a.L.units[k] = lu;
    }
    if (tid == 0) {
        a.L.hdr->n_groups = G;
        a.L.hdr->n_wg = n_wg;
        a.L.hdr->n_units = (int32_t)n_units;
        a.L.hdr->n_shrink = n_shrink;
        a.L.hdr->seg_lo = lo;
        a.L.hdr->seg_hi = hi;
        a.L.hdr->grab = 0;
        a.L.hdr->exits = 0;
    }
}

// ---------------------------------------------------------------------------------------
// delta kernel

struct DeltaArgs {
    PoolView pv;
    const __half *x[kMaxApplyProj];   // per projection slot of the call
    __half *y[kMaxApplyProj];
    PlanLayout L;
    int32_t pitch;          // bytes per row of a ring stage: 2 * largest block + 16
    int32_t nblk;           // hidden blocks
    uint32_t tag;           // this launch's partial-sum tag (never 0)
    int32_t proj[kMaxApplyProj];   // projection of each slot of the call
    // The plan was complete before this launch began (a stored plan's later applies): the
    // lead warp then publishes the CTA's first unit before the grid-dependency wait, and the
    // copy warps start its page-row stages, so that they overlap the end of the kernel
    // before; the lead waits before it claims any unit, a copy warp before its first token
    // stage (x or y0, which the kernel before may still be writing).
    int32_t plan_ready;
};

// A unit as the lead warp hands it to the other warps: the descriptor, the token ids of
// its rows, each row's item, and the page ids of its first rank chunk (A^T rows of a shrink
// unit's chunk, B rows of an expand unit's chunk 0).
constexpr int32_t kGapRow = -2;   // page id of a row between a pack's items: zeros, not an error
struct alignas(16) Rec {
    Unit u;
    int32_t tok[kTok];      // token ids of the unit's token rows (0 past its tokens)
    int32_t pg[kRC];        // page ids of the first chunk's rows (-1 past the rows, kGapRow in a gap)
    int8_t titem[kTok];     // item of each token row
    int32_t end;            // no more units
    int32_t pad[3];
};

// ---- decode-specific helpers (inline PTX) ---------------------------------------------
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

// d = a * b for one 16x8x16 tile (zero accumulator input).
__device__ __forceinline__ void mma16816_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// A unit as 7 x 16 bytes in registers (every lane of the lead loads all of it).
constexpr int kUnitVecs = (int)(sizeof(Unit) / 16);
struct UnitRegs {
    uint4 w[kUnitVecs];
    // 32-bit word i of the unit (i a compile-time constant once loops are unrolled)
    __device__ __forceinline__ uint32_t word(int i) const
    {
        const uint4 v = w[i >> 2];
        return (i & 3) == 0 ? v.x : (i & 3) == 1 ? v.y : (i & 3) == 2 ? v.z : v.w;
    }
    __device__ __forceinline__ uint32_t packed() const { return word(0); }
    __device__ __forceinline__ int rows() const { return (int)word(1); }
    // item j's fields (PackItem at byte 16 + 24 j)
    __device__ __forceinline__ int64_t pt_base(int j) const
    {
        return (int64_t)(((uint64_t)word(5 + 6 * j) << 32) | word(4 + 6 * j));
    }
    __device__ __forceinline__ int tok_start(int j) const { return (int)word(6 + 6 * j); }
    __device__ __forceinline__ uint32_t geo(int j) const { return word(7 + 6 * j); }
    __device__ __forceinline__ void set_word(int i, uint32_t x)
    {
        uint4 &v = w[i >> 2];
        if ((i & 3) == 0) v.x = x; else if ((i & 3) == 1) v.y = x; else if ((i & 3) == 2) v.z = x; else v.w = x;
    }
};
static_assert(sizeof(Unit) % 16 == 0 && offsetof(Unit, item) == 16, "Unit layout for UnitRegs");
__device__ __forceinline__ void load_unit(const Unit *p, UnitRegs &r)
{
    const uint4 *s = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < kUnitVecs; ++i) r.w[i] = __ldcg(s + i);
}

// Tagged partial words: relaxed 64-bit accesses at GPU scope (single-copy atomic).
__device__ __forceinline__ void st_word(unsigned long long *p, float v, uint32_t tag)
{
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long *p)
{
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

// Position in the ring: the slot of the next stage and the parity of its phase.  Walking the
// ring one stage at a time needs no division.
struct RingPos {
    uint32_t slot, phase;
    __device__ __forceinline__ void next()
    {
        if (++slot == NST) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// A unit's fields, unpacked.
struct UnitShape {
    int nt, expand, pj, b, c;
    int nch;         // rank chunks the unit covers (an expand covers every chunk of the rank)
};
__device__ __forceinline__ UnitShape unit_shape(uint32_t packed, int rows)
{
    UnitShape s;
    s.nt = (int)(packed & 31u) + 1;
    s.expand = (int)((packed >> 5) & 1u);
    s.pj = (int)((packed >> 6) & 7u);
    s.b = (int)((packed >> 9) & 7u);
    s.c = (int)((packed >> 12) & 15u);
    s.nch = s.expand ? ceil_div(rows, kRC) : 1;
    return s;
}
// rows of the i-th chunk the unit covers
__device__ __forceinline__ int chunk_rows(int rows, const UnitShape &s, int i)
{
    const int c = s.expand ? i : s.c;
    return min(kRC, rows - kRC * c);
}

// A unit's ring stages: one stage of its token rows (x of a shrink, y0 of an expand), then its
// rank rows (A^T rows of the shrink's chunk, or B rows of every chunk; 8 per stage).
__global__ void __launch_bounds__(kThreads, 1) delta_kernel(const __grid_constant__ DeltaArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int P = a.pitch;
    const int stageB = 8 * P;                                                    // one 8-row ring stage
    uint8_t *ring = smem;                                                        // [NST][8][P]
    uint8_t *zrow = ring + NST * stageB;                                         // [P] zeros: rows past the rank / tokens
    float *pset = reinterpret_cast<float *>(zrow + P);                           // [8 warps][kRegionFloats] partials / y0
    __half *ubuf = reinterpret_cast<__half *>(pset + kPtmpFloats);               // [QU][8][kUPitch] u (fp16)
    Rec *recs = reinterpret_cast<Rec *>(ubuf + QU * kTok * kUPitch);             // [QD] units in flight
    uint64_t *bars = reinterpret_cast<uint64_t *>(recs + QD);
    uint64_t *full = bars, *empty = bars + NST;              // ring stages
    uint64_t *rfull = bars + 2 * NST, *rempty = rfull + QD;  // unit records
    uint64_t *ufull = rempty + QD, *uempty = ufull + QU;     // u buffers
    uint64_t *psfull = uempty + QU, *psempty = psfull + 1;   // shrink partials (consumers -> reduce warp)
    __shared__ int s_abort;
    __shared__ int s_done;                                   // units the consumers have finished
    __shared__ int s_blk[kMaxBlocks + 1];                    // first element of each hidden block

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.pv.hidden;
    const int NB = a.nblk;
    int32_t *status = a.pv.status;
    volatile int *abort = &s_abort;
    volatile int *done = &s_done;
    const uint32_t ring_s = smem_u32(ring), zrow_s = smem_u32(zrow);
    const uint32_t ubuf_s = smem_u32(ubuf);

    for (int o = tid * 16; o < P; o += kThreads * 16) *reinterpret_cast<uint4 *>(zrow + o) = make_uint4(0, 0, 0, 0);
    if (tid <= kMaxBlocks) {
        // hidden block b: whole 16-element steps [s_blk[b], s_blk[b+1])
        const int nk16 = d / 16;
        s_blk[tid] = tid <= NB ? 16 * ((tid * nk16) / NB) : d;
    }
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int q = 0; q < QD; ++q) {
            mbar_init(&rfull[q], 1);
            mbar_init(&rempty[q], kRecReaders);
        }
        for (int q = 0; q < QU; ++q) {
            mbar_init(&ufull[q], 1);
            mbar_init(&uempty[q], kConsumerWarps);
        }
        mbar_init(psfull, kConsumerWarps);
        mbar_init(psempty, 1);
        s_abort = 0;
        s_done = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the plan of this batch is complete and visible; the lead of a launch over a stored plan
    // waits later (see DeltaArgs::plan_ready)
    const bool lead_early = a.plan_ready != 0 && warp == kWarpLead;
    const bool copy_early = a.plan_ready != 0 && warp >= kWarpCopy0 && warp < kWarpCopy0 + kCopyWarps;
    if (!lead_early && !copy_early) griddep_wait();
    griddep_launch_dependents();
    const int n_units = __ldcg(&a.L.hdr->n_units);

    // read record k's header (every reader walks the records in order); false at the end
    auto take_record = [&](int k, uint32_t &packed, int &rows) -> bool {
        const uint32_t q = k % QD;
        wait_phase<false>(&rfull[q], (k / QD) & 1, abort, status);
        if (*abort) return false;
        const int end = recs[q].end;
        packed = recs[q].u.packed;
        rows = recs[q].u.rows;
        return !end;
    };
    auto release_record = [&](int k) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[k % QD]);
    };

    if (warp == kWarpLead) {
        // ================================== lead (metadata) ==================================
        // Takes units in list order (the first by the CTA's index, then from the plan's
        // counter) and publishes each with its token ids and first chunk's page ids.
        const int G = (int)gridDim.x;
        const int32_t *pt = a.pv.pt_arena;
        // the token id of token row `lane` and the page ids of rows `lane`, `lane` + 32 of the
        // unit's first chunk, with the token's item; every lane holds the whole unit
        auto fetch_rest = [&](const UnitRegs &u, int &tok, int &titem, int32_t &p0, int32_t &p1) {
            const uint32_t packed = u.packed();
            const int rows = u.rows();
            const int nt = (int)(packed & 31u) + 1, ni = (int)((packed >> 16) & 3u) + 1;
            const bool expand = (packed & 32u) != 0;
            const int c = expand ? 0 : (int)((packed >> 12) & 15u);
            int ti = 0, tstart = 0, t0 = 0;
#pragma unroll
            for (int j = 0; j < kPackItems; ++j) {
                const uint32_t g = u.geo(j);
                if (j < ni && lane >= geo_t0(g)) {
                    ti = j;
                    tstart = u.tok_start(j);
                    t0 = geo_t0(g);
                }
            }
            tok = lane < nt ? __ldcg(a.L.tok_order + tstart + lane - t0) : 0;
            titem = ti;
            const int rows_c = min(kRC, rows - kRC * c);
            auto page_of = [&](int r) -> int32_t {
                if (r >= rows_c) return -1;
                int64_t base = 0;
                int row0 = 0, rank = 0;
#pragma unroll
                for (int j = 0; j < kPackItems; ++j) {
                    const uint32_t g = u.geo(j);
                    if (j < ni && r >= geo_row0(g)) {
                        row0 = geo_row0(g);
                        rank = geo_rank(g);
                        base = u.pt_base(j);
                    }
                }
                const int within = r + kRC * c - row0;
                return within < rank ? __ldcg(pt + base + (expand ? rank : 0) + within) : kGapRow;
            };
            p0 = page_of(lane);
            p1 = page_of(lane + 32);
        };
        // unit k from its list entry and its work group: the unit's bits of packed, the
        // projection slot's page-table bases and partial offsets
        auto resolve = [&](const UnitRegs &wg, int2 lu, UnitRegs &u) {
            u = wg;
            const uint32_t lp = (uint32_t)lu.y;
            const int pj = (int)((lp >> 6) & 7u);
            const int proj = a.proj[pj];
            const int ni = (int)((wg.packed() >> 16) & 3u) + 1;
            u.set_word(0, wg.packed() | lp);
#pragma unroll
            for (int j = 0; j < kPackItems; ++j) {
                if (j < ni) {
                    const uint32_t g = wg.geo(j);
                    const int rank = geo_rank(g), nch = ceil_div(rank, kRC);
                    const int64_t ptb = wg.pt_base(j) + (int64_t)proj * 2 * rank;
                    u.set_word(4 + 6 * j, (uint32_t)(uint64_t)ptb);
                    u.set_word(5 + 6 * j, (uint32_t)((uint64_t)ptb >> 32));
                    u.set_word(9 + 6 * j, wg.word(9 + 6 * j) + (uint32_t)(pj * nch * NB * geo_nt(g) * kRC));
                }
            }
        };
        auto load_lu = [&](int idx) { return __ldcg(reinterpret_cast<const int2 *>(a.L.units) + idx); };
        // A four-stage software pipeline; in one pass the record of a unit is published (its
        // token and page ids were loaded in the pass before), the next unit is resolved and
        // its token and page ids loaded, the work group of the one after it loaded, the list
        // entry of a claimed unit loaded, and a new unit claimed from the plan's counter.
        // Claims stay at most kClaimAhead units ahead of the units the consumers have
        // finished: units claimed early are a static schedule, and at the end of the list
        // the CTAs that claimed slower units would finish late.  A pass with nothing to
        // publish leaves a bubble in the pipeline rather than waiting; only an empty pipeline
        // waits (bounded) for the consumers.
        bool vB = false, vC = false, vD = false;   // stage valid: list entry, work group, resolved unit
        bool apend = false, exhausted = false;     // a claim in flight; the list has run out
        int grab = 0;                              // lane 0: the last claim's counter value
        int2 luB = make_int2(0, 0), luC = make_int2(0, 0);
        UnitRegs wC{}, uD{};
        int dtok = 0, dti = 0;
        int32_t dp0 = -1, dp1 = -1;
        int nclaimed = 0, kp = 0;                  // units claimed, records published
        bool waited = !lead_early;                 // past the grid-dependency wait
        {
            // the first unit is list entry blockIdx.x: its entry is loaded before the count of
            // units is known (an index inside the list's allocation; used only if valid)
            const int2 lu0 = a.L.cap_units > 0 ? load_lu((int)min((int64_t)blockIdx.x, a.L.cap_units - 1))
                                               : make_int2(0, 0);
            if ((int)blockIdx.x < n_units) {
                luB = lu0;
                vB = true;
                nclaimed = 1;
                if (kClaimAhead > 1 && waited) {
                    if (lane == 0) grab = atomicAdd(&a.L.hdr->grab, 1);
                    apend = true;
                    ++nclaimed;
                }
            } else {
                exhausted = true;
            }
        }
        uint64_t t_wait = 0;
        for (uint32_t it = 0;; ++it) {
            if (vD) {
                const uint32_t q = kp % QD;
                if (kp >= QD) wait_phase<false>(&rempty[q], ((kp / QD) - 1) & 1, abort, status);
                if (*abort) {
                    vB = vC = vD = apend = false;
                    exhausted = true;
                } else {
                    uint4 v = uD.w[0];
#pragma unroll
                    for (int i = 1; i < kUnitVecs; ++i)
                        if (lane == i) v = uD.w[i];
                    if (lane < kUnitVecs) reinterpret_cast<uint4 *>(&recs[q].u)[lane] = v;
                    if (lane == 0) recs[q].end = 0;
                    if (lane < kTok) {
                        recs[q].tok[lane] = dtok;
                        recs[q].titem[lane] = (int8_t)dti;
                    }
                    recs[q].pg[lane] = dp0;
                    recs[q].pg[lane + 32] = dp1;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&rfull[q]);
                    ++kp;
                }
            }
            vD = vC;
            if (vC) {
                resolve(wC, luC, uD);
                fetch_rest(uD, dtok, dti, dp0, dp1);
            }
            vC = vB;
            if (vB) {
                luC = luB;
                load_unit(a.L.wgs + luB.x, wC);
            }
            vB = false;
            if (apend) {
                const int idx = G + __shfl_sync(0xffffffffu, grab, 0);
                apend = false;
                if (idx < n_units) {
                    luB = load_lu(idx);
                    vB = true;
                } else {
                    exhausted = true;
                }
            }
            if (!waited && kp >= 1) {
                // the first unit is published: from here on the counter is used, which the
                // launch before resets at its end
                griddep_wait();
                waited = true;
            }
            if (waited && !exhausted && nclaimed - __shfl_sync(0xffffffffu, *done, 0) < kClaimAhead) {
                if (lane == 0) grab = atomicAdd(&a.L.hdr->grab, 1);
                apend = true;
                ++nclaimed;
            }
            if (vB || vC || vD || apend) {
                t_wait = 0;
                continue;
            }
            if (exhausted) {
                if (!waited) {
                    griddep_wait();
                    waited = true;
                }
                const uint32_t q = kp % QD;
                if (kp >= QD) wait_phase<false>(&rempty[q], ((kp / QD) - 1) & 1, abort, status);
                if (lane == 0) {
                    recs[q].end = 1;
                    mbar_arrive(&rfull[q]);
                    // the last lead of the launch to be done claiming resets the counter, so
                    // that the plan serves further launches (one per layer of an iteration)
                    if (atomicAdd(&a.L.hdr->exits, 1) == (int)gridDim.x - 1) {
                        atomicExch(&a.L.hdr->grab, 0);
                        atomicExch(&a.L.hdr->exits, 0);
                    }
                }
                break;
            }
            // every claimed unit is published and the consumers are kClaimAhead behind: wait
            // for them to finish one (bounded in time)
            __nanosleep(64);
            if (t_wait == 0) t_wait = global_timer_ns();
            if ((it & 15u) == 0 && global_timer_ns() - t_wait > kWaitLimitNs) {
                set_status(status, SLORA_DEV_TIMEOUT);
                *abort = 1;
            }
            if (*abort) exhausted = true;
        }
        return;
    }

    if (warp >= kWarpCopy0 && warp < kWarpCopy0 + kCopyWarps) {
        // ==================================== copy warps =====================================
        // Every copy warp walks every unit's stages; stage g of the CTA goes to copy warp
        // g % kCopyWarps, which waits for its ring slot, then lanes 0-7 each bulk-copy one
        // row's slice of the unit's hidden block (several warps keep enough copies in flight).
        const int cw = warp - kWarpCopy0;
        const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);
        const int32_t *pt = a.pv.pt_arena;
        RingPos pos{0, 0};
        uint32_t sc = 0;   // stages of the CTA so far
        bool waited = !copy_early;   // past the grid-dependency wait
        for (int k = 0;; ++k) {
            uint32_t packed;
            int rows;
            const bool have = take_record(k, packed, rows);
            const uint32_t q = k % QD;
            if (!have) {
                release_record(k);
                break;
            }
            const UnitShape sh = unit_shape(packed, rows);
            const int64_t ptb0 = recs[q].u.item[0].pt_base;   // later chunks: one item only
            const int kb = s_blk[sh.b];
            const uint32_t sliceB = (uint32_t)(s_blk[sh.b + 1] - kb) * 2;
            const int r8 = lane & 7;
            const int tok = recs[q].tok[r8];
            int32_t pg_first[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) pg_first[j] = recs[q].pg[8 * j + r8];
            release_record(k);
            // lane r < 8 copies row r of a stage from src (when ok), rows left out zero-filled
            // when zero_rest; completion on the slot's full barrier
            auto issue = [&](const __half *src, bool ok, bool zero_rest) {
                if (sc >= NST) wait_phase<false>(&empty[pos.slot], pos.phase ^ 1u, abort, status);
                if (__any_sync(0xffffffffu, *abort != 0)) return;   // after an abort nothing more is issued
                const uint32_t dst = ring_s + pos.slot * stageB;
                const bool mine = ok && lane < 8;
                const uint32_t m = __ballot_sync(0xffffffffu, mine);
                if (mine) bulk_g2s_s(dst + lane * P, src + kb, sliceB, &full[pos.slot]);
                if (zero_rest && (m & 0xffu) != 0xffu) {
                    for (int r = 0; r < 8; ++r) {
                        if ((m >> r) & 1u) continue;
                        for (uint32_t o = lane * 16; o < sliceB; o += 32 * 16)
                            *reinterpret_cast<uint4 *>(ring + pos.slot * stageB + r * P + o) = make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_proxy_async_smem();   // before later bulk copies land in the same rows
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&full[pos.slot], (uint32_t)__popc(m) * sliceB);
            };
            // token stage
            if ((int)(sc % kCopyWarps) == cw) {
                if (!waited) {
                    griddep_wait();
                    waited = true;
                }
                issue((sh.expand ? a.y[sh.pj] : a.x[sh.pj]) + (int64_t)tok * d, r8 < sh.nt, false);
            }
            ++sc;
            pos.next();
            // rank stages
#pragma unroll 1
            for (int i = 0; i < sh.nch; ++i) {
                const int crow = chunk_rows(rows, sh, i);
                const int ns = ceil_div(crow, 8);
                // B rows of chunk i > 0 of an expand (a unit of one item: rows is its rank)
                const int64_t base = ptb0 + rows + (int64_t)kRC * i;
#pragma unroll 1
                for (int s = 0; s < ns; ++s, ++sc, pos.next()) {
                    if ((int)(sc % kCopyWarps) != cw) continue;
                    const int row = 8 * s + r8;
                    int32_t pg = -1;
                    if (row < crow) {
                        if (i == 0) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (j == s) pg = pg_first[j];
                        } else {
                            pg = __ldcg(pt + base + row);
                        }
                    }
                    bool ok = row < crow && pg >= 0;
                    if (ok && pg >= a.pv.num_pages) {
                        set_status(status, SLORA_DEV_BAD_PAGE);
                        ok = false;
                    }
                    // kGapRow: the rows between a pack's items, zeros by design
                    if (lane < 8 && row < crow && pg == -1) set_status(status, SLORA_DEV_BAD_PAGE);
                    issue(pool + (int64_t)(ok ? pg : 0) * d, ok, sh.expand != 0);
                }
            }
        }
        // no bulk copy may land after the CTA exits: wait (bounded) for this warp's last ones
        for (uint32_t i = 0; i < NST && i < sc; ++i) {
            const uint32_t g = sc - 1 - i;
            if ((int)(g % kCopyWarps) == cw) mbar_wait_bounded(&full[g % NST], (g / NST) & 1, status);
        }
        return;
    }

    if (warp == kWarpReduce || warp == kWarpGather) {
        // ============================== reduce and gather warps ============================
        // Reduce warp, shrink units of this CTA: sums the consumer warps' partials in warp
        // order and writes the unit's partial as tagged words.  Gather warp, expand units ahead
        // of the consumers: waits until the partial words of every hidden block carry this
        // launch's tag, sums them in block order and rounds u to fp16 once, into the next u
        // buffer (lane l covers tokens l>>4, +2 per round, columns 4 (l & 15) .. +3).  Two
        // warps, so that the gather can start on the first expand units while the last shrink
        // units of the CTA still run.
        const bool reducer = warp == kWarpReduce;
        const uint32_t tag = a.tag;
        uint32_t uj = 0;   // u buffers filled
        uint32_t sr = 0;   // shrink partials summed
        for (int k = 0;; ++k) {
            uint32_t packed;
            int rows;
            const bool have = take_record(k, packed, rows);
            const uint32_t q = k % QD;
            // the items' shapes and partial offsets, and each token row's item
            uint32_t ig[kPackItems];
            int iu[kPackItems];
#pragma unroll
            for (int j = 0; j < kPackItems; ++j) {
                ig[j] = recs[q].u.item[j].geo;
                iu[j] = recs[q].u.item[j].uoff;
            }
            const unsigned long long titems = *reinterpret_cast<const unsigned long long *>(recs[q].titem);
            release_record(k);
            if (!have) break;
            const int nt = (int)(packed & 31u) + 1;
            // token row t's item: first row, rank, first token, tokens, partial offset
            auto item_of = [&](int t, int &row0, int &rank, int &t0, int &nti, int &uoff) {
                const int j = (int)((titems >> (8 * t)) & 0xffu);
                uint32_t g = ig[0];
                uoff = iu[0];
#pragma unroll
                for (int jj = 1; jj < kPackItems; ++jj)
                    if (jj == j) {
                        g = ig[jj];
                        uoff = iu[jj];
                    }
                row0 = geo_row0(g);
                rank = geo_rank(g);
                t0 = geo_t0(g);
                nti = geo_nt(g);
            };
            if (!(packed & 32u)) {
                if (!reducer) continue;
                const int c = (int)((packed >> 12) & 15u), b = (int)((packed >> 9) & 7u);
                const int rows_c = min(kRC, rows - kRC * c), ld = 16 * ceil_div(rows_c, 16);
                wait_phase<false>(psfull, sr & 1, abort, status);
#pragma unroll 1
                for (int e = 4 * lane; e < nt * ld; e += 128) {
                    const int t = e / ld, j = e - t * ld;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int g = 0; g < kConsumerWarps; ++g) {
                        const float4 pv = *reinterpret_cast<const float4 *>(pset + g * kRegionFloats + t * kRC + j);
                        v.x += pv.x;
                        v.y += pv.y;
                        v.z += pv.z;
                        v.w += pv.w;
                    }
                    int row0, rank, t0, nti, uoff;
                    item_of(t, row0, rank, t0, nti, uoff);
                    const int rank_c = min(kRC, rank - kRC * c);
                    unsigned long long *o =
                        a.L.upart + uoff + ((int64_t)(c * NB + b) * nti + (t - t0)) * kRC + (j - row0);
                    const int w0 = j - row0;
                    if (w0 >= 0 && w0 < rank_c) st_word(o, v.x, tag);
                    if (w0 + 1 >= 0 && w0 + 1 < rank_c) st_word(o + 1, v.y, tag);
                    if (w0 + 2 >= 0 && w0 + 2 < rank_c) st_word(o + 2, v.z, tag);
                    if (w0 + 3 >= 0 && w0 + 3 < rank_c) st_word(o + 3, v.w, tag);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(psempty);
                ++sr;
                continue;
            }
            if (reducer) continue;
            const int nch = ceil_div(rows, kRC);
            const int j4 = 4 * (lane & 15);
#pragma unroll 1
            for (int c = 0; c < nch; ++c) {
                const uint32_t qu = uj % QU;
                if (uj >= QU) wait_phase<false>(&uempty[qu], ((uj / QU) - 1) & 1, abort, status);
                __half *ub = ubuf + qu * kTok * kUPitch;
#pragma unroll 1
                for (int tr = 0; tr < nt; tr += 2) {
                    const int t = tr + (lane >> 4);
                    // this lane's values: columns j4 .. j4+3 of token row t lie in its item's rows
                    // of the chunk (zeros elsewhere)
                    int nv = 0, bstride = 0;
                    const unsigned long long *sp = a.L.upart;
                    if (t < nt) {
                        int row0, rank, t0, nti, uoff;
                        item_of(t, row0, rank, t0, nti, uoff);
                        const int rank_c = min(kRC, rank - kRC * c), w0 = j4 - row0;
                        if (w0 >= 0 && w0 < rank_c) {
                            nv = min(4, rank_c - w0);
                            sp = a.L.upart + uoff + ((int64_t)c * NB * nti + (t - t0)) * kRC + w0;   // block 0
                            bstride = nti * kRC;                                                // blocks apart
                        }
                    }
                    float wv[kMaxBlocks][4];
                    // poll until every word carries the tag (each was written once, by its
                    // shrink unit, earlier in the list); bounded in time
                    uint64_t t_start = 0;
                    for (uint32_t it = 0;; ++it) {
                        bool ready = true;
#pragma unroll
                        for (int bb = 0; bb < kMaxBlocks; ++bb)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const unsigned long long w = (bb < NB && e < nv) ? ld_word(sp + bb * bstride + e)
                                                                                 : ((unsigned long long)tag << 32);
                                ready &= (uint32_t)(w >> 32) == tag;
                                wv[bb][e] = __uint_as_float((uint32_t)w);
                            }
                        if (__all_sync(0xffffffffu, ready)) break;
                        if (*abort) break;
                        __nanosleep(128);
                        if (it == kPollsBeforeTimer) t_start = global_timer_ns();
                        if (it > kPollsBeforeTimer && (it & 15u) == 0 && global_timer_ns() - t_start > kWaitLimitNs) {
                            set_status(status, SLORA_DEV_TIMEOUT);
                            *abort = 1;
                            break;
                        }
                    }
                    if (t < nt) {
                        float sm[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = 0.f;
#pragma unroll
                            for (int bb = 0; bb < kMaxBlocks; ++bb)
                                if (bb < NB) v += wv[bb][e];
                            sm[e] = e < nv ? v : 0.f;
                        }
                        __half2 h[2];
                        h[0] = __floats2half2_rn(sm[0], sm[1]);
                        h[1] = __floats2half2_rn(sm[2], sm[3]);
                        *reinterpret_cast<uint2 *>(ub + t * kUPitch + j4) = *reinterpret_cast<const uint2 *>(h);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ufull[qu]);
                ++uj;
            }
        }
        return;
    }

    // ===================================== consumers =====================================
    const int w = warp;
    const int q4 = lane >> 3, rr = lane & 7, gid = lane >> 2, tig = lane & 3;
    RingPos cur{0, 0};   // the next stage to consume
    uint32_t uj = 0;     // u buffers consumed
    auto wait_at = [&](const RingPos &p) { wait_phase<false>(&full[p.slot], p.phase, abort, status); };
    uint32_t sj = 0;     // shrink units done (uses of the partial set)
    float *region = pset + w * kRegionFloats;   // this warp's shrink partials
    // The record of the next unit is read while the current one runs: its header, the
    // token id of this lane's row gid and the scaling of that token's item.
    auto item_scaling = [&](uint32_t q) { return recs[q].u.item[recs[q].titem[gid] & (kPackItems - 1)].scaling; };
    uint32_t upk;
    int urows;
    bool have = take_record(0, upk, urows);
    int tk = recs[0].tok[gid];
    float scl = item_scaling(0);
    release_record(0);
    for (int k = 0; have; ++k) {
        const UnitShape sh_ = unit_shape(upk, urows);
        const int nt = sh_.nt;
        const int kb = s_blk[sh_.b], KS = s_blk[sh_.b + 1] - kb;
        const RingPos tpos = cur;   // the token stage
        cur.next();
        wait_at(tpos);
        uint32_t npk;
        int nrows;
        const bool nhave = take_record(k + 1, npk, nrows);
        const int ntk = recs[(k + 1) % QD].tok[gid];
        const float nscl = item_scaling((k + 1) % QD);
        release_record(k + 1);
        const uint32_t tstage = ring_s + tpos.slot * stageB;

        if (!sh_.expand) {
            // ---- shrink: u^T = A^T x^T, rank rows on the MMA's M and tokens on its N.  Warp w
            //      contracts K steps [w n/8, (w+1) n/8) of the block for every 16-row block of
            //      the chunk; the 8 warp partials are summed in warp order ----
            const int rows = chunk_rows(urows, sh_, 0), nb = ceil_div(rows, 16), ns = ceil_div(rows, 8);
            const int nsteps = KS / 16;
            const int ks0 = (w * nsteps) / kConsumerWarps, nks = ((w + 1) * nsteps) / kConsumerWarps - ks0;
            uint32_t xf[kXs / 2][4];   // this warp's x fragments (the MMA's B operand), two K steps each
            {
                const uint32_t trow = tstage + rr * P;
#pragma unroll
                for (int i = 0; i < kXs / 2; ++i)
                    if (2 * i < nks) ldsm_x4(trow + (16 * (ks0 + 2 * i) + 8 * q4) * 2, xf[i]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[tpos.slot]);
#pragma unroll 1
            for (int blk = 0; blk < nb; ++blk) {
                const RingPos lo = cur;
                cur.next();
                const bool has_hi = 2 * blk + 1 < ns;
                const RingPos hi = cur;
                if (has_hi) cur.next();
                wait_at(lo);
                if (has_hi) wait_at(hi);
                // A operand rows: 0-7 from stage lo, 8-15 from stage hi (or zeros)
                const uint32_t arow = (q4 & 1) ? (has_hi ? ring_s + hi.slot * stageB + rr * P : zrow_s)
                                               : ring_s + lo.slot * stageB + rr * P;
                float pacc[2][4] = {};   // even / odd K steps: two independent MMA chains
                if (nks == kXs) {
                    // the usual case: every A^T fragment is loaded before the first MMA, so the
                    // loads' latency is paid once per block rather than once per K step
                    uint32_t af[kXs][4];
#pragma unroll
                    for (int i = 0; i < kXs; ++i)
                        ldsm_x4(arow + (16 * (ks0 + i) + 8 * (q4 >> 1)) * 2, af[i]);   // A^T rows
#pragma unroll
                    for (int i = 0; i < kXs; ++i)
                        mma16816(pacc[i & 1], af[i], xf[i >> 1][2 * (i & 1)], xf[i >> 1][2 * (i & 1) + 1]);
                } else {
#pragma unroll
                    for (int i = 0; i < kXs; ++i) {
                        if (i < nks) {
                            uint32_t af[4];
                            ldsm_x4(arow + (16 * (ks0 + i) + 8 * (q4 >> 1)) * 2, af);   // A^T rows
                            mma16816(pacc[i & 1], af, xf[i >> 1][2 * (i & 1)], xf[i >> 1][2 * (i & 1) + 1]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[lo.slot]);
                    if (has_hi) mbar_arrive(&empty[hi.slot]);
                }
                // the partial set is free once the reduce warp has summed the previous shrink
                // unit (waited for only now, so that the first block's loads and MMAs overlap it)
                if (blk == 0 && sj > 0) wait_phase<false>(psempty, (sj - 1) & 1, abort, status);
                // rows gid, gid + 8 of the block; tokens 2 tig, 2 tig + 1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    region[(2 * tig) * kRC + 16 * blk + gid + 8 * h] = pacc[0][2 * h] + pacc[1][2 * h];
                    region[(2 * tig + 1) * kRC + 16 * blk + gid + 8 * h] = pacc[0][2 * h + 1] + pacc[1][2 * h + 1];
                }
            }
            // hand the partial to the reduce warp, which sums the 8 warps' partials in order
            __syncwarp();
            if (lane == 0) mbar_arrive(psfull);
            ++sj;
        } else {
            // ---- expand: y = u B over the block's columns, the item's tokens on the MMA's M
            //      (rows 0-7; rows 8-15 zero) and the columns on its N; warp w takes the column
            //      pairs [pp0, pp1) (16 columns each), over the rank chunks ----
            const int npair = KS / 16;
            const int pp0 = (w * npair) / kConsumerWarps, pp1 = ((w + 1) * npair) / kConsumerWarps;
            // A unit of at most 64 rank rows (9 stages) keeps its token stage (y0) until the
            // epilogue; a longer one would hold the ring, so it first copies this lane's y0
            // values (token gid, columns 16 (pp0+p) + 8 n2 + 2 tig, +1) to the warp's region,
            // once the reduce warp has summed the partials the region held.
            const bool hold = urows <= kRC;
            uint32_t *yv = reinterpret_cast<uint32_t *>(region);
            if (!hold) {
                if (sj > 0) wait_phase<false>(psempty, (sj - 1) & 1, abort, status);
                const uint8_t *trow = ring + tpos.slot * stageB + gid * P;
#pragma unroll
                for (int p = 0; p < kPairs; ++p)
#pragma unroll
                    for (int n2 = 0; n2 < 2; ++n2)
                        if (pp0 + p < pp1)
                            yv[(2 * p + n2) * 32 + lane] =
                                *reinterpret_cast<const uint32_t *>(trow + (16 * (pp0 + p) + 8 * n2 + 2 * tig) * 2);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[tpos.slot]);
            }
            float acc[2 * kPairs][4];
#pragma unroll 1
            for (int c = 0; c < sh_.nch; ++c) {
                const uint32_t qu = uj % QU;
                wait_phase<false>(&ufull[qu], (uj / QU) & 1, abort, status);
                const int rows = chunk_rows(urows, sh_, c), nb = ceil_div(rows, 16), ns = ceil_div(rows, 8);
                const uint32_t ub = ubuf_s + qu * (kTok * kUPitch * 2);
#pragma unroll 1
                for (int blk = 0; blk < nb; ++blk) {
                    const RingPos lo = cur;
                    cur.next();
                    const bool has_hi = 2 * blk + 1 < ns;
                    const RingPos hi = cur;
                    if (has_hi) cur.next();
                    wait_at(lo);
                    if (has_hi) wait_at(hi);
                    // u rows (the MMA's A operand): the item's tokens in rows 0-7, zeros in rows 8-15
                    uint32_t af[4];
                    ldsm_x4((q4 & 1) ? zrow_s + (16 * blk + 8 * (q4 >> 1)) * 2
                                     : ub + (rr * kUPitch + 16 * blk + 8 * (q4 >> 1)) * 2, af);
                    // B rows (the MMA's B operand, transposed on load): 0-7 from stage lo, 8-15 from hi
                    const uint32_t brow = (q4 & 1) ? (has_hi ? ring_s + hi.slot * stageB + rr * P : zrow_s)
                                                   : ring_s + lo.slot * stageB + rr * P;
                    if (pp1 - pp0 == kPairs) {
                        // the usual case: the B fragments are loaded kAhead column pairs ahead of
                        // their MMAs, so the loads' latency is paid once per block, not per pair
                        constexpr int kAhead = 3;   // (more would spill registers)
                        uint32_t bf[kAhead][4];
#pragma unroll
                        for (int p = 0; p < kAhead; ++p)
                            ldsm_x4_t(brow + (16 * (pp0 + p) + 8 * (q4 >> 1)) * 2, bf[p]);
                        const bool zc = c == 0 && blk == 0;
#pragma unroll
                        for (int p = 0; p < kPairs; ++p) {
                            if (zc) {
                                mma16816_zc(acc[2 * p], af, bf[p % kAhead][0], bf[p % kAhead][1]);
                                mma16816_zc(acc[2 * p + 1], af, bf[p % kAhead][2], bf[p % kAhead][3]);
                            } else {
                                mma16816(acc[2 * p], af, bf[p % kAhead][0], bf[p % kAhead][1]);
                                mma16816(acc[2 * p + 1], af, bf[p % kAhead][2], bf[p % kAhead][3]);
                            }
                            if (p + kAhead < kPairs)
                                ldsm_x4_t(brow + (16 * (pp0 + p + kAhead) + 8 * (q4 >> 1)) * 2, bf[p % kAhead]);
                        }
                    } else if (c == 0 && blk == 0) {
                        // the first block starts the accumulators (zero C operand)
#pragma unroll
                        for (int p = 0; p < kPairs; ++p) {
                            if (pp0 + p < pp1) {
                                uint32_t bf[4];
                                ldsm_x4_t(brow + (16 * (pp0 + p) + 8 * (q4 >> 1)) * 2, bf);
                                mma16816_zc(acc[2 * p], af, bf[0], bf[1]);
                                mma16816_zc(acc[2 * p + 1], af, bf[2], bf[3]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int p = 0; p < kPairs; ++p) {
                            if (pp0 + p < pp1) {
                                uint32_t bf[4];
                                ldsm_x4_t(brow + (16 * (pp0 + p) + 8 * (q4 >> 1)) * 2, bf);
                                mma16816(acc[2 * p], af, bf[0], bf[1]);
                                mma16816(acc[2 * p + 1], af, bf[2], bf[3]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[lo.slot]);
                        if (has_hi) mbar_arrive(&empty[hi.slot]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&uempty[qu]);
                ++uj;
            }
            // ---- epilogue: y = y0 + s * acc for token gid: columns 2 tig, 2 tig + 1 of each n-tile ----
            __half *yrow = a.y[sh_.pj] + (int64_t)tk * d + kb;
            const bool store = !*abort && gid < nt;
            if (hold) {
                // y0 of four n-tiles (rows 0-7 of the token stage) per fragment load
                const uint32_t yaddr = tstage + rr * P + (16 * pp0 + 8 * q4) * 2;
#pragma unroll
                for (int p2 = 0; p2 < kPairs / 2; ++p2) {
                    if (pp0 + 2 * p2 < pp1) {
                        uint32_t yf[4];
                        ldsm_x4(yaddr + p2 * 64, yf);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int p = 2 * p2 + (i >> 1), n2 = i & 1;
                            if (store && pp0 + p < pp1) {
                                const int col = 16 * (pp0 + p) + 8 * n2 + 2 * tig;
                                const float2 y0 = __half22float2(*reinterpret_cast<const __half2 *>(&yf[i]));
                                const float *ac = acc[2 * p + n2];
                                *reinterpret_cast<__half2 *>(yrow + col) =
                                    __floats2half2_rn(fmaf(scl, ac[0], y0.x), fmaf(scl, ac[1], y0.y));
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[tpos.slot]);
            } else if (store) {
#pragma unroll
                for (int p = 0; p < kPairs; ++p) {
                    if (pp0 + p < pp1) {
#pragma unroll
                        for (int n2 = 0; n2 < 2; ++n2) {
                            const int col = 16 * (pp0 + p) + 8 * n2 + 2 * tig;
                            const float2 y0 =
                                __half22float2(*reinterpret_cast<const __half2 *>(&yv[(2 * p + n2) * 32 + lane]));
                            const float *ac = acc[2 * p + n2];
                            *reinterpret_cast<__half2 *>(yrow + col) =
                                __floats2half2_rn(fmaf(scl, ac[0], y0.x), fmaf(scl, ac[1], y0.y));
                        }
                    }
                }
            }
        }
        if (w == 0 && lane == 0) *done = k + 1;
        upk = npk;
        urows = nrows;
        tk = ntk;
        scl = nscl;
        have = nhave;
    }
}

}  // namespace

size_t plan_scratch_bytes(int32_t T, int32_t max_rank, int32_t hidden, int32_t max_adapters, int32_t n_proj)
{
    size_t total = 0;
    const int32_t chunk = plan_chunk(max_adapters);
    const int32_t cap = T < chunk ? T : chunk;
    carve(nullptr, cap, n_proj < 1 ? 1 : n_proj, n_blocks(hidden), max_rank, &total);
    return total;
}

// Bytes per row of a stage or token buffer for a hidden size: the widest block + 16 (the
// padding keeps the rows' fragment loads free of bank conflicts).
inline int delta_pitch(int hidden)
{
    const int NB = n_blocks(hidden);
    return 2 * 16 * ceil_div(hidden / 16, NB) + 16;
}
inline size_t delta_smem_bytes(int hidden)
{
    const size_t P = (size_t)delta_pitch(hidden);
    return NST * 8 * P + P + (size_t)kPtmpFloats * 4 + (size_t)QU * kTok * kUPitch * 2 + QD * sizeof(Rec) +
           (2 * NST + 2 * QD + 2 * QU + 2) * 8;
}

// Kernel attributes and the delta grid's resident CTAs, per device (the attributes are
// per-device state; calls may come from several threads).
struct DeltaLaunchState {
    bool attrs = false;
    int occ_hidden = -1;
    int occ_blocks = 1;
};
constexpr int kMaxLaunchDevices = 64;
std::mutex g_delta_mu;
DeltaLaunchState g_delta_state[kMaxLaunchDevices];

// The launches of a batch.  For every chunk of at most `chunk` tokens: the plan into the
// chunk's scratch (make_plans) and the decode kernel over it (pl non-null); then the segment
// kernel (pl non-null and n_seg > 0).  `scratch` holds one PlanScratch per chunk, or a single
// one that every chunk reuses in turn (n_scratch == 1).
static cudaError_t launch_batch(const PoolView &pv, const ProjList *pl, int32_t n_slots, int32_t T,
                                const int32_t *idx, const int32_t *seg_indptr, int32_t n_seg,
                                const float *scaling, PlanScratch *scratch, int n_scratch, bool make_plans,
                                bool plan_ready, int num_sms, cudaStream_t stream, int *launches,
                                cudaEvent_t after_plan)
{
    if (pv.hidden > kMaxBlocks * kMaxSlice || n_slots < 1 || n_slots > kMaxApplyProj || n_scratch < 1)
        return cudaErrorInvalidValue;
    if (pl && pl->n != n_slots) return cudaErrorInvalidValue;
    for (int i = 0; i < n_scratch; ++i)
        if (n_slots > scratch[i].cap_proj) return cudaErrorInvalidValue;
    int device = 0;
    cudaError_t de = cudaGetDevice(&device);
    if (de != cudaSuccess) return de;
    if (device < 0 || device >= kMaxLaunchDevices) return cudaErrorInvalidDevice;
    const size_t dsmem = delta_smem_bytes(pv.hidden);
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
    if (pv.hidden != ls.occ_hidden) {
        int nb = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, delta_kernel, kThreads, dsmem);
        if (e != cudaSuccess) return e;
        ls.occ_blocks = nb > 0 ? nb : 1;
        ls.occ_hidden = pv.hidden;
    }
    const int occ_blocks = ls.occ_blocks;
    lk.unlock();

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(num_sms * occ_blocks);
    cfg2.blockDim = dim3(kThreads);
    cfg2.dynamicSmemBytes = dsmem;
    cfg2.stream = stream;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;

    int32_t chunk = plan_chunk(pv.max_adapters);
    if (scratch[0].max_chunk > 0 && scratch[0].max_chunk < chunk) chunk = scratch[0].max_chunk;
    const int NB = n_blocks(pv.hidden);
    if (n_scratch > 1 && (int64_t)n_scratch * chunk < T) return cudaErrorInvalidValue;

    for (int32_t tb = 0, c = 0; tb < T; tb += chunk, ++c) {
        const int32_t te = tb + chunk < T ? tb + chunk : T;
        PlanScratch &sc = scratch[n_scratch > 1 ? c : 0];
        const int32_t cap = sc.cap_tokens < chunk ? sc.cap_tokens : chunk;
        if (te - tb > cap) return cudaErrorInvalidValue;
        const PlanLayout L = carve(sc.base, cap, sc.cap_proj, NB, sc.max_rank, nullptr);
        cudaError_t e = cudaSuccess;
        uint32_t tag = 0;
        if (pl) {
            if (sc.tag == 0) {
                // fresh scratch or a wrapped tag sequence: no partial word may carry a tag in use
                e = cudaMemsetAsync(L.upart, 0, (size_t)L.cap_words * 8, stream);
                if (e != cudaSuccess) return e;
            }
            tag = ++sc.tag;
            if (sc.tag == 0xffffffffu) sc.tag = 0;
        }
        if (make_plans) {
            const int32_t groups = (te - tb) < pv.max_adapters ? (te - tb) : pv.max_adapters;
            int hs = 1024;
            while (hs < 2 * groups && hs < kMaxHash) hs <<= 1;
            const int dcache = pv.max_adapters <= kPlanDirCache ? 1 : 0;
            PlanArgs pa{};
            pa.pv = pv;
            pa.idx = idx;
            pa.T = T;
            pa.seg_indptr = seg_indptr;
            pa.n_seg = n_seg;
            pa.t_begin = tb;
            pa.t_end = te;
            pa.hash_size = hs;
            pa.dir_cache = dcache;
            pa.n_proj = n_slots;
            pa.nblk = NB;
            if (pl)
                for (int j = 0; j < pl->n; ++j) pa.proj[j] = pl->proj[j];
            pa.scaling = scaling;
            pa.L = L;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1);
            const bool small = te - tb <= kPlanThreadsSmall;
            cfg.blockDim = dim3(small ? kPlanThreadsSmall : kPlanThreads);
            cfg.dynamicSmemBytes = plan_smem_bytes(hs) + (dcache ? (size_t)pv.max_adapters * sizeof(DirEntry) : 0);
            cfg.stream = stream;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = small ? cudaLaunchKernelEx(&cfg, plan_kernel<kPlanThreadsSmall>, pa)
                      : cudaLaunchKernelEx(&cfg, plan_kernel<kPlanThreads>, pa);
            if (e != cudaSuccess) return e;
            *launches += 1;
            if (after_plan && tb == 0) {
                e = cudaEventRecord(after_plan, stream);
                if (e != cudaSuccess) return e;
            }
        }
        if (!pl) continue;
        DeltaArgs da{};
        da.pv = pv;
        for (int j = 0; j < pl->n; ++j) {
            da.x[j] = reinterpret_cast<const __half *>(pl->x[j]);
            da.y[j] = reinterpret_cast<__half *>(pl->y[j]);
        }
        da.L = L;
        da.pitch = delta_pitch(pv.hidden);
        da.nblk = NB;
        da.tag = tag;
        for (int j = 0; j < pl->n; ++j) da.proj[j] = pl->proj[j];
        da.plan_ready = plan_ready && !make_plans ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg2, delta_kernel, da);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (pl && n_seg > 0) {
        cudaError_t e = launch_prefill(pv, *pl, T, idx, seg_indptr, n_seg, scaling, num_sms, stream);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaSuccess;
}

cudaError_t launch_lora_apply(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                              const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                              PlanScratch &scratch, int num_sms, cudaStream_t stream, int *launches,
                              cudaEvent_t after_plan)
{
    return launch_batch(pv, &pl, pl.n, T, idx, seg_indptr, n_seg, scaling, &scratch, 1, true, false, num_sms,
                        stream, launches, after_plan);
}

cudaError_t launch_plans(const PoolView &pv, int32_t n_slots, int32_t T, const int32_t *idx,
                         const int32_t *seg_indptr, int32_t n_seg, const float *scaling, PlanScratch *chunks,
                         int n_chunks, int num_sms, cudaStream_t stream, int *launches)
{
    return launch_batch(pv, nullptr, n_slots, T, idx, seg_indptr, n_seg, scaling, chunks, n_chunks, true, false,
                        num_sms, stream, launches, nullptr);
}

cudaError_t launch_planned(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                           const int32_t *seg_indptr, int32_t n_seg, const float *scaling, PlanScratch *chunks,
                           int n_chunks, bool plan_ready, int num_sms, cudaStream_t stream, int *launches)
{
    return launch_batch(pv, &pl, pl.n, T, idx, seg_indptr, n_seg, scaling, chunks, n_chunks, false, plan_ready,
                        num_sms, stream, launches, nullptr);
}

int32_t plan_chunk_tokens(int32_t max_adapters) { return plan_chunk(max_adapters); }

}  // namespace slora
