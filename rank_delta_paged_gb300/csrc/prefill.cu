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
// Work unit: one 128-token tile of one segment for one projection of the call (a call may
// cover several projections of a layer; unit u is tile u / n_proj of projection slot
// u % n_proj).  Persistent clusters of C CTAs (C = 1, 2, 4 or 8, chosen on the host from
// the number of units: rounds of units over the resident clusters against bytes per CTA)
// take units in turn (batches of at most 32 segments deal them costliest first: segments
// by their adapter's rank, descending, in rounds of alternating direction); CTA c of a
// cluster owns hidden slice c: the K range of its part
// of the shrink and the N range of its part of the expand, so every byte of x, y0, y and
// of the adapter's pages is moved by exactly one CTA.  In such a batch the units of the
// last, partial round (all of them when there is one round) are split by expand columns
// into 2 or 4 parts, the most the clusters that round would leave idle can take: each part
// runs on its own cluster, repeats the whole shrink (so x and the A^T rows move again) and
// forms its share of every CTA's columns of y.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 3      scheduler and token loader: maps the cluster's next unit to (segment,
//               tile), checks the tile's tokens agree on the adapter, reads the directory
//               and the page table (invalid pages read as zeros) and publishes a unit
//               descriptor with the unit's page ids through a two-slot ring; then one lane
//               streams the unit's token tiles (128 x 64 of x for the shrink, then of y0
//               for the expand) by TMA tensor-tile loads with the 128-byte swizzle into a
//               ring of 16 KiB slots, as many as shared memory holds (5 to 8), as fast as
//               slots free up.
//   warps 0-1, 8-11  page-row gather: the adapter's page rows for each stage (64-element
//               pieces of the A^T rows, or of the B rows) go through the page table into a
//               48 KiB ring in the same swizzled layout, 16 bytes per cp.async, spread over
//               192 threads (a gather runs at about 10 GB/s per issuing warp).  Its slots
//               hold r_pad rows of 128 bytes, so a small rank keeps more stages in flight
//               (16 slots at rank 8 or 16, 3 at rank 128).  The
//               copies signal the slot's mbarrier as they land
//               (cp.async.mbarrier.arrive.noinc), so no thread waits for data.  The token
//               stream runs up to a whole ring ahead; the page rows, mostly L2 hits, follow
//               just in time, so a slot of either ring is held only as long as it must be.
//   warp 2      one thread issues tcgen05.mma: the shrink M=128, N=r (padded to a
//               multiple of 16 with zero rows), K=16 per instruction into TMEM columns
//               0..127; the expand M=128, N=64, K=r into four 64-column TMEM buffers.
//   warps 4-7   exchange and epilogue (warp 4 + q reads TMEM lanes 32q..32q+31).  After
//               the shrink, the partial U of each CTA is reduced over the cluster: rows
//               are owned round the cluster, partial rows go to their owner's shared memory
//               (st.shared::cluster), the owner sums the C partials in CTA order, rounds
//               to fp16 once (the only extra rounding) and writes the row into every CTA's
//               U operand.  Then, tile by tile, each warp forms y = y0 + s * acc for its 32
//               rows in place in the y0 slot and writes them back with its own TMA
//               tensor-tile store (a ragged last tile of a segment is stored row by row, so
//               no token of another segment is touched); the last warp done with a slot
//               returns it to the ring, so the four warps never wait for one another there.
// Every wait is bounded; a unit whose tokens disagree on their adapter, or whose adapter
// is not resident, is skipped with a device status code.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"
#include "tcgen05.h"

namespace slora {
namespace {

constexpr int kWarps = 12;
constexpr int kThreads = 32 * kWarps;
constexpr int kMmaWarp = 2;
constexpr int kSchedWarp = 3;
constexpr int kEpiWarp0 = 4;                  // warps 4-7: one per TMEM lane quarter
constexpr int kEpiWarps = 4;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kProdWarps = 6;                 // warps 0-1 and 8-11 gather page rows
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int MT = 128;                       // tokens per unit
constexpr int KBLK = 64;                      // K elements (shrink) or columns (expand) per stage
constexpr int kTileBytes = MT * 128;          // 128 rows x 64 fp16, 128-byte rows
constexpr int kUBytes = 2 * kTileBytes;       // U operand: 128 x 128 fp16, two 64-column atoms
constexpr int NB = 4;                         // expand accumulator buffers in TMEM
constexpr uint32_t kTmemCols = 512;           // U at 0..127, expand buffer b at 128 + 64 b
static_assert(128 + NB * 64 + 16 <= (int)kTmemCols, "tensor-memory columns the warm-up load reads");
constexpr int kXPitchMax = kMaxPrefillRank * 4 + 16;
constexpr int kMaxClusterP = 8;
constexpr int kPRingBytes = 3 * kTileBytes;   // page-row ring: slots of r_pad * 128 bytes
constexpr int kMaxPSlots = 16;
constexpr int kMaxTSlots = 8;                 // token-tile ring (as many as shared memory holds)
constexpr size_t kSmemLimit = 227 * 1024;     // dynamic + static shared memory of one CTA
constexpr size_t kStaticReserve = 1024;       // the kernel's static shared memory, rounded up

constexpr int kCompute = 0, kSkip = 1, kEnd = 2;
constexpr int kPgPerLane = 2 * kMaxPrefillRank / 32;   // page ids per scheduler lane
struct alignas(64) UnitDesc {
    int32_t m0, mlen, rank, r_pad;
    float sc;
    int32_t flag;
    int32_t pj;        // projection slot of the call
    int32_t part;      // expand columns: 0 all of the CTA's tiles, else part j of P: 8 P + j
    int32_t pg[2 * kMaxPrefillRank];   // pool pages of the A^T rows, then of the B rows; -1 reads zeros
};

struct PrefillArgs {
    // per projection slot of the call:
    CUtensorMap tmap_x[kMaxApplyProj];   // x [T][hidden], box 64 x 128, 128-byte swizzle
    CUtensorMap tmap_y[kMaxApplyProj];   // y likewise (y0 loads)
    CUtensorMap tmap_ys[kMaxApplyProj];  // y with 64 x 32 boxes: each epilogue warp stores its own 32 rows
    __half *y[kMaxApplyProj];
    int32_t proj[kMaxApplyProj];
    int32_t n_proj;
    PoolView pv;
    const int32_t *idx;
    const int32_t *seg_indptr;
    const float *scaling;
    int32_t T;
    int32_t n_seg;
    int32_t C;       // CTAs per cluster
    int32_t slice;   // hidden elements per CTA, a multiple of 64
    int32_t nt;      // token-tile slots
    int32_t split;   // most parts a unit may be split into by expand columns (1, 2 or 4)
};
static_assert(sizeof(PrefillArgs) <= 4096, "kernel parameters");

// Shared memory: token-tile ring, page-row ring, the U operand, two unit descriptors,
// and the buffer that receives other CTAs' partial rows.
constexpr size_t xbuf_bytes(int C) { return (size_t)(C - 1) * (MT / C) * kXPitchMax; }
constexpr size_t fixed_bytes(int C)
{
    return 1024 + (size_t)kPRingBytes + kUBytes + 2 * sizeof(UnitDesc) + xbuf_bytes(C);
}
constexpr int tslots_for(int C)
{
    const size_t n = (kSmemLimit - kStaticReserve - fixed_bytes(C)) / kTileBytes;
    return n > (size_t)kMaxTSlots ? kMaxTSlots : (int)n;
}
constexpr size_t smem_bytes_for(int C) { return fixed_bytes(C) + (size_t)tslots_for(C) * kTileBytes; }
static_assert(tslots_for(8) >= 5 && tslots_for(2) >= 6, "token ring depth");

// When every cp.async this thread issued so far has landed, arrive on the mbarrier (the
// arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Barrier of the epilogue warps that also ORs a flag over them.
__device__ __forceinline__ bool epi_sync_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(kEpiThreads)
                 : "memory");
    return r != 0;
}

// Page-row slots for a unit of padded rank r_pad: each holds r_pad rows of 128 bytes, so a
// small rank keeps many stages in flight (16 at rank 8 or 16, 3 at rank 128).
__device__ __forceinline__ int pslots_for(int r_pad)
{
    const int n = kPRingBytes / (r_pad * 128);
    return n > kMaxPSlots ? kMaxPSlots : n;
}

__device__ __forceinline__ uint4 pack_h8(const float *f)
{
    uint4 r;
    __half2 *h = reinterpret_cast<__half2 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nts = a.nt;
    uint8_t *tring = smem;                                  // nts x 16 KiB: x or y0 tiles
    uint8_t *pring = tring + nts * kTileBytes;              // page rows
    uint8_t *Us = pring + kPRingBytes;
    UnitDesc *desc = reinterpret_cast<UnitDesc *>(Us + kUBytes);
    uint8_t *xbuf = reinterpret_cast<uint8_t *>(desc + 2);

    __shared__ __align__(8) uint64_t fullT[kMaxTSlots], emptyT[kMaxTSlots], fullP[kMaxPSlots], emptyP[kMaxPSlots];
    __shared__ __align__(8) uint64_t dfull[2], dempty[2], accfull[NB], accempty[NB];
    __shared__ __align__(8) uint64_t ubar, ufull, ufree, xfull, fin;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_stored[kMaxTSlots];   // epilogue warps done with an expand slot
    __shared__ __align__(16) uint4 s_warm[kMaxClusterP];   // slot q: written by CTA q, never read

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = a.C;
    const uint32_t crank = cluster_ctarank();
    volatile int *abort = &s_abort;
    int32_t *status = a.pv.status;

    // The kernel is launched only right after a decode kernel of the same call, which
    // starts it (programmatic dependent launch) only once everything enqueued before the
    // call has completed; it reads nothing the decode kernel writes (segment and decode
    // tokens are disjoint rows), so it waits for that kernel only at its end: its work
    // overlaps the decode kernel's tail, and its completion still implies the decode
    // kernel's, for whatever the stream runs next.
    griddep_launch_dependents();

    if (warp == kMmaWarp) {
        tc::tmem_alloc(&s_tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < nts; ++i) {
            mbar_init(&fullT[i], 1);
            mbar_init(&emptyT[i], 1);
        }
        for (int i = 0; i < kMaxPSlots; ++i) {
            mbar_init(&fullP[i], kProdThreads);
            mbar_init(&emptyP[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], kProdWarps + 1 + kEpiWarps);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&accfull[i], 1);
            mbar_init(&accempty[i], kEpiWarps);
        }
        mbar_init(&ubar, 1);
        mbar_init(&ufull, C);
        mbar_init(&ufree, C);
        mbar_init(&xfull, C > 1 ? C - 1 : 1);
        mbar_init(&fin, 1);
        s_abort = 0;
        for (int i = 0; i < kMaxTSlots; ++i) s_stored[i] = 0;
        fence_mbar_init();
    }
    // every segment well formed?
    int bad = 0;
    for (int i = tid; i < a.n_seg; i += kThreads) {
        const int lo = a.seg_indptr[i], hi = a.seg_indptr[i + 1];
        if (lo < 0 || hi < lo || hi > a.T) bad = 1;
    }
    tc::fence_before_sync();
    bad = __syncthreads_or(bad);
    tc::fence_after_sync();
    if (C > 1) cluster_sync_all();   // every CTA's barriers exist before any remote access
    const uint32_t tmem = s_tmem;
    if (bad && tid == 0) set_status(status, SLORA_DEV_BAD_SEGMENT);

    const int d = a.pv.hidden;
    const int k_lo = (int)crank * a.slice;
    const int k_hi = min(d, k_lo + a.slice);
    const int nkb = (k_hi - k_lo) / KBLK;   // shrink K blocks = expand column tiles
    // A unit split in P parts runs on P clusters: each does the whole shrink (same
    // arithmetic, so the same U) and expands part j of every CTA's column tiles, tiles
    // [nkb j / P, nkb (j + 1) / P), so y is bit for bit the same.
    auto e_first = [nkb](int part) { return part == 0 ? 0 : nkb * (part & 7) / (part >> 3); };
    auto e_count = [nkb](int part) {
        return part == 0 ? nkb : nkb * ((part & 7) + 1) / (part >> 3) - nkb * (part & 7) / (part >> 3);
    };

    if (bad) {
        // nothing to do
    } else if (warp == kSchedWarp) {
        // ---------------------------------------------------------------- scheduler
        const uint32_t cl = cluster_id_x(), ncl = ncluster_x();
        int s0 = 0, base = 0;   // window of 32 segments and the tiles before it
        uint32_t gT = 0;        // token tiles issued
        // Batches of at most 32 segments deal their units costliest first: lane s holds
        // segment s; the segments are sorted by their adapter's rank, descending (ties:
        // lower index first), and the units (tile, projection slot) of the sorted segments
        // go to the clusters in rounds of one unit per cluster, walked in alternating
        // direction.  The units of the last round, which would leave clusters idle (r units
        // after `full` full rounds), are split by expand columns into the most parts P (2 or
        // 4) with P r at most the clusters: places full ncl + P k + j of the deal are the
        // parts of unit full ncl + k.  Every cluster then holds `full` units and at most one
        // part; with a single round (full = 0) every unit is split.
        // Larger batches take the units in order, cluster c every ncl-th.
        const bool lpt = a.n_seg <= 32;
        int s_lo = 0, s_hi = 0, ord = 0, upref = 0, n_units = 0;
        int n_whole = 0, n_parts = 1, n_virt = 0;   // units dealt whole; parts of the rest; places
        int l_ad = -1;                     // lane s: segment s's adapter (its first token's)
        DirEntry l_e{0, 0.f, -1};          // and that adapter's directory entry
        if (lpt) {
            int key = 0x7fffffff;
            if (lane < a.n_seg) {
                s_lo = a.seg_indptr[lane];
                s_hi = a.seg_indptr[lane + 1];
                int rank = 0;
                if (s_hi > s_lo && s_lo >= 0 && s_lo < a.T) {
                    const int ad = a.idx[s_lo];
                    l_ad = ad;
                    if (ad >= 0 && ad < a.pv.max_adapters) {
                        const DirEntry e = a.pv.dir[ad];
                        l_e = e;
                        if (e.pt_off >= 0 && e.rank > 0) rank = min(e.rank, 255);
                    }
                }
                key = ((255 - rank) << 8) | lane;
            }
#pragma unroll
            for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
                for (int j = k >> 1; j > 0; j >>= 1) {
                    const int o = __shfl_xor_sync(0xffffffffu, key, j);
                    const bool up = (lane & k) == 0, low = (lane & j) == 0;
                    key = (low == up) ? min(key, o) : max(key, o);
                }
            }
            const bool valid = key != 0x7fffffff;
            ord = valid ? (key & 0xff) : 0;   // the segment at sorted place `lane`
            const int sl = __shfl_sync(0xffffffffu, s_lo, ord), sh = __shfl_sync(0xffffffffu, s_hi, ord);
            int incl = valid ? (sh - sl + MT - 1) / MT * a.n_proj : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            upref = incl;   // units of sorted places 0 .. lane
            n_units = __shfl_sync(0xffffffffu, incl, 31);
            const int full = n_units / (int)ncl, r = n_units - full * (int)ncl;
            n_whole = n_units;
            if (r > 0)
                for (int P = a.split; P > 1; P >>= 1)
                    if (P * r <= (int)ncl) {
                        n_whole = full * (int)ncl;
                        n_parts = P;
                        break;
                    }
            n_virt = n_whole + n_parts * (n_units - n_whole);
        }
        for (uint32_t i = 0;; ++i) {
            int tile = -1, lo = 0, hi = 0, pj = 0, part = 0, seg_l = 0;
            if (lpt) {
                int p = (int)(i * ncl + ((i & 1) ? (ncl - 1 - cl) : cl));
                if (p < n_virt) {
                    if (p >= n_whole) {
                        const int k = p - n_whole;
                        part = 8 * n_parts + k % n_parts;
                        p = n_whole + k / n_parts;
                    }
                    const int q = __ffs(__ballot_sync(0xffffffffu, upref > p)) - 1;
                    const int prev = __shfl_sync(0xffffffffu, upref, q > 0 ? q - 1 : 0);
                    const int o = p - (q > 0 ? prev : 0);
                    tile = o / a.n_proj;
                    pj = o - tile * a.n_proj;
                    const int seg = __shfl_sync(0xffffffffu, ord, q);
                    lo = __shfl_sync(0xffffffffu, s_lo, seg);
                    hi = __shfl_sync(0xffffffffu, s_hi, seg);
                    seg_l = seg;
                }
            }
            const int vu = (int)(cl + i * ncl);            // unit: (tile mt, projection slot pj)
            const int mt = vu / a.n_proj;
            if (!lpt) pj = vu - mt * a.n_proj;
            while (!lpt && s0 < a.n_seg) {
                const int j = s0 + lane;
                int l = 0, h = 0;
                if (j < a.n_seg) {
                    l = a.seg_indptr[j];
                    h = a.seg_indptr[j + 1];
                }
                const int t = (h - l + MT - 1) / MT;
                int incl = t;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                const int tot = __shfl_sync(0xffffffffu, incl, 31);
                if (base + tot <= mt) {
                    base += tot;
                    s0 += 32;
                    continue;
                }
                const int f = __ffs(__ballot_sync(0xffffffffu, base + incl > mt)) - 1;
                tile = mt - (base + __shfl_sync(0xffffffffu, incl - t, f));
                lo = __shfl_sync(0xffffffffu, l, f);
                hi = __shfl_sync(0xffffffffu, h, f);
                break;
            }
            int flag = kEnd, m0 = 0, mlen = 0, rank = 0;
            float sc = 0.f;
            int32_t pgv[kPgPerLane];   // this lane's page ids of the unit (j = lane + 32 k)
            if (tile >= 0) {
                flag = kSkip;
                m0 = lo + tile * MT;
                mlen = min(MT, hi - m0);
                // The segment's adapter and directory entry come from the lanes of the sort
                // (batches of at most 32 segments) or are loaded here; the page ids are loaded
                // beside the check of the segment's tokens and used only if it passes, so the
                // descriptor waits for one round of loads after the adapter is known.
                int ad;
                DirEntry e{0, 0.f, -1};
                if (lpt) {
                    ad = __shfl_sync(0xffffffffu, l_ad, seg_l);
                    e.rank = __shfl_sync(0xffffffffu, l_e.rank, seg_l);
                    e.scaling = __shfl_sync(0xffffffffu, l_e.scaling, seg_l);
                    e.pt_off = __shfl_sync(0xffffffffu, l_e.pt_off, seg_l);
                } else {
                    ad = a.idx[lo];
                    if (ad >= 0 && ad < a.pv.max_adapters) e = a.pv.dir[ad];
                }
                const bool usable = ad >= 0 && ad < a.pv.max_adapters && e.pt_off >= 0 && e.rank > 0 &&
                                    e.rank <= kMaxPrefillRank;
                const int64_t pt_u = usable ? e.pt_off + (int64_t)a.proj[pj] * 2 * e.rank : 0;
#pragma unroll
                for (int k = 0; k < kPgPerLane; ++k) {
                    const int j = lane + 32 * k;
                    pgv[k] = usable && j < 2 * e.rank ? a.pv.pt_arena[pt_u + j] : -1;
                }
                // a segment whose tokens disagree on the adapter is skipped as a whole: every
                // unit checks its whole segment
                bool mixed = false;
                for (int q = lo + lane; q < hi; q += 32) mixed |= a.idx[q] != ad;
                if (__any_sync(0xffffffffu, mixed)) {
                    if (lane == 0) set_status(status, SLORA_DEV_BAD_SEGMENT);
                } else if (ad == -1) {
                    // base model only
                } else if (ad < -1 || ad >= a.pv.max_adapters) {
                    if (lane == 0) set_status(status, SLORA_DEV_BAD_ADAPTER);
                } else if (e.pt_off < 0 || e.rank <= 0) {
                    if (lane == 0) set_status(status, SLORA_DEV_NOT_RESIDENT);
                } else if (e.rank <= kMaxPrefillRank) {   // larger ranks take the decode path
                    flag = kCompute;
                    rank = e.rank;
                    sc = a.scaling ? a.scaling[ad] : e.scaling;
                }
            }
            wait_phase<false>(&dempty[i & 1], ((i >> 1) & 1) ^ 1, abort, status);
            if (__any_sync(0xffffffffu, *abort)) break;
            UnitDesc *u = &desc[i & 1];
            if (flag == kCompute) {
                bool badp = false;
#pragma unroll
                for (int k = 0; k < kPgPerLane; ++k) {
                    const int j = lane + 32 * k;
                    if (j < 2 * rank) {
                        int32_t p = pgv[k];
                        if (p < 0 || p >= a.pv.num_pages) {
                            badp = true;   // the row reads as zeros
                            p = -1;
                        }
                        u->pg[j < rank ? j : kMaxPrefillRank + j - rank] = p;
                    }
                }
                if (__any_sync(0xffffffffu, badp) && lane == 0) set_status(status, SLORA_DEV_BAD_PAGE);
            }
            if (lane == 0) {
                u->m0 = m0;
                u->mlen = mlen;
                u->rank = rank;
                u->r_pad = (rank + 15) / 16 * 16;
                u->sc = sc;
                u->flag = flag;
                u->pj = pj;
                u->part = part;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&dfull[i & 1]);
            if (flag == kEnd) break;
            // the unit's token tiles: x for the shrink, then y0 for the expand, as slots free up
            if (flag == kCompute && lane == 0) {
                const int e0 = e_first(part), ne = e_count(part);
                for (int st = 0; st < nkb + ne; ++st) {
                    const bool shrink = st < nkb;
                    const int col = k_lo + (shrink ? st : e0 + st - nkb) * KBLK;
                    const uint32_t sT = gT % nts;
                    wait_phase<false>(&emptyT[sT], ((gT / nts) & 1) ^ 1, abort, status);
                    if (*abort) break;
                    mbar_arrive_expect_tx(&fullT[sT], kTileBytes);
                    tma_load_2d(smem_u32(tring + sT * kTileBytes),
                                shrink ? (const void *)&a.tmap_x[pj] : (const void *)&a.tmap_y[pj], col, m0,
                                &fullT[sT]);
                    ++gT;
                }
            }
            __syncwarp();
        }
        // the CTA stays until its last tensor-tile loads have landed
        if (lane == 0)
            for (uint32_t q = gT > (uint32_t)nts ? gT - nts : 0; q < gT; ++q)
                mbar_wait_bounded(&fullT[q % nts], (q / nts) & 1, status);
    } else if (warp < kMmaWarp || warp >= kEpiWarp0 + kEpiWarps) {
        // ---------------------------------------------------------------- producer
        // 192 threads; thread pt copies 16-byte chunks pt, pt + 192, ... of the stage's page
        // rows (chunk q: row q / 8, column chunk q % 8)
        const int pt = warp < kMmaWarp ? tid : tid - 32 * (kEpiWarp0 + kEpiWarps) + 32 * kMmaWarp;
        const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);
        uint32_t pfill = 0;         // bit s: parity of the number of fills of page slot s
        int cur_np = 0, cur_sz = 0;  // the page ring's current slot count and size
        for (uint32_t i = 0;; ++i) {
            wait_phase<false>(&dfull[i & 1], (i >> 1) & 1, abort, status);
            if (__any_sync(0xffffffffu, *abort)) break;
            const UnitDesc *u = &desc[i & 1];
            const int flag = u->flag, r_pad = u->r_pad, e0 = e_first(u->part), ne = e_count(u->part);
            if (flag == kEnd) break;
            bool ab = false;
            if (flag == kCompute) {
                const int np = pslots_for(r_pad), psz = r_pad * 128;
                if (psz != cur_sz) {   // new slot size: every slot of the old layout must be free
                    for (int q = 0; q < cur_np; ++q)
                        wait_phase<false>(&emptyP[q], ((pfill >> q) & 1) ^ 1, abort, status);
                    cur_np = np;
                    cur_sz = psz;
                }
                int sP = 0;
                for (int st = 0; st < nkb + ne; ++st) {
                    const bool shrink = st < nkb;
                    const int col = k_lo + (shrink ? st : e0 + st - nkb) * KBLK;
                    wait_phase<false>(&emptyP[sP], ((pfill >> sP) & 1) ^ 1, abort, status);
                    if (__any_sync(0xffffffffu, *abort)) {
                        ab = true;
                        break;
                    }
                    uint8_t *rows = pring + sP * psz;
                    const int32_t *pg = u->pg + (shrink ? 0 : kMaxPrefillRank);
                    const int rank = u->rank;
#pragma unroll
                    for (int k = 0; k < (kMaxPrefillRank * 8 + kProdThreads - 1) / kProdThreads; ++k) {
                        const int q = pt + kProdThreads * k;
                        const int j = q >> 3, ch = q & 7;
                        if (j < r_pad) {
                            const int32_t p = pg[j];   // rows r..r_pad-1 were never written: masked below
                            const bool v = j < rank && p >= 0;
                            const __half *src = v ? pool + (int64_t)p * d + col + ch * 8 : pool;
                            cp_async16(rows + j * 128 + ((ch ^ (j & 7)) << 4), src, v ? 16u : 0u);
                        }
                    }
                    cp_async_arrive_noinc(&fullP[sP]);   // the stage's consumer fences the proxies
                    pfill ^= 1u << sP;
                    sP = sP + 1 == np ? 0 : sP + 1;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[i & 1]);   // done with the descriptor
            if (ab) break;
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            uint32_t g = 0, e = 0, ui = 0;
            uint32_t pcons = 0;   // bit s: parity of the number of times page slot s was consumed
            const uint32_t ua = smem_u32(Us);
            for (uint32_t i = 0;; ++i) {
                wait_phase<false>(&dfull[i & 1], (i >> 1) & 1, abort, status);
                if (*abort) break;
                const int flag = desc[i & 1].flag, r_pad = desc[i & 1].r_pad, ne = e_count(desc[i & 1].part);
                mbar_arrive(&dempty[i & 1]);
                if (flag == kEnd) break;
                if (flag != kCompute) continue;
                const uint32_t idesc_s = tc::idesc_f16_f32(MT, r_pad, 0, 0);
                const int np = pslots_for(r_pad), psz = r_pad * 128;
                int sP = 0;
                for (int kb = 0; kb < nkb && !*abort; ++kb) {
                    const uint32_t sT = g % nts;
                    wait_phase<false>(&fullT[sT], (g / nts) & 1, abort, status);
                    wait_phase<false>(&fullP[sP], (pcons >> sP) & 1, abort, status);
                    if (*abort) break;
                    tc::fence_proxy_async_smem();   // the cp.async page rows, for the tensor core
                    tc::fence_after_sync();
                    const uint32_t xa = smem_u32(tring + sT * kTileBytes), aa = smem_u32(pring + sP * psz);
#pragma unroll
                    for (int kk = 0; kk < KBLK / 16; ++kk)
                        tc::mma_f16(tmem, tc::smem_desc_sw128(xa + kk * 32, 16, 1024),
                                    tc::smem_desc_sw128(aa + kk * 32, 16, 1024), idesc_s, (kb | kk) != 0);
                    tc::commit(&emptyT[sT]);
                    tc::commit(&emptyP[sP]);
                    pcons ^= 1u << sP;
                    sP = sP + 1 == np ? 0 : sP + 1;
                    ++g;
                }
                if (*abort) break;
                tc::commit(&ubar);
                wait_phase<true>(&ufull, ui & 1, abort, status);
                if (*abort) break;
                tc::fence_after_sync();
                fence_proxy_async_all();
                const uint32_t idesc_e = tc::idesc_f16_f32(MT, KBLK, 0, 1);
                for (int nt = 0; nt < ne; ++nt) {
                    const uint32_t b = e % NB;
                    wait_phase<false>(&fullP[sP], (pcons >> sP) & 1, abort, status);
                    if (e >= (uint32_t)NB) wait_phase<false>(&accempty[b], ((e / NB) - 1) & 1, abort, status);
                    if (*abort) break;
                    tc::fence_proxy_async_smem();
                    tc::fence_after_sync();
                    const uint32_t ba = smem_u32(pring + sP * psz);
                    for (int ks = 0; ks < r_pad / 16; ++ks) {
                        const uint32_t a_addr = ua + (ks >> 2) * kTileBytes + (ks & 3) * 32;
                        tc::mma_f16(tmem + 128 + b * 64, tc::smem_desc_sw128(a_addr, 16, 1024),
                                    tc::smem_desc_sw128(ba + ks * 2048, 8192, 1024), idesc_e, ks != 0);
                    }
                    tc::commit(&emptyP[sP]);
                    tc::commit(&accfull[b]);
                    pcons ^= 1u << sP;
                    sP = sP + 1 == np ? 0 : sP + 1;
                    ++g;
                    ++e;
                }
                if (*abort) break;
                ++ui;
            }
            // every MMA issued has completed before tensor memory is released
            tc::commit(&fin);
            mbar_wait_bounded(&fin, 0, status);
        }
    } else {
        // ---------------------------------------------------------------- exchange + epilogue
        const int qd = warp & 3;           // TMEM lane quarter this warp may access
        const int m = 32 * qd + lane;      // the tile row (token) of this thread
        const int et = tid - 32 * kEpiWarp0;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const uint32_t ua = smem_u32(Us);
        uint32_t g = 0, e = 0, ui = 0;
        int pend = -1;   // (lane 0) token slot this warp's last tensor-tile store may still be reading
        if (C > 1) {
            // A launch's first tensor-memory load and first stores into another CTA's shared
            // memory take one to two microseconds each; made here, while the first unit's
            // shrink runs, they are not paid inside its exchange.  Columns from 384 on are
            // never written (U 0..127, the expand buffers 128..383), and each CTA stores
            // only into its own slot of the peers' s_warm.
            uint32_t wv[16];
            tc::ld_32x32b_x16(tmem + lane_base + 128 + NB * 64, wv);
            tc::ld_wait();
            for (int q = 0; q < C; ++q)
                if (q != (int)crank) st_cluster_v4(mapa(smem_u32(&s_warm[crank]), (uint32_t)q), make_uint4(wv[0], 0u, 0u, 0u));
        }
        for (uint32_t i = 0;; ++i) {
            wait_phase<false>(&dfull[i & 1], (i >> 1) & 1, abort, status);
            if (epi_sync_or(*abort)) break;
            const UnitDesc *ud = &desc[i & 1];
            const int flag = ud->flag, m0 = ud->m0, mlen = ud->mlen, r_pad = ud->r_pad, pj = ud->pj;
            const int e0 = e_first(ud->part), ne = e_count(ud->part);
            const float sc = ud->sc;
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[i & 1]);
            if (flag == kEnd) break;
            if (flag != kCompute) continue;
            const int nkc = r_pad / 16;

            // ---- U = the cluster's partial products summed, rounded to fp16 ----
            wait_phase<false>(&ubar, ui & 1, abort, status);
            tc::fence_after_sync();
            auto u_off = [&](int kc, int half) -> uint32_t {
                return (uint32_t)((kc >> 2) * kTileBytes + m * 128 + (((2 * (kc & 3) + half) ^ (m & 7)) << 4));
            };
            if (C == 1) {
                for (int kc = 0; kc < nkc; ++kc) {
                    uint32_t v[16];
                    tc::ld_32x32b_x16(tmem + lane_base + kc * 16, v);
                    tc::ld_wait();
                    float f[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) f[t] = __uint_as_float(v[t]);
                    *reinterpret_cast<uint4 *>(Us + u_off(kc, 0)) = pack_h8(f);
                    *reinterpret_cast<uint4 *>(Us + u_off(kc, 1)) = pack_h8(f + 8);
                }
                tc::fence_proxy_async_smem();
            } else {
                // rows are owned in blocks of R; with R = 16 the two halves of a warp have
                // different owners, so the (warp-wide) TMEM loads run in every lane
                const int R = MT / C, owner = m / R, rl = m - owner * R;
                const bool mine = owner == (int)crank;
                const int xpitch = r_pad * 4 + 16;
                if (__any_sync(0xffffffffu, !mine)) {
                    // the owner has read its buffer for the previous unit (it signalled ufull)
                    if (ui >= 1) wait_phase<true>(&ufull, (ui - 1) & 1, abort, status);
                    const int slot = (int)crank < owner ? (int)crank : (int)crank - 1;
                    const uint32_t dst = mapa(smem_u32(xbuf + (slot * R + rl) * xpitch), (uint32_t)owner);
                    for (int kc = 0; kc < nkc; ++kc) {
                        uint32_t v[16];
                        __syncwarp();
                        tc::ld_32x32b_x16(tmem + lane_base + kc * 16, v);
                        tc::ld_wait();
                        if (!mine) {
#pragma unroll
                            for (int w4 = 0; w4 < 4; ++w4)
                                st_cluster_v4(dst + kc * 64 + w4 * 16,
                                              make_uint4(v[4 * w4], v[4 * w4 + 1], v[4 * w4 + 2], v[4 * w4 + 3]));
                        }
                    }
                }
                tc::fence_before_sync();
                if (epi_sync_or(*abort)) break;
                if (et == 0)
                    for (int q = 0; q < C; ++q)
                        if (q != (int)crank) mbar_arrive_remote(mapa(smem_u32(&xfull), (uint32_t)q));
                if (__any_sync(0xffffffffu, mine)) {
                    wait_phase<true>(&xfull, ui & 1, abort, status);
                    // every CTA's expand of the previous unit is done with its U operand
                    if (ui >= 1) wait_phase<true>(&ufree, (ui - 1) & 1, abort, status);
                    tc::fence_after_sync();
                    for (int kc = 0; kc < nkc; ++kc) {
                        uint32_t v[16];
                        __syncwarp();
                        tc::ld_32x32b_x16(tmem + lane_base + kc * 16, v);
                        tc::ld_wait();
                        if (!mine) continue;
                        float f[16];
                        for (int src = 0; src < C; ++src) {
                            float p[16];
                            if (src == (int)crank) {
#pragma unroll
                                for (int t = 0; t < 16; ++t) p[t] = __uint_as_float(v[t]);
                            } else {
                                const int slot = src < (int)crank ? src : src - 1;
                                const float4 *xp =
                                    reinterpret_cast<const float4 *>(xbuf + (slot * R + rl) * xpitch + kc * 64);
#pragma unroll
                                for (int w4 = 0; w4 < 4; ++w4) {
                                    const float4 x4 = xp[w4];
                                    p[4 * w4] = x4.x;
                                    p[4 * w4 + 1] = x4.y;
                                    p[4 * w4 + 2] = x4.z;
                                    p[4 * w4 + 3] = x4.w;
                                }
                            }
#pragma unroll
                            for (int t = 0; t < 16; ++t) f[t] = src == 0 ? p[t] : f[t] + p[t];
                        }
                        const uint4 lo4 = pack_h8(f), hi4 = pack_h8(f + 8);
                        const uint32_t o0 = ua + u_off(kc, 0), o1 = ua + u_off(kc, 1);
                        for (int q = 0; q < C; ++q) {
                            st_cluster_v4(mapa(o0, (uint32_t)q), lo4);
                            st_cluster_v4(mapa(o1, (uint32_t)q), hi4);
                        }
                    }
                    fence_proxy_async_all();
                }
            }
            tc::fence_before_sync();
            if (epi_sync_or(*abort)) break;
            if (et == 0)
                for (int q = 0; q < C; ++q) mbar_arrive_remote(mapa(smem_u32(&ufull), (uint32_t)q));
            g += nkb;

            // ---- y = y0 + s * (U B), one 64-column tile at a time, in place in the y0 slot ----
            // Each warp forms and stores its own 32 rows; the last warp done with a slot
            // returns it to the ring, so the warps never wait for one another here.
            const bool full_tile = mlen == MT;
            bool ab = false;
            auto release = [&](int slot) {
                if (atomicAdd(&s_stored[slot], 1) == kEpiWarps - 1) {
                    atomicExch(&s_stored[slot], 0);
                    mbar_arrive(&emptyT[slot]);
                }
            };
            for (int nt = 0; nt < ne; ++nt) {
                const uint32_t sT = g % nts, b = e % NB;
                wait_phase<false>(&accfull[b], (e / NB) & 1, abort, status);
                tc::fence_after_sync();
                uint32_t v[64];
                tc::ld_32x32b_x32(tmem + lane_base + 128 + b * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
                tc::ld_32x32b_x32(tmem + lane_base + 128 + b * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                tc::ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[b]);
                wait_phase<false>(&fullT[sT], (g / nts) & 1, abort, status);   // the y0 tile has landed
                if (__any_sync(0xffffffffu, *abort)) {
                    ab = true;
                    break;
                }
                uint8_t *yt = tring + sT * kTileBytes;
                // the row's eight 16-byte chunks: all loads first, then the arithmetic, then
                // all stores, so the shared-memory latencies overlap
                uint4 yrow[8];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    yrow[cc] = *reinterpret_cast<const uint4 *>(yt + m * 128 + ((cc ^ (m & 7)) << 4));
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&yrow[cc]);
                    float o[8];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 f2 = __half22float2(h2[t]);
                        o[2 * t] = fmaf(sc, __uint_as_float(v[8 * cc + 2 * t]), f2.x);
                        o[2 * t + 1] = fmaf(sc, __uint_as_float(v[8 * cc + 2 * t + 1]), f2.y);
                    }
                    yrow[cc] = pack_h8(o);
                }
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4 *>(yt + m * 128 + ((cc ^ (m & 7)) << 4)) = yrow[cc];
                const int n0 = k_lo + (e0 + nt) * KBLK;
                if (full_tile) {
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&a.tmap_ys[pj], n0, m0 + 32 * qd, smem_u32(yt + 32 * qd * 128));
                        bulk_commit();
                        if (pend >= 0) {   // this warp's store of the previous tile has read its slot
                            bulk_wait_read<1>();
                            release(pend);
                        }
                        pend = (int)sT;
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int qq = lane + 32 * k;
                        const int row = 32 * qd + (qq >> 3), c8 = qq & 7;
                        if (row < mlen) {
                            const uint4 val = *reinterpret_cast<const uint4 *>(yt + row * 128 + ((c8 ^ (row & 7)) << 4));
                            *reinterpret_cast<uint4 *>(a.y[pj] + (int64_t)(m0 + row) * d + n0 + c8 * 8) = val;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) release((int)sT);
                }
                ++g;
                ++e;
            }
            // the unit's last slot is released before the next unit's shrink needs the ring
            if (lane == 0 && pend >= 0) {
                bulk_wait_read<0>();
                release(pend);
                pend = -1;
            }
            if (epi_sync_or(ab || *abort)) break;
            if (C > 1 && et == 0)
                for (int q = 0; q < C; ++q) mbar_arrive_remote(mapa(smem_u32(&ufree), (uint32_t)q));
            ++ui;
        }
        if (lane == 0) bulk_wait<0>();
    }

    griddep_wait();   // the decode kernel of the call has completed (see the top)
    tc::fence_before_sync();
    __syncthreads();
    if (C > 1) cluster_sync_all();   // no CTA of the cluster still touches this one's shared memory
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side ------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [T][hidden] fp16, 64 x box_rows boxes with the 128-byte swizzle; rows past T read as
// zeros and are not written.
cudaError_t token_map(CUtensorMap *m, const void *base, int hidden, int T, int box_rows = MT)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)hidden * 2};
    const cuuint32_t box[2] = {KBLK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_forced_cluster = 0;
int g_prefill_split = 1;

inline int slice_for(int hidden, int C) { return (hidden / 64 + C - 1) / C * 64; }

}  // namespace

// The kernel attribute and the resident clusters for C = 1, 2, 4, 8, per device (the
// attribute is per-device state; calls may come from several threads).
struct PrefillLaunchState {
    bool attr = false;
    int ncl[4] = {0, 0, 0, 0};
};
constexpr int kMaxLaunchDevices = 64;
std::mutex g_prefill_mu;
PrefillLaunchState g_prefill_state[kMaxLaunchDevices];

cudaError_t launch_prefill(const PoolView &pv, const ProjList &pl, int32_t T, const int32_t *idx,
                           const int32_t *seg_indptr, int32_t n_seg, const float *scaling, int num_sms,
                           cudaStream_t stream)
{
    int device = 0;
    cudaError_t de = cudaGetDevice(&device);
    if (de != cudaSuccess) return de;
    if (device < 0 || device >= kMaxLaunchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_prefill_mu);
    PrefillLaunchState &ls = g_prefill_state[device];
    int *ncl_cache = ls.ncl;   // resident clusters for C = 1, 2, 4, 8
    if (!ls.attr) {
        size_t most = 0;
        for (int c = 1; c <= kMaxClusterP; c *= 2) most = smem_bytes_for(c) > most ? smem_bytes_for(c) : most;
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
        if (e != cudaSuccess) return e;
        ls.attr = true;
    }
    if (pl.n < 1 || pl.n > kMaxApplyProj) return cudaErrorInvalidValue;
    for (int j = 0; j < pl.n; ++j)
        if ((reinterpret_cast<uintptr_t>(pl.x[j]) | reinterpret_cast<uintptr_t>(pl.y[j])) & 15u)
            return cudaErrorInvalidValue;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;

    auto clusters = [&](int C, int lg) -> int {
        if (ncl_cache[lg] == 0) {
            attr[1].val.clusterDim.x = C;
            cfg.gridDim = dim3(C * num_sms);
            cfg.dynamicSmemBytes = smem_bytes_for(C);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, prefill_kernel, &cfg) != cudaSuccess) n = 0;
            ncl_cache[lg] = n > 0 ? n : -1;
        }
        return ncl_cache[lg];
    };

    // CTAs per cluster: the C that minimises the modelled time rounds(C) * (1 + R / C), where
    // rounds(C) = ceil(units / resident clusters of C) and R is the time one CTA takes to
    // move a unit's bytes at C = 1 relative to a unit's fixed cost (6 at hidden 4096, in
    // proportion to hidden: the value that picks the fastest of C = 2, 4 and 8 measured on
    // 16 x 512-token segments and on a mixed-iteration layer); ties go to the smaller C.
    // Units are 128-token tiles per projection; the host does not read the segments, so T
    // bounds their number.
    const int units = (T + MT - 1) / MT * pl.n;
    const double R = std::max(2.0, 6.0 * pv.hidden / 4096.0);
    int C = 1, lgC = 0;
    double best = 1e300;
    for (int lg = 0; lg <= 3; ++lg) {
        const int c = 1 << lg;
        if (lg > 0) {
            const int sl = slice_for(pv.hidden, c);
            if (sl < 256 || (c - 1) * sl >= pv.hidden) break;
        }
        const int n = clusters(c, lg);
        if (n <= 0) continue;
        const double cost = (double)((units + n - 1) / n) * (1.0 + R / c);
        if (cost < best - 1e-9) {
            best = cost;
            C = c;
            lgC = lg;
        }
    }
    if (g_forced_cluster > 0) {
        for (lgC = 0; (1 << lgC) < g_forced_cluster; ++lgC) {
        }
        C = 1 << lgC;
        const int sl = slice_for(pv.hidden, C);
        if (C > kMaxClusterP || (C - 1) * sl >= pv.hidden) return cudaErrorInvalidValue;
    }
    int ncl = clusters(C, lgC);
    if (ncl <= 0) ncl = C == 1 ? num_sms : 1;

    PrefillArgs pa;
    memset(&pa, 0, sizeof(pa));
    for (int j = 0; j < pl.n; ++j) {
        cudaError_t e = token_map(&pa.tmap_x[j], pl.x[j], pv.hidden, T);
        if (e != cudaSuccess) return e;
        e = token_map(&pa.tmap_y[j], pl.y[j], pv.hidden, T);
        if (e != cudaSuccess) return e;
        e = token_map(&pa.tmap_ys[j], pl.y[j], pv.hidden, T, 32);
        if (e != cudaSuccess) return e;
        pa.y[j] = reinterpret_cast<__half *>(pl.y[j]);
        pa.proj[j] = pl.proj[j];
    }
    pa.n_proj = pl.n;
    pa.pv = pv;
    pa.idx = idx;
    pa.seg_indptr = seg_indptr;
    pa.scaling = scaling;
    pa.T = T;
    pa.n_seg = n_seg;
    pa.C = C;
    pa.slice = slice_for(pv.hidden, C);
    pa.nt = tslots_for(C);
    // a unit splits into P parts by expand columns only when every CTA of a cluster has at
    // least P column tiles (the last CTA's slice may be shorter)
    {
        const int nkb_min = std::min(pa.slice / KBLK, (pv.hidden - (C - 1) * pa.slice) / KBLK);
        pa.split = !g_prefill_split ? 1 : (nkb_min >= 4 ? 4 : (nkb_min >= 2 ? 2 : 1));
    }

    attr[1].val.clusterDim.x = C;
    cfg.gridDim = dim3(C * ncl);
    cfg.dynamicSmemBytes = smem_bytes_for(C);
    return cudaLaunchKernelEx(&cfg, prefill_kernel, pa);
}

}  // namespace slora

// Test hook: force the prefill kernel's cluster size (1, 2, 4 or 8; 0 = chosen from the
// batch).
extern "C" slora_status slora_debug_set_prefill_cluster(int32_t ctas)
{
    if (ctas != 0 && ctas != 1 && ctas != 2 && ctas != 4 && ctas != 8) return SLORA_ERR_INVALID_ARG;
    slora::g_forced_cluster = ctas;
    return SLORA_OK;
}

// Test hook: allow (1, the default) or forbid (0) splitting a segment unit in two by
// expand columns when the batch leaves clusters idle.
extern "C" slora_status slora_debug_set_prefill_split(int32_t on)
{
    if (on != 0 && on != 1) return SLORA_ERR_INVALID_ARG;
    slora::g_prefill_split = on;
    return SLORA_OK;
}
