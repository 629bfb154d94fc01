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
//     first, then expand items (adapter, 2048 output columns, <= 4 tokens).
//
//   delta_kernel (one persistent CTA per SM): claims items in list order from a global
//     counter.  Warp 0 streams each item's page rows into a 4-stage shared-memory ring
//     with 1-D bulk copies (TMA engine), several tiles ahead of the compute:
//       shrink  u[t][j] = sum_k x[t][k] * At[j][k]     (A^T rows + x rows per K tile;
//               fp32 partials per thread, one butterfly reduce-scatter per warp, written
//               to a small fp32 scratch, then a release increment of the group's counter)
//       expand  y[t][c] = y0[t][c] + s * sum_j u[t][j] * B[j][c]
//               (B row segments per 8-row tile; waits, with a time limit, until every
//               shrink item of its group has been published)
//     Each used adapter page row is read from HBM once per token chunk of its group (the
//     repeats of hot adapters hit L2).  Ranks 1..1024 run in the same launch: the last
//     rank chunk of an adapter simply has fewer rows; nothing in the pool is padded.
//
// Per-token arithmetic is fixed by the thread layout (which K elements a thread sums,
// the butterfly order, the row order of the expand), never by how tokens are grouped,
// so results do not depend on the batch, its order, or the physical pages.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.h"

namespace slora {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int RS = 8;       // A^T rows per shrink item
constexpr int TS = 4;       // tokens per shrink item
constexpr int TE = 4;       // tokens per expand item
constexpr int RB = 8;       // B rows per expand tile
constexpr int KC = 2048;    // K elements per shrink tile (= 8 * kThreads)
constexpr int CE = 2048;    // output columns per expand item (= 8 * kThreads)
constexpr int NS = 4;       // pipeline stages
constexpr int kStageBytes = (RS + TS) * KC * 2;       // 48 KiB
constexpr int kMaxRank = 1024;
constexpr int kUBytes = TE * kMaxRank * 4;            // 16 KiB
constexpr int kSmemBytes = NS * kStageBytes + kUBytes + kWarps * 32 * 4;

constexpr int kPlanThreads = 1024;
constexpr int kMaxPlanTokens = 4096;                  // token-index range per plan
constexpr int kMaxHash = 2 * kMaxPlanTokens;

static_assert(KC == 8 * kThreads && CE == 8 * kThreads, "one 16-byte vector per thread per row");
static_assert(RB * CE * 2 <= kStageBytes, "expand tile fits a stage");
static_assert(RS * TS == 32, "shrink item partials = one value per lane after the butterfly");

struct PlanHeader {
    int32_t n_groups, n_shrink, n_expand, claim;
    int32_t seg_lo, seg_hi, pad0, pad1;
};
struct GroupRec {
    int32_t adapter, tok_begin, n_tok, rank;
    float scaling;
    int32_t u_off;
    int64_t pt_base;  // arena index of this projection's page table
};
struct Item {
    int32_t g, a, t0, nt;  // a = first rank row (shrink) or column chunk (expand)
};

struct PlanLayout {
    PlanHeader *hdr;
    int32_t *tok_order;
    GroupRec *groups;
    int32_t *done;
    Item *items;
    float *u;
    int64_t cap_items;
    int64_t cap_u;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Number of column chunks of the expand.
__host__ __device__ inline int n_col_chunks(int d) { return ceil_div(d, CE); }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

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
    L.cap_u = cap * (int64_t)max_rank;
    L.hdr = (PlanHeader *)take(sizeof(PlanHeader));
    L.tok_order = (int32_t *)take(cap * 4);
    L.groups = (GroupRec *)take(cap * sizeof(GroupRec));
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

struct PlanArgs {
    PoolView pv;
    int32_t proj;
    const int32_t *idx;
    int32_t T;
    const int32_t *seg_indptr;
    int32_t n_seg;
    int32_t t_begin, t_end;
    int32_t hash_size;  // power of two >= 2 * (t_end - t_begin)
    PlanLayout L;
};

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const __grid_constant__ PlanArgs a)
{
    extern __shared__ int plan_smem[];
    const int HS = a.hash_size;
    const int Tc = a.t_end - a.t_begin;
    int *keys = plan_smem;            // [HS] adapter id or -1
    int *gid = keys + HS;             // [HS] group id of an occupied slot
    int *garr = gid + HS;             // [Tc] adapter of group g
    int *cnt = garr + kMaxPlanTokens; // [Tc] tokens per group, then the placement cursor
    short *tslot = reinterpret_cast<short *>(cnt + kMaxPlanTokens);  // [Tc] slot of token
    __shared__ int warp_tot[33];
    __shared__ int s_lo, s_hi, s_G, s_nsh, s_nex;
    const int tid = threadIdx.x;

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
    }
    for (int h = tid; h < HS; h += kPlanThreads)
        keys[h] = -1;
    for (int g = tid; g < Tc; g += kPlanThreads)
        cnt[g] = 0;
    __syncthreads();
    const int lo = s_lo, hi = s_hi;

    // insert the decode tokens of [t_begin, t_end)
    for (int i = tid; i < Tc; i += kPlanThreads) {
        const int t = a.t_begin + i;
        int slot = -1;
        const bool in_seg = t >= lo && t < hi;
        const int ad = a.idx[t];
        // segment tokens run on the tensor cores unless their adapter's rank is too large
        // for that path; segment errors are reported there
        const bool mine = !in_seg || (ad >= 0 && ad < a.pv.max_adapters && a.pv.dir[ad].pt_off >= 0 &&
                                      a.pv.dir[ad].rank > kMaxPrefillRank);
        if (mine) {
            if (ad >= 0 && ad < a.pv.max_adapters) {
                const DirEntry e = a.pv.dir[ad];
                if (e.pt_off >= 0 && e.rank > 0 && e.rank <= kMaxRank) {
                    int h = (int)(((uint32_t)ad * 2654435761u) & (uint32_t)(HS - 1));
                    for (;;) {
                        int k = atomicCAS(&keys[h], -1, ad);
                        if (k == -1 || k == ad) break;
                        h = (h + 1) & (HS - 1);
                    }
                    slot = h;
                } else {
                    set_status(a.pv.status, SLORA_DEV_NOT_RESIDENT);
                }
            } else if (ad != -1) {
                set_status(a.pv.status, SLORA_DEV_BAD_ADAPTER);
            }
        }
        tslot[i] = (short)slot;
    }
    __syncthreads();

    // groups = occupied slots, numbered in slot order
    {
        const int per = HS / kPlanThreads;
        const int h0 = tid * per;
        int c = 0;
        for (int h = h0; h < h0 + per; ++h)
            c += keys[h] != -1;
        int total;
        int base = block_excl_scan(c, warp_tot, &total);
        for (int h = h0; h < h0 + per; ++h) {
            if (keys[h] != -1) {
                gid[h] = base;
                garr[base] = keys[h];
                ++base;
            }
        }
        if (tid == 0) s_G = total;
    }
    __syncthreads();
    const int G = s_G;
    for (int i = tid; i < Tc; i += kPlanThreads)
        if (tslot[i] >= 0)
            atomicAdd(&cnt[gid[tslot[i]]], 1);
    __syncthreads();

    // per-group totals: tokens, shrink items, expand items, u floats
    const int d = a.pv.hidden;
    const int nch = n_col_chunks(d);
    const int per_g = ceil_div(G > 0 ? G : 1, kPlanThreads);
    const int g0 = tid * per_g;
    int my_tok = 0, my_sh = 0, my_ex = 0, my_u = 0;
    for (int g = g0; g < g0 + per_g && g < G; ++g) {
        const int r = a.pv.dir[garr[g]].rank;
        const int n = cnt[g];
        my_tok += n;
        my_sh += ceil_div(r, RS) * ceil_div(n, TS);
        my_ex += nch * ceil_div(n, TE);
        my_u += n * r;
    }
    int tot_tok, tot_sh, tot_ex, tot_u;
    int off_tok = block_excl_scan(my_tok, warp_tot, &tot_tok);
    int off_sh = block_excl_scan(my_sh, warp_tot, &tot_sh);
    int off_ex = block_excl_scan(my_ex, warp_tot, &tot_ex);
    int off_u = block_excl_scan(my_u, warp_tot, &tot_u);
    if (tid == 0) {
        s_nsh = tot_sh;
        s_nex = tot_ex;
    }
    __syncthreads();
    if ((int64_t)tot_sh + tot_ex > a.L.cap_items || (int64_t)tot_u > a.L.cap_u) {
        // cannot happen with the host's sizing; refuse the batch rather than overrun
        if (tid == 0) {
            set_status(a.pv.status, SLORA_DEV_BAD_SEGMENT);
            a.L.hdr->n_groups = 0;
            a.L.hdr->n_shrink = 0;
            a.L.hdr->n_expand = 0;
            a.L.hdr->claim = 0;
        }
        return;
    }
    for (int g = g0; g < g0 + per_g && g < G; ++g) {
        const int ad = garr[g];
        const DirEntry e = a.pv.dir[ad];
        const int r = e.rank, n = cnt[g];
        GroupRec rec;
        rec.adapter = ad;
        rec.tok_begin = off_tok;
        rec.n_tok = n;
        rec.rank = r;
        rec.scaling = e.scaling;
        rec.u_off = off_u;
        rec.pt_base = e.pt_off + (int64_t)a.proj * 2 * r;
        a.L.groups[g] = rec;
        a.L.done[g] = 0;
        const int ntc_s = ceil_div(n, TS), ntc_e = ceil_div(n, TE);
        for (int jc = 0; jc < ceil_div(r, RS); ++jc)
            for (int tc = 0; tc < ntc_s; ++tc)
                a.L.items[off_sh++] = Item{g, jc * RS, tc * TS, min(TS, n - tc * TS)};
        for (int c = 0; c < nch; ++c)
            for (int tc = 0; tc < ntc_e; ++tc)
                a.L.items[tot_sh + off_ex++] = Item{g, c, tc * TE, min(TE, n - tc * TE)};
        off_tok += n;
        off_u += n * r;
    }
    __syncthreads();
    // token placement: cnt becomes the cursor
    for (int g = tid; g < G; g += kPlanThreads)
        cnt[g] = 0;
    __syncthreads();
    for (int i = tid; i < Tc; i += kPlanThreads) {
        const int h = tslot[i];
        if (h >= 0) {
            const int g = gid[h];
            const int pos = __ldcg(&a.L.groups[g].tok_begin) + atomicAdd(&cnt[g], 1);
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

__device__ __forceinline__ int item_tiles(const GroupRec &g, bool shrink, int d)
{
    return shrink ? ceil_div(d, KC) : ceil_div(g.rank, RB);
}

__global__ void __launch_bounds__(kThreads, 1) delta_kernel(const __grid_constant__ DeltaArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *stages = smem;
    float *u_s = reinterpret_cast<float *>(smem + NS * kStageBytes);
    float *red = u_s + TE * kMaxRank;
    __shared__ __align__(8) uint64_t full[NS];
    __shared__ int tile_item[NS], tile_sub[NS];
    __shared__ int s_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.pv.hidden;
    const __half *pool = reinterpret_cast<const __half *>(a.pv.pool);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s)
            mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();   // the plan of this batch is complete and visible
    griddep_launch_dependents();

    const int n_sh = a.L.hdr->n_shrink;
    const int n_tot = n_sh + a.L.hdr->n_expand;

    // ---- producer state (warp 0; lane 0 authoritative) ----
    int p_item = -1, p_sub = 0, p_nsub = 0;

    auto produce = [&](int s) {
        int item = 0, sub = 0;
        if (lane == 0) {
            if (p_item < 0 || (p_item < n_tot && p_sub >= p_nsub)) {
                p_item = atomicAdd(&a.L.hdr->claim, 1);
                if (p_item > n_tot) p_item = n_tot;
                p_sub = 0;
                if (p_item < n_tot) {
                    const Item it = a.L.items[p_item];
                    p_nsub = item_tiles(a.L.groups[it.g], p_item < n_sh, d);
                }
            }
            item = p_item;
            sub = p_sub;
            if (p_item < n_tot) ++p_sub;
        }
        item = __shfl_sync(0xffffffffu, item, 0);
        sub = __shfl_sync(0xffffffffu, sub, 0);
        if (item >= n_tot) {
            if (lane == 0) {
                tile_item[s] = -1;
                mbar_arrive(&full[s]);
            }
            return;
        }
        const Item it = a.L.items[item];
        const GroupRec g = a.L.groups[it.g];
        uint8_t *st = stages + s * kStageBytes;
        const __half *src = nullptr;
        uint32_t bytes = 0;
        void *dst = nullptr;
        if (item < n_sh) {
            const int k0 = sub * KC;
            const int kc = min(KC, d - k0);
            const int nrows = min(RS, g.rank - it.a);
            if (lane < nrows) {
                const int32_t page = a.pv.pt_arena[g.pt_base + it.a + lane];
                if (page >= 0 && page < a.pv.num_pages) {
                    src = pool + (int64_t)page * d + k0;
                    bytes = kc * 2;
                    dst = st + lane * (KC * 2);
                } else {
                    set_status(a.pv.status, SLORA_DEV_BAD_PAGE);
                }
            } else if (lane >= RS && lane < RS + it.nt) {
                const int tok = a.L.tok_order[g.tok_begin + it.t0 + (lane - RS)];
                src = a.x + (int64_t)tok * d + k0;
                bytes = kc * 2;
                dst = st + lane * (KC * 2);
            }
        } else {
            const int c0 = it.a * CE;
            const int ce = min(CE, d - c0);
            const int j0 = sub * RB;
            const int nrows = min(RB, g.rank - j0);
            if (lane < nrows) {
                const int32_t page = a.pv.pt_arena[g.pt_base + g.rank + j0 + lane];
                if (page >= 0 && page < a.pv.num_pages) {
                    src = pool + (int64_t)page * d + c0;
                    bytes = ce * 2;
                    dst = st + lane * (CE * 2);
                } else {
                    set_status(a.pv.status, SLORA_DEV_BAD_PAGE);
                }
            }
        }
        uint32_t total = bytes;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            total += __shfl_xor_sync(0xffffffffu, total, o);
        if (lane == 0) {
            tile_item[s] = item;
            tile_sub[s] = sub;
            if (total > 0)
                mbar_arrive_expect_tx(&full[s], total);
            else
                mbar_arrive(&full[s]);
        }
        __syncwarp();
        if (bytes > 0)
            bulk_g2s(dst, src, bytes, &full[s]);
    };

    if (warp == 0)
        for (int s = 0; s < NS; ++s)
            produce(s);

    float acc[TS][RS];   // shrink: [token][row]; expand: [token][column of the vector]
    uint4 yv[TE];
    int cur_item = -1;
    GroupRec cg;
    Item cit;
    bool ok = true;
    int c = 0;
    bool timed_out = false;

    for (;; ++c) {
        const int s = c % NS;
        const uint32_t parity = (uint32_t)(c / NS) & 1u;
        if (!mbar_wait_bounded(&full[s], parity, a.pv.status)) {
            timed_out = true;
            break;
        }
        const int item = tile_item[s];
        const int sub = tile_sub[s];
        if (item < 0)
            break;
        const uint8_t *st = stages + s * kStageBytes;
        const bool shrink = item < n_sh;
        if (item != cur_item) {
            // ---- item start ----
            cur_item = item;
            cit = a.L.items[item];
            cg = a.L.groups[cit.g];
#pragma unroll
            for (int t = 0; t < TS; ++t)
#pragma unroll
                for (int j = 0; j < RS; ++j)
                    acc[t][j] = 0.f;
            ok = true;
            if (!shrink) {
                const int c0 = cit.a * CE;
                const bool active = c0 + 8 * tid < d;
#pragma unroll
                for (int t = 0; t < TE; ++t) {
                    if (t < cit.nt && active) {
                        const int tok = a.L.tok_order[cg.tok_begin + cit.t0 + t];
                        yv[t] = *reinterpret_cast<const uint4 *>(a.y + (int64_t)tok * d + c0 + 8 * tid);
                    }
                }
                // wait until every shrink item of the group has published its u values
                if (tid == 0) {
                    const int need = ceil_div(cg.rank, RS) * ceil_div(cg.n_tok, TS);
                    int flag = 1;
                    if (ld_acquire_gpu(&a.L.done[cit.g]) < need) {
                        const uint64_t t0 = global_timer_ns();
                        for (;;) {
                            __nanosleep(64);
                            if (ld_acquire_gpu(&a.L.done[cit.g]) >= need) break;
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
                const int r = cg.rank;
                const int nu = cit.nt * r;
                const float *ug = a.L.u + cg.u_off + (int64_t)cit.t0 * r;
                for (int i = tid; i < nu; i += kThreads)
                    u_s[i] = __ldcg(ug + i);
                __syncthreads();
            }
        }
        // ---- tile compute ----
        if (shrink) {
            const int k0 = sub * KC;
            const int nrows = min(RS, cg.rank - cit.a);
            if (k0 + 8 * tid < d) {
                float xf[TS][8];
#pragma unroll
                for (int t = 0; t < TS; ++t)
                    if (t < cit.nt)
                        h8_to_f(lds128(st + (RS + t) * (KC * 2) + 16 * tid), xf[t]);
#pragma unroll
                for (int j = 0; j < RS; ++j) {
                    if (j < nrows) {
                        float af[8];
                        h8_to_f(lds128(st + j * (KC * 2) + 16 * tid), af);
#pragma unroll
                        for (int t = 0; t < TS; ++t) {
                            if (t < cit.nt) {
                                float v = acc[t][j];
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    v = fmaf(xf[t][e], af[e], v);
                                acc[t][j] = v;
                            }
                        }
                    }
                }
            }
        } else {
            const int c0 = cit.a * CE;
            const int j0 = sub * RB;
            const int nrows = min(RB, cg.rank - j0);
            const int r = cg.rank;
            if (c0 + 8 * tid < d) {
#pragma unroll
                for (int j = 0; j < RB; ++j) {
                    if (j < nrows) {
                        float bf[8];
                        h8_to_f(lds128(st + j * (CE * 2) + 16 * tid), bf);
#pragma unroll
                        for (int t = 0; t < TE; ++t) {
                            if (t < cit.nt) {
                                const float uu = u_s[t * r + j0 + j];
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    acc[t][e] = fmaf(uu, bf[e], acc[t][e]);
                            }
                        }
                    }
                }
            }
        }
        const bool last = sub == item_tiles(cg, shrink, d) - 1;
        if (last) {
            if (shrink) {
                // ---- reduce the 32 partials over the CTA, publish u ----
                float v[32];
#pragma unroll
                for (int t = 0; t < TS; ++t)
#pragma unroll
                    for (int j = 0; j < RS; ++j)
                        v[t * RS + j] = acc[t][j];
                const float ws = warp_reduce_scatter32(v);
                red[warp * 32 + lane] = ws;
                __syncthreads();
                if (tid < 32) {
                    float tot = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w)
                        tot += red[w * 32 + tid];
                    const int t = tid / RS, j = tid % RS;
                    if (t < cit.nt && cit.a + j < cg.rank)
                        __stcg(a.L.u + cg.u_off + (int64_t)(cit.t0 + t) * cg.rank + cit.a + j, tot);
                }
                __syncthreads();
                if (tid == 0) {
                    __threadfence();
                    atomicAdd(&a.L.done[cit.g], 1);
                }
            } else if (ok) {
                const int c0 = cit.a * CE;
                if (c0 + 8 * tid < d) {
                    const float sc = a.scaling ? a.scaling[cg.adapter] : cg.scaling;
#pragma unroll
                    for (int t = 0; t < TE; ++t) {
                        if (t < cit.nt) {
                            const int tok = a.L.tok_order[cg.tok_begin + cit.t0 + t];
                            float y0f[8], out[8];
                            h8_to_f(yv[t], y0f);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                out[e] = fmaf(sc, acc[t][e], y0f[e]);
                            *reinterpret_cast<uint4 *>(a.y + (int64_t)tok * d + c0 + 8 * tid) = f_to_h8(out);
                        }
                    }
                }
            }
        }
        __syncthreads();   // stage s and the item scratch are free
        if (warp == 0)
            produce(s);
    }
    if (timed_out) {
        // Copies of this CTA may still be in flight into the stages ahead: wait for each
        // (bounded) before the CTA's shared memory is released.
        for (int k = 1; k < NS; ++k) {
            const int cc = c + k;
            mbar_wait_bounded(&full[cc % NS], (uint32_t)(cc / NS) & 1u, a.pv.status);
        }
    }
}

}  // namespace

size_t plan_scratch_bytes(int32_t T, int32_t max_rank, int32_t hidden)
{
    size_t total = 0;
    const int32_t cap = T < kMaxPlanTokens ? T : kMaxPlanTokens;
    carve(nullptr, cap, max_rank, hidden, &total);
    return total;
}

cudaError_t launch_lora_apply(const PoolView &pv, int32_t proj, const uint16_t *x, uint16_t *y,
                              int32_t T, const int32_t *idx, const int32_t *seg_indptr,
                              int32_t n_seg, const float *scaling, const PlanScratch &scratch,
                              int num_sms, cudaStream_t stream, int *launches)
{
    static bool attrs_set = false;
    if (!attrs_set) {
        cudaError_t e = cudaFuncSetAttribute(delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (2 * kMaxHash + 2 * kMaxPlanTokens) * 4 + kMaxPlanTokens * 2);
        if (e != cudaSuccess) return e;
        attrs_set = true;
    }
    const int32_t cap = scratch.cap_tokens < kMaxPlanTokens ? scratch.cap_tokens : kMaxPlanTokens;
    PlanLayout L = carve(scratch.base, cap, scratch.max_rank, pv.hidden, nullptr);

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    for (int32_t tb = 0; tb < T; tb += kMaxPlanTokens) {
        const int32_t te = tb + kMaxPlanTokens < T ? tb + kMaxPlanTokens : T;
        int hs = 1024;
        while (hs < 2 * (te - tb)) hs <<= 1;
        PlanArgs pa{pv, proj, idx, T, seg_indptr, n_seg, tb, te, hs, L};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPlanThreads);
        cfg.dynamicSmemBytes = (size_t)(2 * hs + 2 * kMaxPlanTokens) * 4 + kMaxPlanTokens * 2;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, plan_kernel, pa);
        if (e != cudaSuccess) return e;
        *launches += 1;

        DeltaArgs da{pv, reinterpret_cast<const __half *>(x), reinterpret_cast<__half *>(y), scaling, L};
        cudaLaunchConfig_t cfg2 = {};
        cfg2.gridDim = dim3(num_sms);
        cfg2.blockDim = dim3(kThreads);
        cfg2.dynamicSmemBytes = kSmemBytes;
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
