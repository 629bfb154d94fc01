/*
 * slora.h -- C ABI of libslora.so: a Unified Paging pool of LoRA adapter rows and
 * the heterogeneous-rank batched LoRA delta over it, on one GB300 (sm_103a).
 *
 * What the library computes (for every token t whose adapter is a):
 *
 *     y[t] <- y[t] + s_a * (x[t] A_a) B_a
 *
 * with A_a (hidden x r_a) and B_a (r_a x hidden) fp16, accumulation in fp32 and one
 * final rounding of y to fp16.  Sources: S-LoRA: Serving Thousands of Concurrent LoRA
 * Adapters (explainer), "What this paper explains" (shapes of A and B; the delta is
 * kept separate from the shared base) and "The mechanism" (one base, the delta x A B
 * computed on the fly per request's adapter; a host-resident adapter store; Unified
 * Paging of adapter tiles and KV blocks in one pool with a block table); S-LoRA:
 * Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU, section 2 (the
 * per-token loop with a per-adapter scaling) and section 3 (one kernel invocation for a
 * batch of heterogeneous-rank adapters, gathering hidden states and matching them to
 * the adapters' pages through the paging table).
 *
 * Pool layout.  The pool is one device allocation of `num_pages` fixed-size pages;
 * a page holds one fp16 row of length `hidden` (hidden * 2 bytes).  An adapter with
 * rank r occupies 2 * r * n_proj pages: for each projection p, the r rows of A^T
 * (row j = column j of A) followed by the r rows of B.  Its page table lists those
 * pages in that order: pt[p][0..r) for A^T, pt[p][r..2r) for B.  Pages are handed out
 * from one free list shared with the caller's KV blocks (slora_pages_alloc/free), so
 * adapter pages and KV pages interleave in the pool (Unified Paging: explainer, "The
 * mechanism" and "What to notice when reading"; S-LoRA: Multiplexing ..., section 2).
 *
 * Conventions for every call:
 *   - Every call returns slora_status; SLORA_OK is 0.  No C++ exception crosses the
 *     boundary.  slora_last_error() gives a message for the calling thread's most
 *     recent failure.
 *   - "host" pointers are ordinary CPU pointers; "device" pointers are CUDA device
 *     pointers on the pool's device.  The caller owns every buffer it passes; the pool
 *     owns its device pool, page tables, adapter directory, pinned host store, side
 *     stream and events.
 *   - slora_stream_t is a cudaStream_t (NULL = the legacy default stream).  Calls that
 *     take a stream enqueue work on it and return without waiting, unless noted.
 *   - One pool is used by one host thread at a time.
 *   - Device-side checks never trap: a kernel that meets a bad adapter index, a
 *     non-resident adapter, an out-of-range page or a segment whose tokens disagree on
 *     their adapter records a code in the pool's device status word and skips that
 *     work (such a segment as a whole); slora_get_device_status() reads and clears it.
 */
#ifndef SLORA_H
#define SLORA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct slora_pool *slora_pool_t;
typedef struct slora_pagealloc *slora_pagealloc_t;
typedef void *slora_stream_t; /* a cudaStream_t */

typedef enum slora_status {
    SLORA_OK = 0,
    SLORA_ERR_INVALID_ARG = 1,      /* bad pointer, size, id, rank or projection */
    SLORA_ERR_POOL_FULL = 2,        /* not enough free pages (nothing was allocated) */
    SLORA_ERR_NOT_REGISTERED = 3,   /* adapter id not in the host store */
    SLORA_ERR_NOT_RESIDENT = 4,     /* adapter id not loaded in the pool */
    SLORA_ERR_ALREADY_RESIDENT = 5, /* single-adapter load of a resident adapter */
    SLORA_ERR_CUDA = 6,             /* a CUDA runtime call failed (see slora_last_error) */
    SLORA_ERR_DEVICE_CHECK = 7,     /* a kernel skipped work after a failed check */
    SLORA_ERR_DEVICE_TIMEOUT = 8,   /* a bounded device wait gave up */
    SLORA_ERR_HOST_ALLOC = 9,       /* pinned or ordinary host allocation failed */
    SLORA_ERR_ALREADY_REGISTERED = 10,
    SLORA_ERR_UNSUPPORTED = 11      /* device is not sm_103 or a size exceeds a kernel limit */
} slora_status;

/* Device status codes (slora_get_device_status), first error wins. */
#define SLORA_DEV_OK 0
#define SLORA_DEV_BAD_ADAPTER 1   /* token adapter index >= max_adapters or < -1 */
#define SLORA_DEV_NOT_RESIDENT 2  /* token's adapter has no pages in the pool */
#define SLORA_DEV_BAD_PAGE 3      /* page-table entry outside [0, num_pages) */
#define SLORA_DEV_BAD_SEGMENT 4   /* segment tokens disagree on their adapter, or bad bounds */
#define SLORA_DEV_TIMEOUT 5       /* a bounded wait inside a kernel gave up */

const char *slora_status_str(slora_status s);
/* Message of the calling thread's last failed call ("" if none).  Valid until the
 * thread's next failing call. */
const char *slora_last_error(void);
/* Library version as major * 10000 + minor * 100 + patch: 200 (0.2.0).  0.2.0 adds
 * slora_lora_apply_multi, residency under pool pressure (slora_adapters_acquire /
 * release, slora_pages_alloc_evict, slora_pool_get_stats, slora_lru_*) and the padded
 * batched-GEMM comparison path (slora_lora_apply_bmm). */
int32_t slora_version(void);

/* ---------------------------------------------------------------------------
 * Host page allocator.  The free list behind the pool, usable without a GPU.
 * Pages are int32 indices in [0, num_pages).  shuffle_seed != 0 permutes the free
 * list once at creation (a seeded Fisher-Yates shuffle driven by splitmix64) so that
 * consecutive allocations land on scattered pages; 0 keeps ascending order.
 * alloc() pops n pages or fails with SLORA_ERR_POOL_FULL and allocates nothing.
 * free() returns pages; a page that is out of range or not allocated fails the whole
 * call with SLORA_ERR_INVALID_ARG before any page is returned.
 * ------------------------------------------------------------------------- */
slora_status slora_pagealloc_create(int64_t num_pages, uint64_t shuffle_seed,
                                    slora_pagealloc_t *out);
slora_status slora_pagealloc_destroy(slora_pagealloc_t a);
slora_status slora_pagealloc_alloc(slora_pagealloc_t a, int64_t n, int32_t *out_pages /*host [n]*/);
slora_status slora_pagealloc_free(slora_pagealloc_t a, int64_t n, const int32_t *pages /*host [n]*/);
slora_status slora_pagealloc_num_free(slora_pagealloc_t a, int64_t *out);

/* ---------------------------------------------------------------------------
 * Host-only recency index of resident adapters: the eviction policy the pool applies
 * under pressure (slora_adapters_acquire, slora_pages_alloc_evict), exposed like the page
 * allocator for callers that keep their own residency and for tests without a GPU.
 * (The explainer's "The mechanism": adapters the running batches do not use can leave
 * GPU memory; the pages do not name a policy, so this is least-recently-used among the
 * adapters no running batch holds.)
 *   insert()  id becomes present, unpinned, most recently used (no-op if present)
 *   remove()  SLORA_ERR_INVALID_ARG if absent or pinned
 *   touch()   most recently used; pin() / unpin() count holds (an unpin without a pin is
 *             SLORA_ERR_INVALID_ARG); absent ids are SLORA_ERR_INVALID_ARG
 *   victims() up to max_out present, unpinned ids not in exclude[], least recently used
 *             first, into out_ids (host [max_out]); *out_n = how many
 * ------------------------------------------------------------------------- */
typedef struct slora_lru *slora_lru_t;
slora_status slora_lru_create(slora_lru_t *out);
slora_status slora_lru_destroy(slora_lru_t l);
slora_status slora_lru_insert(slora_lru_t l, int32_t id);
slora_status slora_lru_remove(slora_lru_t l, int32_t id);
slora_status slora_lru_touch(slora_lru_t l, int32_t id);
slora_status slora_lru_pin(slora_lru_t l, int32_t id);
slora_status slora_lru_unpin(slora_lru_t l, int32_t id);
slora_status slora_lru_victims(slora_lru_t l, int32_t n_exclude, const int32_t *exclude /*host*/,
                               int32_t max_out, int32_t *out_ids /*host*/, int32_t *out_n);

/* ---------------------------------------------------------------------------
 * Pool.
 *   device        CUDA device ordinal (must be compute capability 10.3)
 *   hidden        row length; a multiple of 64, 64 <= hidden <= 8192 (the decode kernel
 *                 cuts a row into at most 8 blocks of at most 1024 elements)
 *   num_pages     pool slots, 1 <= num_pages < 2^31; pool bytes = num_pages * hidden * 2
 *   n_proj        projections per adapter (e.g. layers x {q,k,v,o}); >= 1
 *   max_adapters  adapter ids are 0 .. max_adapters-1
 *   shuffle_seed  free-list permutation (see the page allocator)
 * Allocates the device pool, page-table arena, directory and status word, and a
 * non-blocking side stream for adapter uploads.  destroy() waits for the pool's own
 * streams, then frees everything it owns, including the pinned host store.
 * ------------------------------------------------------------------------- */
slora_status slora_pool_create(int device, int32_t hidden, int64_t num_pages, int32_t n_proj,
                               int32_t max_adapters, uint64_t shuffle_seed, slora_pool_t *out);
slora_status slora_pool_destroy(slora_pool_t pool);
/* Free slots in the pool (host bookkeeping; no device sync). */
slora_status slora_pool_num_free(slora_pool_t pool, int64_t *out);
/* Device address of page 0 (page i starts at base + i * hidden * 2 bytes). */
slora_status slora_pool_base(slora_pool_t pool, void **out);

/* KV side of the unified allocator.  pages_alloc pops n slots from the same free list
 * adapters use and writes them to out_pages (host).  pages_free returns KV slots; it
 * records an event on `stream` after which the slots may be rewritten by adapter
 * loads, so work already enqueued on `stream` may still read them. */
slora_status slora_pages_alloc(slora_pool_t pool, int64_t n, int32_t *out_pages);
slora_status slora_pages_free(slora_pool_t pool, int64_t n, const int32_t *pages,
                              slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host adapter store (explainer, "The mechanism": all adapters live in host memory and
 * only those the running batch needs are fetched to the GPU).
 * register() copies the caller's factors into pinned host memory owned by the pool:
 *   At_host  fp16 [n_proj][rank][hidden]  rows of A^T (row j = column j of A)
 *   B_host   fp16 [n_proj][rank][hidden]  rows of B
 *   rank     1 <= rank <= 1024; scaling is the default s for this adapter
 * The caller's buffers may be freed when the call returns.
 * unregister() evicts the adapter first if it is resident (see evict).
 * ------------------------------------------------------------------------- */
slora_status slora_adapter_register(slora_pool_t pool, int32_t adapter_id, int32_t rank,
                                    float scaling, const uint16_t *At_host,
                                    const uint16_t *B_host);
slora_status slora_adapter_unregister(slora_pool_t pool, int32_t adapter_id,
                                      slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Load / evict (explainer, "Algorithm / figure walkthrough" steps 2 and 4; "The
 * mechanism": unused adapters leave GPU memory and stay on the host).
 *
 * load() takes 2 * rank * n_proj pages from the free list, writes the adapter's page
 * table into its pinned host copy, and on the pool's side stream runs the load kernel,
 * which reads the pinned store rows and their page ids straight from host memory
 * (over the CPU-GPU link: no staging buffer, no copy per adapter; the copy-engine mode
 * of slora_pool_set_load_mode stages the rows in device memory first) and writes each row
 * to its page, bit for bit, and the page ids to the device page-table arena; then it
 * publishes the directory entry.  `stream` then waits on an event recorded after that
 * work, so kernels enqueued later on `stream` see the adapter; the host call does not
 * wait for the upload.  The pinned store and page table of an adapter are not
 * rewritten or freed while a load kernel may still read them.  The side stream first waits for
 * the most recent page release (evict / pages_free), so slots freed by work still in
 * flight are not overwritten early.
 * adapters_load() does the same for a list: ids that are already resident are
 * skipped; if the missing ones do not all fit, nothing is loaded and
 * SLORA_ERR_POOL_FULL is returned.
 * evict() enqueues on `stream` the clearing of the directory entry, returns the
 * adapter's pages to the free list and records the release event on `stream`.
 * adapters_evict() does the same for a list with one directory update for all of it:
 * ids that are not resident (or repeated) are skipped; an id that is not registered
 * returns SLORA_ERR_NOT_REGISTERED before anything is evicted.
 * ------------------------------------------------------------------------- */
slora_status slora_adapter_load(slora_pool_t pool, int32_t adapter_id, slora_stream_t stream);
slora_status slora_adapters_load(slora_pool_t pool, int32_t n, const int32_t *adapter_ids /*host*/,
                                 slora_stream_t stream);
slora_status slora_adapter_evict(slora_pool_t pool, int32_t adapter_id, slora_stream_t stream);
slora_status slora_adapters_evict(slora_pool_t pool, int32_t n, const int32_t *adapter_ids /*host*/,
                                  slora_stream_t stream);
slora_status slora_adapter_is_resident(slora_pool_t pool, int32_t adapter_id, int32_t *out);

/* ---------------------------------------------------------------------------
 * Load path selection (explainer, "Algorithm / figure walkthrough" step 2: the next
 * iteration's adapters are prefetched into the pool while the current one computes;
 * "Limitations": host bandwidth bounds how fast adapters swap in).
 *
 * mode SLORA_LOAD_ZERO_COPY (the default): the load kernel reads the pinned store over
 *   the CPU-GPU link itself, as described above.  Its CTAs take SM time from kernels
 *   that run beside a load.
 * mode SLORA_LOAD_COPY_ENGINE: every adapter's pinned store block goes to a device
 *   staging ring with one cudaMemcpyAsync on the side stream (the copy engines move it;
 *   no SM takes part), then one load kernel per ring-full of adapters writes the rows
 *   from the staging ring (HBM) to their pages.  The ring is reused in stream order.
 * staging_bytes: the ring's size for the copy-engine mode (0: 256 MiB); it grows, with a
 *   synchronisation of the side stream, when a load meets an adapter larger than it.
 *   This call allocates the ring (cudaMalloc) when the mode needs one and frees it when
 *   the mode no longer does, after the side stream's pending work.  Results of later
 *   loads do not depend on the mode: both write the same bits to the same pages.
 * Returns SLORA_ERR_INVALID_ARG for another mode or a negative size.
 * ------------------------------------------------------------------------- */
enum { SLORA_LOAD_ZERO_COPY = 0, SLORA_LOAD_COPY_ENGINE = 1 };
slora_status slora_pool_set_load_mode(slora_pool_t pool, int32_t mode, int64_t staging_bytes);
slora_status slora_pool_get_load_mode(slora_pool_t pool, int32_t *mode, int64_t *staging_bytes);
/* Measurement hook.  event: a cudaEvent_t created by the caller on the pool's device, or
 * NULL to clear.  While set, every load that has work records it on the pool's side
 * stream before that work, so the caller can see when a load started relative to work on
 * its own streams.  The pool does not take ownership.  The S-LoRA pages have no
 * counterpart for it. */
slora_status slora_pool_set_load_start_event(slora_pool_t pool, void *event);

/* ---------------------------------------------------------------------------
 * Residency under pool pressure (explainer, "The mechanism": adapters the running
 * batches do not use leave GPU memory and stay on the host; "What to notice when
 * reading": KV blocks and adapters share the pool).  The policy is least recently used
 * among the resident adapters that no running batch holds (see slora_lru_*).
 *
 * adapters_acquire(): makes every listed id resident and holds it (a pin count) until
 *   released.  Missing adapters are loaded as slora_adapters_load does; if the free pages
 *   do not suffice, the least recently acquired (or loaded) resident adapters that are
 *   neither held nor listed are evicted first, on `stream`, so their pages are reused only
 *   after the work enqueued earlier on `stream`.  The listed ids become the most recently
 *   used, later ones in the list more recent.  If even evicting every such adapter would
 *   not free enough pages, SLORA_ERR_POOL_FULL is returned and nothing changes.
 * adapters_release(): drops one hold of each listed id (a repeated id counts once);
 *   SLORA_ERR_INVALID_ARG, with no change, if an id is not held.  Release after
 *   enqueuing the batch's work: later evictions on the same stream follow it.
 * pages_alloc_evict(): slora_pages_alloc for KV blocks that grow into the adapters' share:
 *   evicts least recently used adapters that no batch holds, on `stream`, until n pages are
 *   free; SLORA_ERR_POOL_FULL (nothing changes) if the held adapters leave too few.  The
 *   pages may have held adapter rows until this point of `stream`: write them from work
 *   enqueued on `stream` after the call.
 * slora_adapter_evict / slora_adapters_evict refuse a held adapter (SLORA_ERR_INVALID_ARG).
 * pool_get_stats(): free pages, resident and held adapters, and the adapters loaded and
 *   evicted since the pool was created.
 * ------------------------------------------------------------------------- */
typedef struct slora_pool_stats {
    int64_t free_pages;
    int64_t resident_adapters;
    int64_t pinned_adapters;
    int64_t adapters_loaded;
    int64_t adapters_evicted;
} slora_pool_stats;
slora_status slora_adapters_acquire(slora_pool_t pool, int32_t n, const int32_t *adapter_ids /*host*/,
                                    slora_stream_t stream);
slora_status slora_adapters_release(slora_pool_t pool, int32_t n, const int32_t *adapter_ids /*host*/);
slora_status slora_pages_alloc_evict(slora_pool_t pool, int64_t n, int32_t *out_pages /*host [n]*/,
                                     slora_stream_t stream);
slora_status slora_pool_get_stats(slora_pool_t pool, slora_pool_stats *out);

/* ---------------------------------------------------------------------------
 * The hot path: y += s * (x A) B for a batch of tokens, each with its own adapter.
 *
 *   proj               projection index, 0 <= proj < n_proj
 *   x                  device fp16 [T][hidden], row-major, 16-byte aligned
 *   y                  device fp16 [T][hidden], in/out (y0 in, y0 + delta out); may not
 *                      alias x
 *   T                  tokens, 0 <= T <= 1 << 20 (T = 0 is a no-op)
 *   token_adapter_idx  device int32 [T]; adapter id per token, -1 = no adapter (y kept)
 *   seg_indptr         device int32 [n_seg + 1] or NULL.  Tokens in
 *                      [seg_indptr[i], seg_indptr[i+1]) form prefill segment i; every
 *                      token of a segment must carry the same adapter id.  Segments
 *                      run as dense contractions on the tensor cores (the one place the
 *                      work is a real GEMM); every other token takes the decode path.
 *                      The host reads nothing from it.
 *   n_seg              number of segments (0 if seg_indptr is NULL)
 *   scaling            device float [max_adapters] overriding the registered scaling,
 *                      or NULL to use the registered values
 *   stream             work is enqueued on this stream; nothing waits
 *
 * Tokens with a non-resident or out-of-range adapter are skipped (y unchanged) and
 * set a device status code.  A decode token's result does not depend on the other
 * tokens in the batch, their order, or which pages hold its adapter.  A segment token's
 * result is the same up to the order of the fp32 partial sums of x A: the segment
 * kernel splits hidden over 1, 2, 4 or 8 CTAs, chosen from T, and adds their partial
 * products in CTA order.
 * Scratch: the pool keeps device scratch for the token plan, the decode kernel's work list
 * and the fp32 partial sums of x A its work units exchange, sized on first use and grown
 * when a larger T, more projections per call or a larger registered rank arrives (a
 * growth synchronises the pool's device).
 * Every entry point that works on a pool makes the pool's device current for the call and
 * gives the calling thread its previous current device back before it returns.
 * ------------------------------------------------------------------------- */
slora_status slora_lora_apply(slora_pool_t pool, int32_t proj, const void *x, void *y, int32_t T,
                              const int32_t *token_adapter_idx, const int32_t *seg_indptr,
                              int32_t n_seg, const float *scaling, slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * slora_lora_apply_multi: the same computation as n calls of slora_lora_apply that share
 * the tokens, their adapter ids and segments, one call per entry j with projection
 * projs[j], input x[j] and in/out y[j] (S-LoRA: Multiplexing Thousands of Fine-Tuned
 * Adapters on a Single GPU, section 3: the LoRA computation of every projection of a
 * layer, for a batch of requests with different adapters).  A layer's q, k, v and o
 * projections use the same batch, so one call makes one token plan and launches one
 * decode kernel and one segment kernel for all of them, instead of n of each.
 *
 *   n       entries, 1 <= n <= 8
 *   projs   host int32 [n], each 0 <= projs[j] < n_proj; an index may repeat
 *   x       host array [n] of device pointers, fp16 [T][hidden], 16-byte aligned; entries
 *           may share one buffer (q, k and v read the same hidden states)
 *   y       host array [n] of device pointers, fp16 [T][hidden], in/out, 16-byte aligned;
 *           the y buffers must not overlap each other or any x
 *   T, token_adapter_idx, seg_indptr, n_seg, scaling, stream: as for slora_lora_apply.
 *
 * Every decode token's result is bit for bit that of the separate calls.  A segment
 * token's result is too when the segment kernel uses the same number of CTAs per
 * cluster (it is chosen from T * n here, from T in a single call; the test hook
 * slora_debug_set_prefill_cluster fixes it); otherwise it differs only in the order of
 * the fp32 partial sums of x A.  The host arrays are read during the call only.
 * Errors: SLORA_ERR_INVALID_ARG for n out of range, a null array or pointer, a bad
 * projection index, misalignment, or a y equal to another entry's y or to any x
 * (checked on the pointers; overlapping ranges are the caller's error); nothing is
 * launched then.
 * ------------------------------------------------------------------------- */
slora_status slora_lora_apply_multi(slora_pool_t pool, int32_t n, const int32_t *projs /*host*/,
                                    const void *const *x /*host array*/, void *const *y /*host array*/,
                                    int32_t T, const int32_t *token_adapter_idx,
                                    const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                                    slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * A batch planned once and applied to every layer of an iteration.
 *
 * A serving iteration runs one batch through every layer, so the tokens and their adapters
 * (one batch mixes requests of many adapters: S-LoRA: Serving Thousands of Concurrent LoRA
 * Adapters (explainer), "The mechanism") are the same in every layer.  slora_plan_create
 * makes the token plan of the decode path once (the grouping of the decode tokens by
 * adapter, the work list, the adapters' page-table bases and scaling); slora_plan_apply
 * then runs one layer: the decode kernel over the stored plan and the segments'
 * tensor-core kernel, without the plan kernel.  Its results are bit for bit those of
 * slora_lora_apply_multi with the same arguments.
 *
 *   n_slots            projections each apply covers (1..8), as n of slora_lora_apply_multi
 *   T, token_adapter_idx, seg_indptr, n_seg, scaling
 *                      as for slora_lora_apply_multi, with 1 <= T <= 1 << 20; copied into the
 *                      plan (stream-ordered), so the caller's buffers may change after the call
 *   plan (out)         the plan; device memory of about the pool's plan scratch for T tokens
 *                      and n_slots projections, plus T + n_seg + 1 ints and max_adapters floats
 *   errors             SLORA_ERR_INVALID_ARG for a null pool, out, token map or (n_seg > 0)
 *                      segment pointer, or sizes out of range; SLORA_ERR_CUDA when the
 *                      allocation or a launch fails (nothing is left allocated then)
 *
 * slora_plan_apply(plan, n, projs, x, y, stream): n must equal the plan's n_slots; projs,
 * x and y as for slora_lora_apply_multi (x, y of this layer).  The plan describes the pool
 * as it was when the plan was made: after any load or eviction in the pool (including those
 * of slora_adapters_acquire) every apply of an older plan returns SLORA_ERR_INVALID_ARG and
 * launches nothing.  Applies of one plan must not overlap in time (they share its counter
 * and partial sums): issue them on one stream, or order the streams.
 *
 * slora_plan_remake(plan, token_adapter_idx, seg_indptr, scaling, stream) plans the next
 * iteration's batch into the same plan: the same T, n_seg and n_slots as at creation, any
 * token map, segments and scaling (NULL: the registered values), and the pool as it is now.
 * It allocates nothing.  Enqueue it after the applies of the previous batch (same stream, or
 * ordered streams).
 *
 * slora_plan_destroy waits for the device and frees the plan; NULL is a no-op.  Destroy a
 * pool's plans before the pool.
 * ------------------------------------------------------------------------- */
typedef struct slora_plan *slora_plan_t;
slora_status slora_plan_create(slora_pool_t pool, int32_t n_slots, int32_t T, const int32_t *token_adapter_idx,
                               const int32_t *seg_indptr, int32_t n_seg, const float *scaling,
                               slora_stream_t stream, slora_plan_t *plan);
slora_status slora_plan_apply(slora_plan_t plan, int32_t n, const int32_t *projs /*host*/,
                              const void *const *x /*host array*/, void *const *y /*host array*/,
                              slora_stream_t stream);
slora_status slora_plan_remake(slora_plan_t plan, const int32_t *token_adapter_idx, const int32_t *seg_indptr,
                               const float *scaling, slora_stream_t stream);
slora_status slora_plan_destroy(slora_plan_t plan);

/* ---------------------------------------------------------------------------
 * slora_lora_apply_bmm: the padded batched-GEMM path, kept as the comparison the S-LoRA
 * ablation calls the slower BMM path (explainer, "Results and evidence", Figure 5 narrative;
 * explainer, "Prior limits").
 * Not the hot path: it exists to be measured against slora_lora_apply.  Decode tokens
 * only (no segments): every token gets a dense copy of its adapter's factors zero-padded
 * to R = the pool's largest registered rank rounded up to a multiple of 8 (a gather
 * kernel writes A^T and s * B into the workspace), then two strided batched GEMMs of the
 * cuBLAS library (loaded on first use; SLORA_ERR_UNSUPPORTED if it cannot be) form
 * u_t = fp16(A_t^T x_t) and y_t = y0_t + (s B_t)^T u_t with fp32 accumulation.
 *   proj, x, y, T, token_adapter_idx, scaling, stream: as slora_lora_apply (n_seg = 0)
 *   workspace  device buffer, 16-byte aligned, of at least slora_bmm_workspace_bytes()
 *              bytes (T * R * (4 * hidden + 2), rounded up); owned by the caller
 * Tokens without a resident adapter keep y and set a device status code.
 * ------------------------------------------------------------------------- */
slora_status slora_bmm_workspace_bytes(slora_pool_t pool, int32_t T, size_t *out);
slora_status slora_lora_apply_bmm(slora_pool_t pool, int32_t proj, const void *x, void *y, int32_t T,
                                  const int32_t *token_adapter_idx, const float *scaling,
                                  void *workspace, size_t workspace_bytes, slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * slora_lora_apply_noalloc: the same computation as slora_lora_apply, with the same
 * arguments, for callers that must not allocate device memory during the call.  The
 * S-LoRA pages have no counterpart for it; it exists for callers whose device memory
 * is owned and accounted by a host framework's allocator, or whose serving step cannot
 * absorb a cudaMalloc / cudaFree and the device synchronisation around it (the pool's
 * own plan scratch is allocated on first use and re-allocated when a larger batch or a
 * larger registered rank arrives).
 *
 * Scratch: one fixed 16 MiB device array inside the library, which every GPU that loads
 * the library holds until the process exits.  The call allocates and frees nothing.
 * Limit: one plan's scratch must fit that array; a plan of T' tokens needs about
 *   T' * (116 + NB * (8 * (nch + 1) + 512 * nch)) + 1280 bytes
 * (per token: its slot in the token order and at most one 112-byte work group; per hidden
 * block: the 8-byte work-list entries and the 64 eight-byte tagged partial sums of every
 * 64-row rank chunk), with NB = ceil(hidden / 1024) and nch = ceil(largest registered
 * rank / 64).  A batch runs as one plan when it fits (T' = min(T, 16384) when
 * max_adapters <= 2048, else 2048), otherwise as several plans of half, a quarter, ... of
 * that many tokens, the largest that fits (every token's result is the same whatever plan
 * it is in).  With ranks up to 64 one plan holds about 7,500 tokens at hidden 4096 and
 * 6,000 at hidden 5120.  Only when a plan of 64 tokens does not fit does the call return
 * SLORA_ERR_UNSUPPORTED (with the sizes in slora_last_error()) and launch nothing.
 * The first call on a device looks up the array's device address (once per device,
 * with that device current); make that first call before any stream capture.
 * Every call on a device shares the one array and leaves its plan and partial sums
 * there; the plan kernel rewrites every plan field the delta kernel reads (counters set
 * to zero), and every partial sum carries the tag of the launch that wrote it (a new tag
 * per launch), so stale sums are never taken for new ones.  The first launch on a device,
 * and the launch after the tag sequence wraps, clear the partial region first with
 * cudaMemsetAsync on the call's stream.  Calls whose kernels overlap on the
 * GPU (other streams, other pools, other threads) race on the array: order them on one
 * stream or synchronise between them.
 * ------------------------------------------------------------------------- */
slora_status slora_lora_apply_noalloc(slora_pool_t pool, int32_t proj, const void *x, void *y,
                                      int32_t T, const int32_t *token_adapter_idx,
                                      const int32_t *seg_indptr, int32_t n_seg,
                                      const float *scaling, slora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Observability / test hooks.
 * adapter_pages(): the adapter's page table for projection proj, 2 * rank int32 entries
 *   (A^T rows then B rows) written to out (host).
 * adapter_rank(): registered rank.
 * page_read(): synchronously copies one page (hidden fp16) to host_out.
 * get_device_status(): synchronises the pool's device, returns the device status word
 *   (SLORA_DEV_*) and resets it to 0.
 * ------------------------------------------------------------------------- */
slora_status slora_adapter_pages(slora_pool_t pool, int32_t adapter_id, int32_t proj,
                                 int32_t *out);
slora_status slora_adapter_rank(slora_pool_t pool, int32_t adapter_id, int32_t *out);
slora_status slora_page_read(slora_pool_t pool, int32_t page, uint16_t *host_out);
slora_status slora_get_device_status(slora_pool_t pool, int32_t *status);
/* Number of kernels this pool has launched so far (scatter, directory, plan and delta
 * kernels), counted on the host at each launch. */
slora_status slora_pool_launch_count(slora_pool_t pool, int64_t *out);
/* Measurement hook.  event: a cudaEvent_t created by the caller on the pool's device, or
 * NULL to clear.  While set, every slora_lora_apply call of the pool records it on the
 * call's stream between the token plan and the first delta kernel, so the caller can time
 * the delta kernels alone.  The record breaks the launch overlap of the plan and the
 * delta, so a timing loop that wants the overlapped step leaves it unset.  The pool does
 * not take ownership; clear it before destroying the event.  The S-LoRA pages have no
 * counterpart for it. */
slora_status slora_pool_set_stage_event(slora_pool_t pool, void *event);
/* Test hook.  Forces the number of CTAs per thread-block cluster of the prefill
 * (segment) kernel for every later call in the process: 1, 2, 4 or 8, or 0 to let each
 * call choose from its batch size (the default).  The result does not depend on it up to
 * the summation order of the cluster's partial products.  A cluster size whose hidden
 * slices would leave a CTA without columns makes slora_lora_apply fail with
 * SLORA_ERR_CUDA.  Other values return SLORA_ERR_INVALID_ARG.  The S-LoRA pages have no
 * counterpart for it. */
slora_status slora_debug_set_prefill_cluster(int32_t ctas);
/* Test hook.  1 (the default): in a batch of at most 32 segments, the 128-token units of
 * the prefill kernel's last, partial round of units (all of them when there is a single
 * round) run split into 2 or 4 parts, the most that fit the clusters that round would leave
 * idle; each part runs on its own cluster, repeats the unit's shrink and forms its share
 * of the unit's y columns, so the result is bit for bit that of the unsplit unit.  0: no
 * unit is split.  Applies to every later call in the process; other values return
 * SLORA_ERR_INVALID_ARG.  The S-LoRA pages have no counterpart for it. */
slora_status slora_debug_set_prefill_split(int32_t on);
/* Test hook: host-side fault injection in the adapter load path.  The nth later operation
 * of `kind` (counted over every pool of the process) fails as if its call had failed:
 *   SLORA_FAULT_COPY       a cudaMemcpyAsync into the staging ring (copy-engine mode)
 *   SLORA_FAULT_SCATTER    a load-kernel launch
 *   SLORA_FAULT_DIRECTORY  a directory-update launch
 *   SLORA_FAULT_STAGING    the staging ring's growth allocation (copy-engine mode)
 *   SLORA_FAULT_ARENA      a page-table arena allocation (as if the arena were fragmented)
 * The load then returns SLORA_ERR_CUDA (SLORA_ERR_POOL_FULL for the arena) and takes
 * itself back: the work its side stream already has completes, the directory entries of
 * its adapters are cleared, their pages and arena ranges return to the free lists, and
 * none of them is resident; a later load of the same adapters runs normally.  Nothing is
 * made to fail on the GPU.  kind SLORA_FAULT_NONE or nth 0 clears a pending injection;
 * other values return SLORA_ERR_INVALID_ARG.  The S-LoRA pages have no counterpart for it. */
enum { SLORA_FAULT_NONE = 0, SLORA_FAULT_COPY = 1, SLORA_FAULT_SCATTER = 2, SLORA_FAULT_DIRECTORY = 3,
       SLORA_FAULT_STAGING = 4, SLORA_FAULT_ARENA = 5 };
slora_status slora_debug_inject_load_fault(int32_t kind, int32_t nth);

#ifdef __cplusplus
}
#endif

#endif /* SLORA_H */
