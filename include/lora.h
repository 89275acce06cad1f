/*
 * lora.h -- C ABI of the GB300 (sm_103a) multi-LoRA segmented linear.
 *
 * The library computes, for a batch of n tokens that each name one adapter slot,
 *
 *     y[t,:] = x[t,:] W^T + (alpha_s / r_s) (x[t,:] A_s^T) B_s^T,   s = idx[t],
 *
 * with no LoRA term when idx[t] == -1, over a pool of adapters that lives in device
 * memory with every rank zero-padded to a common r_max.
 *
 * Sources (web pages on multi-LoRA serving):
 *  - "LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排" (blog.lonae.com):
 *      the adapter execution unit (LoRA A/B applied onto the base hidden state, as a
 *      fused kernel or as a separate residual kernel); the two-level bucketing of a
 *      batch (request level, then adapter level); zero-padding low-rank adapters to
 *      the high rank; the adapter storage pool with hot adapters resident in HBM.
 *  - "Multi-LoRA 在线服务隔离：适配器身份、显存配额与跨租户防串用" (ai.codenodex.com),
 *      section "请求身份决定适配器，而非客户端参数": a mixed-adapter batch keeps a
 *      per-request index map; authorisation is default-deny and a missing mapping is
 *      an explicit error, never a fallback to another adapter.
 *  - xpshop.cn article 492 (on-prem multi-LoRA case study), section 三: over-quota
 *      mounts are refused, base/adapter mismatches are refused at mount time, routing
 *      default "base_only", routing resolved once at request entry.
 *
 * Conventions shared by every entry point:
 *  - Ownership: the caller owns every buffer.  The library never allocates device
 *    memory; pools and workspaces are carved out of caller memory.  Handles
 *    (lora_pool_t) are small host structs owned by the library.
 *  - Pointers named *_dev are device pointers; everything else is host memory.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call that touches the device only enqueues work on that stream
 *    and returns without synchronising, except lora_segment_status.
 *  - Layouts are row-major and densely packed: x [n, h_in], W [h_out, h_in] (the
 *    nn.Linear layout), y [n, h_out], adapter A [rank, h_in], adapter B [h_out, rank].
 *    x, W, y, A and B share the pool's dtype.
 *  - Errors: a negative lora_status; lora_last_error() returns a message for the
 *    calling thread.  Argument errors are detected on the host before anything is
 *    enqueued.  Data-dependent errors (an idx out of range or naming an empty slot)
 *    are detected on the device: the segment builder sets its status word to
 *    LORA_EIDX and lora_linear_fwd then leaves y unwritten -- there is no fallback
 *    to base-only output or to another adapter.
 *  - Thread safety: calls on different pools are independent; calls on one pool must
 *    not run concurrently from several host threads.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_F32 = 0,  /* float32: CUDA-core path */
    LORA_F16 = 1,  /* IEEE half: tcgen05 tensor-core path, fp32 accumulation */
    LORA_BF16 = 2  /* bfloat16: tcgen05 tensor-core path, fp32 accumulation */
} lora_dtype;

typedef enum {
    LORA_OK = 0,
    LORA_EINVAL = -1,   /* bad argument (null pointer, bad size, bad dtype, misalignment) */
    LORA_ESLOT = -2,    /* slot index out of range */
    LORA_EBUSY = -3,    /* slot already holds an adapter */
    LORA_ERANK = -4,    /* rank < 1 or rank > r_max */
    LORA_ENOSPACE = -5, /* caller buffer or workspace too small */
    LORA_EIDX = -6,     /* (device) idx outside [-1, n_slots) or naming an empty slot */
    LORA_ECUDA = -7,    /* a CUDA runtime call failed */
    LORA_EUNSUP = -8,   /* shape/dtype combination the library does not support */
    LORA_ETIMEOUT = -9  /* (device) a pipeline wait exceeded its time limit; output invalid */
} lora_status;

typedef enum {
    LORA_VARIANT_AUTO = 0,     /* the library's measured policy picks */
    LORA_VARIANT_FUSED = 1,    /* expand fused into the base GEMM epilogue */
    LORA_VARIANT_SEPARATE = 2, /* base GEMM, then a separate residual expand kernel */
    LORA_VARIANT_CUDA_CORE = 3 /* diagnostic: CUDA-core base GEMM with fused expand, no tensor cores */
} lora_variant;

/* Shape of one pool.  One pool serves one linear layer (one base weight W). */
typedef struct {
    int32_t h_in;     /* input features  (>= 1; multiple of 8 for 16-bit dtypes) */
    int32_t h_out;    /* output features (>= 1; multiple of 8 for 16-bit dtypes) */
    int32_t r_max;    /* padded rank, 1..256 (multiple of 8 for 16-bit dtypes) */
    int32_t n_slots;  /* adapter slots, 1..2048 */
    int32_t dtype;    /* lora_dtype */
} lora_pool_desc;

typedef struct lora_pool* lora_pool_t;

/* Output of lora_segment: device pointers into the caller's segment workspace.
 * Sorted order = stable sort of token positions by idx, with -1 as the smallest key.
 *   perm_dev[j]       original position of the j-th token in sorted order     [n]
 *   seg_start_dev[i]  first sorted position of segment i; seg_start[nseg] = n  [n_slots+2]
 *   seg_slot_dev[i]   slot of segment i (-1 for the base-only run)            [n_slots+1]
 *   nseg_dev          number of segments, the number of shrink items, then two
 *                     words the decode kernels use internally                [4]
 *   status_dev        LORA_OK or LORA_EIDX                                    [1]
 *   idx_dev           copy of the batch's idx (original order)               [n]
 *   items_dev         shrink work items: every adapter segment cut into runs of up to 4
 *                     sorted tokens, {slot, count, token[4], rank, 0} each   [n][8]
 *                     (rank: the slot's rank in the pool the segments were built on, a
 *                     hint -- kernels of another pool check their own slot table) 
 * Segments are rebuilt once per batch and reused by every linear layer that runs
 * over that batch, as long as the workspace stays alive and unmodified.  The linears that
 * use one segment table run on one stream, one after another (a decode shrink kernel tells
 * the fused GEMM after it through the two words above when x may be read). */
typedef struct {
    int32_t* perm_dev;
    int32_t* seg_start_dev;
    int32_t* seg_slot_dev;
    int32_t* nseg_dev;
    int32_t* status_dev;
    int32_t* idx_dev;
    int32_t* items_dev;
    int32_t n_tokens;
    int32_t n_slots;
} lora_segments;

/* ---- adapter pool (device-resident slot table + zero-padded A/B slabs) ---------------
 * Layout inside the caller's buffer (all offsets 256-byte aligned):
 *   slot table  n_slots x {int32 rank, int32 state, float scale, int32 reserved}
 *   A slab      [n_slots, r_max, h_in]   rows >= rank are zero
 *   B slab      [n_slots, h_out, r_max]  columns >= rank are zero
 * scale = alpha / rank with the adapter's true rank. */

/* Bytes a pool with this shape needs.  LORA_EINVAL on a bad shape. */
int lora_pool_bytes(const lora_pool_desc* desc, size_t* bytes);

/* Create a pool inside dev_mem (device, >= lora_pool_bytes, 256-byte aligned).
 * Enqueues one memset on `stream` that empties every slot and zeroes both slabs.
 * The handle is valid until lora_pool_destroy; dev_mem must outlive it. */
int lora_pool_create(const lora_pool_desc* desc, void* dev_mem, size_t bytes, void* stream,
                     lora_pool_t* out);

/* Free the host handle.  The caller's device memory is not touched. */
int lora_pool_destroy(lora_pool_t pool);

/* Mount an adapter into an empty slot: copy A_dev [rank, h_in] and B_dev [h_out, rank]
 * (pool dtype, row-major) into the slot with zero padding up to r_max and mark it ready
 * with scale alpha/rank.  One kernel, stream-ordered.  A_dev / B_dev may be device memory
 * or host memory the device can read (pinned host memory under unified addressing; on
 * GB300 the kernel then reads it over NVLink-C2C, so mounting from host needs no staging
 * copy); they must stay valid until the kernel has run.  Errors: LORA_ESLOT (slot out of
 * range), LORA_ERANK (rank < 1 or > r_max), LORA_EBUSY (slot already mounted: hot swap
 * must unmount first), LORA_EINVAL (null pointers), LORA_ECUDA (launch failed). */
int lora_pool_load_slot(lora_pool_t pool, int slot, const void* A_dev, const void* B_dev, int rank,
                        float alpha, void* stream);

/* Mount `count` adapters in one go: entry i is (slots[i], A[i], B[i], ranks[i], alphas[i])
 * with the meaning of lora_pool_load_slot (the arrays are host memory; A[i] / B[i] device
 * or device-readable host memory).  Every entry is validated before anything is enqueued
 * (errors as lora_pool_load_slot; a slot named twice is LORA_EBUSY).  16-bit pools with
 * 16-byte aligned sources mount up to 32 slots per kernel with 16-byte copies. */
int lora_pool_load_slots(lora_pool_t pool, int count, const int* slots, const void* const* A, const void* const* B,
                         const int* ranks, const float* alphas, void* stream);

/* Mark a slot empty again (stream-ordered).  Work already enqueued on the same stream that
 * reads the slot is unaffected (stream order drains it); batches segmented afterwards that
 * name it fail with LORA_EIDX.  Work on other streams that may still read the slot must be
 * ordered before a later lora_pool_load_slot into it (an event), since that overwrites the
 * slot's rows in the order of its own stream. */
int lora_pool_unload_slot(lora_pool_t pool, int slot, void* stream);

/* ---- segment builder ------------------------------------------------------------------ */

/* Workspace bytes lora_segment needs for n_tokens tokens over n_slots slots. */
int lora_segment_workspace_bytes(int n_tokens, int n_slots, size_t* bytes);

/* Validate idx_dev [n_tokens] (device int32) against the pool's slot table and build
 * the stable segments into ws_dev (device, >= lora_segment_workspace_bytes, 256-byte
 * aligned).  One kernel, no host synchronisation.  n_tokens may be 0.  If any idx is
 * out of range or names an empty slot, *status_dev = LORA_EIDX and nseg = 0. */
int lora_segment(const int32_t* idx_dev, int n_tokens, lora_pool_t pool, void* ws_dev, size_t ws_bytes,
                 lora_segments* out, void* stream);

/* Synchronise `stream` and read the device status word (debug/test helper). */
int lora_segment_status(const lora_segments* seg, void* stream, int* status);

/* ---- LoRA-augmented linear --------------------------------------------------------------- */

/* Workspace bytes lora_linear_fwd needs for n_tokens tokens on this pool. */
int lora_linear_workspace_bytes(lora_pool_t pool, int n_tokens, size_t* bytes);

/* y_dev = x_dev W_dev^T + per-token LoRA term (see top of file).
 *   W_dev [h_out, h_in], x_dev [n, h_in], y_dev [n, h_out]: device, pool dtype, 16-byte
 *   aligned for 16-bit dtypes; n = seg->n_tokens; seg from lora_segment on this pool's
 *   slot count; variant a lora_variant; ws_dev device workspace of
 *   >= lora_linear_workspace_bytes, 256-byte aligned (it receives the shrink output
 *   s = (alpha/r) x A^T, float32 [n, r_max]; successive calls on one stream may share it).
 * If seg's status word is not LORA_OK the kernels leave y untouched. */
int lora_linear_fwd(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev,
                    const lora_segments* seg, int variant, void* ws_dev, size_t ws_bytes, void* stream);

/* lora_linear_fwd plus an L2 prefetch hint (GB300 has a 129 MB L2, larger than one base
 * weight).  prefetch_dev / prefetch_bytes: an optional device range, 16-byte aligned --
 * typically the base weight of the next linear the caller will run on this stream.  Once a
 * decode-path CTA (n <= 256 tokens) has issued its own loads, it streams its share of that
 * range into L2 while its epilogue runs, so the next linear finds most of its weight in L2.
 * Purely a hint: results are identical with or without it; the range is only read.  NULL
 * (or 0 bytes) means no prefetch, which is exactly lora_linear_fwd.  Measured on GB300 with
 * chained 4096 x 4096 decode linears it costs 7-8 % (the prefetch competes with the next
 * linear's own weight stream), so it suits callers whose next weight would otherwise start
 * cold after a long gap. */
int lora_linear_fwd_ex(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev,
                       const lora_segments* seg, int variant, void* ws_dev, size_t ws_bytes,
                       const void* prefetch_dev, size_t prefetch_bytes, void* stream);

/* lora_linear_fwd without a caller workspace.  The multi-LoRA pages have no counterpart to
 * this entry point: it is a convenience of this library for callers that cannot allocate
 * device memory when they call in -- for example an operator plugin inside another engine,
 * which is handed only its inputs and outputs while the engine owns every allocation, or a
 * host held to a fixed device-memory budget that it may not grow.
 * Arguments and results are those of lora_linear_fwd; the shrink output goes to a fixed
 * 4 MiB device array owned by the library (a static device array: every GPU that loads the
 * library holds it until the process exits).  A call needs 4 * n * r_max * p bytes of it, with
 * p = min(ceil(h_in / 1024), 4, max(1, 256 / n)) for 16-bit batches of up to 256 tokens and
 * p = 1 otherwise; larger calls fail with LORA_ENOSPACE and enqueue nothing.  This function
 * calls no cudaMalloc, cudaFree or allocating library routine.  The pool's device must be the
 * current device (LORA_EINVAL otherwise).  Its first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  Every call shares the array, which keeps the last call's contents (a
 * call reads only values it wrote itself, so nothing has to start at zero); calls that can
 * overlap on the GPU (several streams, concurrent graph replays) race with each other. */
int lora_linear_fwd_static_ws(lora_pool_t pool, const void* W_dev, const void* x_dev, void* y_dev,
                              const lora_segments* seg, int variant, void* stream);

/* Which variant LORA_VARIANT_AUTO picks for n_tokens on this pool (1 or 2): fused, except for
 * decode batches (<= 256 tokens) whose fused GEMM could not hold every adapter a CTA needs in
 * shared memory during its main loop (more than 32 tokens per CTA, or more distinct adapters
 * than it can stage); those run the base GEMM and the segmented expand.  Chosen from GB300
 * measurements; host-only, no device access. */
int lora_linear_policy(lora_pool_t pool, int n_tokens, int* variant);

/* ---- grouped projections ---------------------------------------------------------------
 *
 * One adapter usually targets several projections of a layer (the registry entry of the
 * ai.codenodex.com page, section "适配器先进入可信注册表", lists target modules q_proj and
 * v_proj), and the projections of an attention block (q, k, v) or of an MLP (gate, up)
 * read the same x and route every token to the same adapter.  A group runs such
 * projections as one linear over their row-concatenated base weight, sharing one
 * segment table, one pass over x for the shrink and one launch per kernel:
 *
 *     y[:, col_q : col_q + h_out_q] = x W_q^T + (alpha_s / r_s) (x A_{q,s}^T) B_{q,s}^T
 *
 * for slice q = 0..count-1, with col_q = h_out_0 + ... + h_out_{q-1}.
 *   count   1..4 slices; pools[q] is slice q's adapter pool.  Every pool has the same h_in,
 *           r_max, n_slots and dtype (fp16 or bf16; otherwise LORA_EUNSUP), and the same
 *           slots mounted (LORA_EINVAL otherwise; checked against the host-side record of
 *           mounts, so each slot's adapter is mounted into every pool of the group).
 *           With count > 1 every h_out_q is a multiple of 16.
 *   W_dev   [sum h_out_q, h_in]: the slices' base weights stacked row-wise (slice 0 first).
 *   x_dev   [n, h_in];  y_dev [n, sum h_out_q]: slice q's output is its column range.
 *           W, x, y 16-byte aligned, n = seg->n_tokens, seg from lora_segment on pools[0].
 *   ws_dev  >= lora_linear_group_workspace_bytes, 256-byte aligned.
 *   variant LORA_VARIANT_AUTO (lora_linear_group_policy), FUSED or SEPARATE; the CUDA-core
 *           diagnostic variant is LORA_EUNSUP.
 * Errors and the device status word behave as in lora_linear_fwd (y untouched when the
 * segments carry an error).  A group of one is the same computation as lora_linear_fwd. */
int lora_linear_group_workspace_bytes(int count, const lora_pool_t* pools, int n_tokens, size_t* bytes);
int lora_linear_fwd_group(int count, const lora_pool_t* pools, const void* W_dev, const void* x_dev, void* y_dev,
                          const lora_segments* seg, int variant, void* ws_dev, size_t ws_bytes, void* stream);
/* Which variant AUTO picks for a group (1 or 2): for one slice, lora_linear_policy's choice;
 * otherwise separate -- one base GEMM over the concatenated weight, then one segmented expand
 * over every slice -- for batches of up to 256 tokens, fused above.  Measured on GB300;
 * host-only. */
int lora_linear_group_policy(int count, const lora_pool_t* pools, int n_tokens, int* variant);

/* ---- host-tier adapter cache -------------------------------------------------------------
 *
 * The blog.lonae.com page describes a tiered adapter store: hot adapters resident in GPU
 * memory, warm ones in host memory, loaded on demand, unreferenced ones evicted.  A cache
 * manages the slots of `count` pools with the same n_slots (typically every LoRA-augmented
 * projection of a model) and keeps slot s of every pool holding the same adapter, so one
 * segment table serves all of them.
 *   lora_cache_create: the pools must hold no adapters (LORA_EBUSY otherwise); from then on
 *     the cache owns their slots -- mounting or unmounting them directly breaks it.  The
 *     pools must outlive the cache.
 *   lora_cache_register: adapter `id` (>= 0) with, for pool p, A_host[p] [ranks[p], h_in_p]
 *     and B_host[p] [h_out_p, ranks[p]] in the pool's dtype, in page-locked host memory (read
 *     by the mount kernel over NVLink-C2C / PCIe; pageable memory is not accessible to it)
 *     that the caller keeps valid until the adapter is unregistered.  LORA_EBUSY for a known
 *     id, LORA_ERANK for a rank outside [1, r_max].  Nothing is copied yet.
 *   lora_cache_map: for a batch of n tokens naming adapter ids (-1 = base only), makes every
 *     named adapter resident and writes idx_out[t] (host int32: its slot, or -1), the input
 *     of lora_segment.  A resident adapter is a hit; a missing one goes to a free slot, else
 *     to the least recently used slot that this batch does not name (ties: lowest slot),
 *     whose adapter is unmounted.  Mounts (one batched mount per pool) and unmounts are
 *     enqueued on `stream`, so kernels enqueued later on that stream see them, and kernels
 *     enqueued earlier still read the evicted adapter; work on other streams must be ordered
 *     by the caller.  *mounts_out (may be NULL) = adapters mounted by this call.
 *     An unregistered id is LORA_EIDX and more distinct ids than slots is LORA_ENOSPACE;
 *     either way nothing changes and idx_out is not written.  If a mount or unmount fails to
 *     enqueue (LORA_ECUDA), the cache's record may no longer match the pools: destroy the
 *     cache and its pools' contents (recreate the pools) before further use.
 *   lora_cache_unregister: forgets the adapter, unmounting it (on `stream`) if resident.
 *   lora_cache_slot_of: the slot holding adapter id, or -1 if it is not resident.
 *   lora_cache_stats: hits and misses (per distinct adapter per map call), evictions. */
typedef struct lora_cache* lora_cache_t;
int lora_cache_create(int count, const lora_pool_t* pools, lora_cache_t* out);
int lora_cache_destroy(lora_cache_t cache);
int lora_cache_register(lora_cache_t cache, int64_t id, const void* const* A_host, const void* const* B_host,
                        const int* ranks, const float* alphas);
int lora_cache_unregister(lora_cache_t cache, int64_t id, void* stream);
int lora_cache_map(lora_cache_t cache, const int64_t* ids, int n, int32_t* idx_out, int* mounts_out, void* stream);
int lora_cache_slot_of(lora_cache_t cache, int64_t id, int* slot);
int lora_cache_stats(lora_cache_t cache, uint64_t* hits, uint64_t* misses, uint64_t* evictions);

/* Diagnostic of the failure path (the pages have no counterpart).  Every pipeline wait of
 * the tensor-core kernels is bounded: when one runs past its limit the kernel records
 * LORA_ETIMEOUT in the status word, writes none of its output and returns (no trap, no
 * endless spin).  This call runs that same bounded wait in one small kernel on `stream`:
 * the kernel waits on a barrier that completes only if `arrive` is non-zero, for at most
 * limit_ns nanoseconds (<= 100 ms, LORA_EINVAL above).  If the wait gives up, *status_dev
 * (device int32) becomes LORA_ETIMEOUT and out_dev is not written; otherwise out_dev[0..n)
 * (device float32, n <= 2^20) is set to 1.0 and *status_dev is left as it was. */
int lora_wait_selftest(int32_t* status_dev, float* out_dev, int n, int arrive, uint64_t limit_ns, void* stream);

/* ---- adapter loader: background mounts on a copy stream, draining remounts -------------
 *
 * The blog.lonae.com page's adapter loader fills the execution unit's buffers without
 * blocking inference: asynchronous double buffering -- one copy serves the running requests
 * while the next candidate adapter is fetched in the background from pinned host memory.  The
 * xpshop.cn article 492 (section 三) unloads adapters in "draining" mode: requests already
 * running on an adapter finish before it goes.  A loader manages `count` pools with the same
 * n_slots (the projections an adapter targets; slot s of every pool holds the same adapter)
 * and a copy stream owned by the caller.  Ordering is by CUDA events, with no host
 * synchronisation:
 *   lora_loader_mount: enqueue, on the copy stream, mounts of adapters into `count` distinct
 *     slots.  Entry (p, i) = A[p*count + i], B[p*count + i], ranks[...], alphas[...] is slot
 *     slots[i]'s adapter for pool p, with the meaning of lora_pool_load_slots (A/B in pinned
 *     host memory, read by the mount kernel; kept valid by the caller until the copy stream
 *     has passed the mount).  A slot that holds an adapter is drained first: the copy stream
 *     waits for every fence lora_loader_release recorded on it since its last mount, then the
 *     slot is unmounted and remounted.  Everything is validated before anything is enqueued
 *     (LORA_ESLOT, LORA_ERANK, LORA_EBUSY for a slot named twice, LORA_EINVAL).
 *   lora_loader_acquire: make `stream` wait until the latest mount of each named slot has
 *     landed (call it before segmenting a batch that names a freshly mounted slot).
 *   lora_loader_release: record on `stream` a fence after the work enqueued so far, which may
 *     read the named slots; a later remount of any of them waits for it.  Release every slot
 *     a batch names after that batch's linears.
 *   lora_loader_stats: slots mounted so far, fences drained by remounts.
 * The loader's pools must be mounted and unmounted only through it, and must outlive it.
 * Not thread-safe. */
typedef struct lora_loader* lora_loader_t;
int lora_loader_create(int count, const lora_pool_t* pools, void* copy_stream, lora_loader_t* out);
int lora_loader_destroy(lora_loader_t loader);
int lora_loader_mount(lora_loader_t loader, int count, const int* slots, const void* const* A, const void* const* B,
                      const int* ranks, const float* alphas);
int lora_loader_acquire(lora_loader_t loader, int count, const int* slots, void* stream);
int lora_loader_release(lora_loader_t loader, int count, const int* slots, void* stream);
int lora_loader_stats(lora_loader_t loader, uint64_t* mounts, uint64_t* drained_fences);

/* Message of the last failed call on this host thread ("" if none). */
const char* lora_last_error(void);

/* Number of kernels this library has launched in this process (instrumentation). */
uint64_t lora_kernel_launch_count(void);

/* Timing instrumentation for benchmarks: while set (non-NULL cudaEvent_t handles passed as
 * void*), every lora_linear_fwd records before_shrink on its stream before the shrink
 * kernel, before_gemm between the shrink and the base-GEMM kernel, and after_gemm after the
 * base-GEMM kernel.  The records serialise those kernels (no launch overlap), so the
 * intervals are per-kernel durations.  Process-wide, not thread-safe; NULLs disable. */
int lora_set_timing_events(void* before_shrink, void* before_gemm, void* after_gemm);

/* In-step timing instrumentation for benchmarks: while set, every base-GEMM launch (decode,
 * prefill and tall-tile kernels) takes the next of `pairs` pairs of uint64 in stamps_dev
 * (device memory, 8-byte aligned; round robin in launch order, restarting at pair 0 on every
 * call of this function) and records into it the %globaltimer nanoseconds of its first CTA's
 * start (atomicMin into [0]) and of its last CTA's end (atomicMax into [1]); the caller sets
 * every pair to {UINT64_MAX, 0} before the launches it times.  Unlike lora_set_timing_events
 * this does not serialise neighbouring launches, so the intervals are the kernels' durations
 * inside a chain of programmatic dependent launches.  Process-wide, not thread-safe; NULL
 * disables.  LORA_EINVAL for pairs <= 0 with a buffer, or a misaligned buffer. */
int lora_set_kernel_stamps(void* stamps_dev, int pairs);

/* The same for the CUDA-core shrink and segmented-expand kernels of the decode path: while set,
 * each of their launches takes the next of `triples` triples of uint64 (round robin, restarting
 * at triple 0 on every call of this function) and records {first CTA start (atomicMin),
 * first return from its grid-dependency wait (atomicMin), last CTA end (atomicMax; thread 0's
 * exit)}; initialise triples to {UINT64_MAX, UINT64_MAX, 0}.  NULL disables. */
int lora_set_aux_stamps(void* stamps_dev, int triples);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */
