/*
 * lora.h -- C ABI of the GB300 multi-LoRA mixed-batch adapter library.
 *
 * The operation ("Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter
 * Hot-Swap & Memory", section "The kernel trick: gather, do not merge"): a
 * request i that names adapter a(i) needs
 *
 *     y_i = x_i W^T + scale_a * (x_i A_a^T) B_a^T
 *
 * The base product is one matmul shared by the whole batch; the adapter term
 * is a gather of small matmuls, "shrink" (x -> v, width r) then "expand"
 * (v -> y).  SGMV serves contiguous segments of tokens that share an adapter
 * (prefill), BGMV one adapter per token (decode).  Adapters of different
 * ranks live in one paged pool (S-LoRA slide 8: pages of H elements, R of them
 * for a rank-R adapter) and are gathered without padding to a common rank
 * (S-LoRA slide 10, MBGMM/MBGMV).
 *
 * Orientation used throughout.  For adapter a on one adapted matrix:
 *   A_T_a is rank x h_in; its row j is the j-th low-rank direction, so
 *         v[t][j] = sum_k x[t][k] * A_T_a[j][k];
 *   B_a   is rank x h_out, and y[t][n] += scale_a * sum_j v[t][j] * B_a[j][n].
 *   W     is h_out x h_in, row-major (row n = output feature n), like an
 *         nn.Linear weight; the base term is y[t][n] = sum_k x[t][k] W[n][k].
 *
 * Conventions shared by every call:
 *   - Element type: every x, y, W and page holds the pool's dtype (LORA_F32
 *     or LORA_BF16).  v is always fp32.  Arithmetic accumulates in fp32;
 *     bf16 results are rounded to nearest even on store.
 *   - Layout: x is T x h_in, y is T x h_out, v is T x ld_v, all row-major and
 *     dense (row stride = width).  Base pointers of x, y, v, W and the
 *     workspace must be 16-byte aligned (torch allocations are).
 *   - Pointers passed to compute calls are DEVICE pointers owned by the
 *     caller; the library keeps none of them after the call returns.
 *   - Streams: a lora_stream is a cudaStream_t (NULL = legacy default
 *     stream).  Compute calls only enqueue work on it and never synchronise.
 *   - Adapter ids: id < 0 means "no adapter" (the token keeps its base/y0
 *     value).  An id >= max_adapters, or of an adapter not loaded on that
 *     matrix, is a device-detected error: the token gets no adapter term and
 *     bit LORA_DEV_BAD_ADAPTER is set in the pool's device status word.
 *   - Segments: seg_starts has S+1 entries with seg_starts[0] == 0,
 *     non-decreasing, seg_starts[S] == T; segment s covers tokens
 *     seg_starts[s] .. seg_starts[s+1]-1 and uses adapter seg_adapter[s].
 *     Empty segments are legal.  The table lives on the device, so it is
 *     checked there: a violation sets LORA_DEV_BAD_SEGMENTS and the affected
 *     tokens are computed against a clamped segment index (no access leaves
 *     the arrays).
 *   - Host-detectable errors (NULL pointer, bad size, misalignment, unknown
 *     matrix, a pool of the wrong dtype) return a negative status before any
 *     work is enqueued.  No kernel traps, asserts or waits without a bound.
 *
 * Thread safety: a pool may be used from one host thread at a time.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_pool lora_pool;   /* opaque; owns pages, tables, status word */
typedef void *lora_stream;            /* a cudaStream_t */

/* Return codes. */
enum {
    LORA_OK = 0,
    LORA_ERR_ARG = -1,           /* bad argument (NULL, size, alignment, dtype) */
    LORA_ERR_POOL_FULL = -2,     /* not enough free pages for the load */
    LORA_ERR_RANK = -3,          /* rank < 0, rank > max_rank, or ld_v < max_rank */
    LORA_ERR_NOT_LOADED = -4,    /* unload of an entry that holds no adapter */
    LORA_ERR_CUDA = -5,          /* a CUDA runtime call failed (no device, OOM, ...) */
    LORA_ERR_DEVICE_INDEX = -6,  /* lora_get_error: the device status word was non-zero */
    LORA_ERR_SHAPE = -7          /* h_in/h_out disagree with the matrix or exceed the page */
};

/* Element types of the pool (and of x, y, W). */
enum { LORA_F32 = 0, LORA_BF16 = 1 };

/* Bits of the device status word (see lora_get_error). */
enum {
    LORA_DEV_BAD_ADAPTER = 1,    /* an id >= max_adapters, or an unloaded adapter */
    LORA_DEV_BAD_SEGMENTS = 2,   /* a segment table that breaks the rules above */
    LORA_DEV_WAIT_TIMEOUT = 4    /* a pipeline wait inside a kernel gave up */
};

/*
 * Create a paged adapter pool on the current CUDA device.
 *   dtype        LORA_F32 or LORA_BF16.
 *   page_elems   H, elements per page; a multiple of 8 and >= every h_in and
 *                h_out later loaded.  One page holds one row of A_T (h_in
 *                elements) or one row of B (h_out elements).
 *   n_pages      pages to allocate (device memory = n_pages*H*sizeof(dtype)).
 *   max_rank     largest rank any adapter may have (1..1024).
 *   n_matrices   number of adapted matrices (e.g. layers x projections).
 *   max_adapters adapter ids run 0 .. max_adapters-1.
 * A rank-r adapter on one matrix occupies exactly 2r pages (r for A_T, r for
 * B), wherever they are free: ranks are mixed without padding (S-LoRA
 * slides 8 and 10).  On success *out owns all device memory of the pool.
 * Errors: LORA_ERR_ARG, LORA_ERR_CUDA (nothing is left allocated).
 */
int lora_pool_create(lora_pool **out, int dtype, int page_elems, int n_pages,
                     int max_rank, int n_matrices, int max_adapters);

/* Free every device and host resource of the pool.  Synchronises the device
 * first.  NULL is accepted. */
int lora_pool_destroy(lora_pool *pool);

/*
 * Load adapter `adapter` on matrix `matrix`: rank, scale, and HOST arrays
 *   A_T  rank x h_in  (row-major, pool dtype),
 *   B    rank x h_out (row-major, pool dtype).
 * The first load on a matrix fixes that matrix's (h_in, h_out); later loads
 * must match (else LORA_ERR_SHAPE).  A previous adapter in the same entry is
 * replaced (the device is synchronised first).  The device copy and the table
 * update run on `stream` (after the work already queued there) and the call
 * returns once they are complete: the adapter is resident for every kernel
 * launched afterwards, on any stream, and the host arrays may be freed at once.
 * rank == 0 is legal (the adapter adds nothing).
 * Errors: LORA_ERR_ARG, LORA_ERR_RANK, LORA_ERR_SHAPE, LORA_ERR_POOL_FULL
 * (the pool is unchanged), LORA_ERR_CUDA.
 */
int lora_pool_load(lora_pool *pool, int adapter, int matrix, int rank, float scale,
                   int h_in, int h_out, const void *A_T, const void *B, lora_stream stream);

/* Return the entry's pages to the free list and mark it unloaded.
 * Synchronises the device first, so no queued kernel still reads the pages.
 * Errors: LORA_ERR_ARG, LORA_ERR_NOT_LOADED, LORA_ERR_CUDA. */
int lora_pool_unload(lora_pool *pool, int adapter, int matrix);

/*
 * Asynchronous upload (S-LoRA slide 9: the adapters that queued requests will
 * need are copied to the GPU while the current batch computes; "Multi-LoRA
 * Serving", section "Memory: slots, tiers and paging": a host-memory tier with
 * prefetch lets one GPU serve far more adapters than its slots hold).
 *
 * lora_pool_load_async takes the arguments of lora_pool_load and copies the
 * host arrays into a pinned staging slot of the pool (a CPU copy: A_T and B
 * may be freed when the call returns), then ENQUEUES on `stream` the copy to
 * the device, the scatter into the adapter's pages and the copy of its table
 * record, and returns without waiting for them.  The adapter is resident for
 * work enqueued on `stream` after the call, and for work on other streams
 * ordered after it (an event recorded on `stream` after the call).  Kernels
 * of this library launched on `stream` right after it read the new record
 * (the record copy is the last step and is not a kernel).
 * Replacing an adapter: every kernel that may still read the old one must be
 * ordered before the call (same stream, or an event); its pages return to the
 * free list only once `stream` has passed the table update.
 * The staging ring has a few slots; a call that finds its slot still in use
 * waits for that slot's earlier copies.  When the free list is short, pages
 * retired by earlier asynchronous calls are waited for (oldest first).
 * Errors: as lora_pool_load (the pool is unchanged on any error).
 */
int lora_pool_load_async(lora_pool *pool, int adapter, int matrix, int rank, float scale,
                         int h_in, int h_out, const void *A_T, const void *B, lora_stream stream);

/* Marks the entry unloaded by a copy enqueued on `stream` (no wait); its
 * pages return to the free list once `stream` has passed it.  Kernels that
 * may still read the entry must be ordered before the call.
 * Errors: LORA_ERR_ARG, LORA_ERR_NOT_LOADED, LORA_ERR_CUDA. */
int lora_pool_unload_async(lora_pool *pool, int adapter, int matrix, lora_stream stream);

/* One adapter of a prefetch list: lora_pool_load's arguments. */
typedef struct lora_adapter_src {
    int adapter, matrix, rank;
    float scale;
    int h_in, h_out;
    const void *A_T;   /* rank x h_in, host, pool dtype */
    const void *B;     /* rank x h_out, host, pool dtype */
} lora_adapter_src;

/* Prefetch: lora_pool_load_async for every entry of `list` whose (adapter,
 * matrix) is not resident yet (resident entries are left as they are), in
 * list order, on `stream`.  Returns the number of uploads enqueued (>= 0), or
 * the first error (entries before it stay enqueued). */
int lora_pool_prefetch(lora_pool *pool, const lora_adapter_src *list, int n, lora_stream stream);

/* Pages currently free (host bookkeeping; pages retired by asynchronous calls
 * count once the stream has passed them -- an event query, no wait). -1 on
 * NULL. */
int lora_pool_free_pages(const lora_pool *pool);

/*
 * SGMV shrink (prefill; MBGMM for mixed ranks):
 *   v[t][j] = sum_k x[t][k] * A_T_a[j][k],  j < rank_a,  a = adapter of t's segment.
 * x: T x h_in (pool dtype); v: T x ld_v fp32 with ld_v >= the pool's max_rank.
 * Only v[t][0..rank_a-1] of tokens with a valid adapter are written.
 * Errors: LORA_ERR_ARG, LORA_ERR_RANK (ld_v < max_rank), LORA_ERR_SHAPE.
 */
int lora_sgmv_shrink(lora_pool *pool, int matrix, const void *x, float *v, int ld_v,
                     const int *seg_starts, const int *seg_adapter, int S, int T,
                     lora_stream stream);

/*
 * SGMV expand:  y[t][n] += scale_a * sum_j v[t][j] * B_a[j][n]  (read-modify-write).
 * v as produced by lora_sgmv_shrink; y: T x h_out (pool dtype).
 * Errors as lora_sgmv_shrink.
 */
int lora_sgmv_expand(lora_pool *pool, int matrix, const float *v, int ld_v, void *y,
                     const int *seg_starts, const int *seg_adapter, int S, int T,
                     lora_stream stream);

/*
 * BGMV (decode; MBGMV for mixed ranks): shrink and expand fused, one adapter
 * id per token:  y[t][n] += scale_a * sum_j (sum_k x[t][k] A_T_a[j][k]) B_a[j][n].
 * x: T x h_in, y: T x h_out (read-modify-write), token_adapter: T device int32.
 * Errors: LORA_ERR_ARG, LORA_ERR_SHAPE.
 */
int lora_bgmv(lora_pool *pool, int matrix, const void *x, void *y,
              const int *token_adapter, int T, lora_stream stream);

/* Bytes of device workspace lora_layer_forward needs for T tokens on this
 * matrix (0 on a bad argument). */
size_t lora_layer_forward_workspace_size(const lora_pool *pool, int matrix, int S, int T);

/*
 * Adapted layer: the shared base product for the whole mixed batch plus each
 * token's own low-rank term (the base product is computed once for every
 * token, and each token then receives its own adapter's update, "Multi-LoRA
 * Serving", section "The kernel trick: gather, do not merge"):
 *   y[t][n] = sum_k x[t][k] * W[n][k] + scale_a * sum_j (sum_k x[t][k] A_T_a[j][k]) B_a[j][n]
 * y is OVERWRITTEN.  W: h_out x h_in (pool dtype).  Tokens without an
 * adapter (or with an invalid one) get the base term only.
 * workspace: device scratch of at least lora_layer_forward_workspace_size()
 * bytes, owned by the caller, contents undefined on entry and exit.
 * Streams: part of the call's work (planning the rows whose M-tile is not
 * fused into the GEMM, and their shrink) may run on an internal stream, one per host thread
 * and device, that the call forks from `stream` and joins back to it with
 * events; the call's work as a whole stays ordered after earlier work on
 * `stream` and before later work on it, and under stream capture the fork
 * and join become graph edges.  The internal stream and its events are
 * created by the first such call on a thread: make that call outside stream
 * capture.
 * Errors: LORA_ERR_ARG (includes ws_bytes too small), LORA_ERR_SHAPE.
 */
int lora_layer_forward(lora_pool *pool, int matrix, const void *x, const void *W, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T,
                       void *workspace, size_t ws_bytes, lora_stream stream);

/*
 * lora_layer_forward without caller-provided workspace, for callers that
 * cannot allocate device memory: a serving runtime whose device memory is
 * carved into a fixed arena at start-up, a decode loop that must not call
 * cudaMalloc/cudaFree (they synchronise the whole device), or a C plugin with
 * no allocator of its own.  The pages describe no such variant; it exists
 * for these callers only.
 *
 * Same operation, arguments and errors as lora_layer_forward, minus the
 * workspace.  The scratch comes from one static device array of
 * LORA_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library keeps until the process exits.  Requires
 * lora_layer_forward_workspace_size(pool, matrix, S, T) <=
 * LORA_NOALLOC_SCRATCH_BYTES (about T * max_rank * 4 bytes plus a small
 * per-token plan; else LORA_ERR_ARG) and the pool's device to be current
 * (else LORA_ERR_ARG).  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  All calls share the array:
 * calls whose work overlaps on the GPU race and must be serialised by the
 * caller.  Allocates nothing (no cudaMalloc/cudaFree or allocating library
 * routine).
 */
#define LORA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int lora_layer_forward_noalloc(lora_pool *pool, int matrix, const void *x, const void *W, void *y,
                               const int *seg_starts, const int *seg_adapter, int S, int T,
                               lora_stream stream);

/*
 * FP8 base ("Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap &
 * Memory", the failure assumptions and "Operating it": the base may run in
 * FP8 while adapters trained on a bf16 base keep working in bf16).
 *
 * lora_quantize_e4m3: per-row quantisation of x (T x h bf16, device, h a
 * multiple of 8) to e4m3 codes q (T x h bytes, device, 8-byte aligned) and
 * fp32 scales sx (T, device):
 *   a = max_k |x[t][k]|, sx[t] = a / 448 and r = 448 / a (two fp32
 *             divisions per row),
 *   q[t][k] = e4m3(x[t][k] * r)  (the product in fp32, then rounded to the
 *             nearest e4m3 value, ties to the even code, saturating at +-448;
 *             e4m3 = 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *             infinities);
 *   a row with a < 2^-120 (a row of zeros included) gets sx[t] = 1 and +0 codes.
 * Errors: LORA_ERR_ARG.
 */
int lora_quantize_e4m3(const void *x, int T, int h, void *q, float *sx, lora_stream stream);

/* Workspace lora_layer_forward_fp8 needs: lora_layer_forward's plus the
 * codes and scales of x (0 on a bad argument). */
size_t lora_layer_forward_fp8_workspace_size(const lora_pool *pool, int matrix, int S, int T);

/*
 * lora_layer_forward with an FP8 base product:
 *   y[t][n] = sx[t] * w_scale * sum_k q[t][k] * W8[n][k]
 *           + scale_a * sum_j (sum_k x[t][k] A_T_a[j][k]) B_a[j][n]
 * W8: h_out x h_in e4m3 codes (device, the base weight quantised by the
 * caller with the per-tensor scale w_scale > 0); x: bf16 as for
 * lora_layer_forward -- quantised here per row (lora_quantize_e4m3) for the
 * base product, used unquantised for the low-rank term.  The base product
 * runs on the tensor cores (kind::f8f6f4), so the pool must be bf16, h_in a
 * multiple of 128 and h_out a multiple of 32 (else LORA_ERR_SHAPE).  y is
 * overwritten.  Workspace, streams and errors as lora_layer_forward.
 */
int lora_layer_forward_fp8(lora_pool *pool, int matrix, const void *x, const void *W8, float w_scale, void *y,
                           const int *seg_starts, const int *seg_adapter, int S, int T,
                           void *workspace, size_t ws_bytes, lora_stream stream);

/*
 * Synchronise the device, read the pool's device status word into
 * *device_status (may be NULL), and clear it.  Returns LORA_OK when the word
 * was zero, LORA_ERR_DEVICE_INDEX when any LORA_DEV_* bit was set, or
 * LORA_ERR_CUDA when the device reported an error.
 */
int lora_get_error(lora_pool *pool, int *device_status);

/* Static English text for a return code. */
const char *lora_strerror(int status);

/* Kernels this library has launched since it was loaded (host-side count,
 * summed over all pools; launches replayed from a captured CUDA graph are
 * not counted again). */
unsigned long long lora_launch_count(void);

/*
 * Two-tier adapter residency cache (host code; no device access).
 *
 * "Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap & Memory",
 * section "Memory: slots, tiers and paging" and its adapter-cache simulation:
 * a few GPU slots (here: adapters resident in the paged pool), backed by a
 * larger host-RAM tier, backed by disk.  Each tier keeps its adapters in
 * least-recently-used order and evicts the least recently used one when a
 * new one would exceed its slot count.  A request first looks in the GPU
 * tier; only on a GPU miss is the host tier looked up (and reordered).  A
 * slot count of 0 keeps nothing.
 *
 * The cache decides residency only and moves no data: a caller maps a GPU
 * hit to "already in the pool", a host hit to an upload from pinned host
 * memory (lora_pool_load_async), a disk hit to a fetch plus that upload, and
 * the GPU tier's eviction to lora_pool_unload_async.
 */
typedef struct lora_tier_cache lora_tier_cache;
enum { LORA_TIER_GPU = 0, LORA_TIER_HOST = 1, LORA_TIER_DISK = 2 };

/* Adapter ids 0..n_keys-1; both tiers start empty.  Errors: LORA_ERR_ARG. */
int lora_tier_cache_create(lora_tier_cache **out, int n_keys, int gpu_slots, int host_slots);
int lora_tier_cache_destroy(lora_tier_cache *cache);   /* NULL accepted */

/* One request for `adapter`: returns the tier that served it (LORA_TIER_*),
 * or LORA_ERR_ARG for an id out of range.  *gpu_evicted (may be NULL) gets
 * the adapter the GPU tier dropped to make room, or -1. */
int lora_tier_cache_touch(lora_tier_cache *cache, int adapter, int *gpu_evicted);

/* Bit 0: the adapter is in the GPU tier; bit 1: in the host tier.
 * LORA_ERR_ARG for an id out of range. */
int lora_tier_cache_resident(const lora_tier_cache *cache, int adapter);

/* Replays a request trace (adapter ids in 0..n_keys-1) through a fresh
 * cache: counts[0] GPU hits, counts[1] host hits, counts[2] disk loads.
 * Errors: LORA_ERR_ARG (NULL, n < 0, an id out of range). */
int lora_tier_sim(const int *trace, long long n, int n_keys, int gpu_slots, int host_slots,
                  long long *counts);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */
