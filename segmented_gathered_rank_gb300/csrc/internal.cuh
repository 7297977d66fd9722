// Internal declarations shared by the library's translation units.
//
// Pool layout in HBM (all owned by lora_pool):
//   pages   n_pages x page_elems elements of the pool dtype.  One page holds
//           one row of A_T (h_in elements) or one row of B (h_out elements);
//           a rank-r adapter on one matrix owns 2r pages anywhere in the
//           pool (S-LoRA slide 8: pages of H elements, R of them for a
//           rank-R adapter), so mixed ranks need no padding.
//   table   one record of rec_ints int32 per (adapter, matrix), record index
//           adapter * n_matrices + matrix:
//             [0] rank (-1 = not loaded)   [1] scale (float bits)
//             [2] [3] reserved
//             [4 .. 4+r)      page ids of the rows of A_T
//             [4+r .. 4+2r)   page ids of the rows of B
//           rec_ints = 4 + 2*max_rank rounded up to a multiple of 4, so a
//           record starts on a 16-byte boundary.
//   status  one int32 device status word (LORA_DEV_* bits).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <vector>

#include "lora.h"

namespace lora {

constexpr int kRecHeader = 4;

// The tensor-core GEMM adds the adapter term itself for an M-tile of
// kFuseTileRows rows that all use one adapter of rank <= kFuseMaxRank (in
// 32-rank rounds); the plan marks such tiles, the tensor-core shrink computes
// their v, and the warp-MMA shrink and the expand skip their rows.
constexpr int kFuseTileRows = 128;
constexpr int kFuseMaxRank = 128;

// Everything a kernel needs to resolve (adapter, matrix) -> rows of pages.
struct PoolView {
    void *pages;
    const int *table;
    int *status;
    long long page_elems;
    int n_pages;
    int rec_ints;
    int n_matrices;
    int max_adapters;
    int max_rank;
};

extern std::atomic<unsigned long long> g_launches;
inline void count_launch(int n = 1) { g_launches.fetch_add((unsigned long long)n); }

}  // namespace lora

struct lora_pool {
    int device;
    int dtype;
    int esize;
    int page_elems;
    int n_pages;
    int max_rank;
    int n_matrices;
    int max_adapters;
    int rec_ints;
    void *d_pages;
    int *d_table;
    int *d_status;
    std::vector<int> free_pages;      // stack of free page ids
    std::vector<int> host_table;      // mirror of the device table
    std::vector<int> mat_h_in;        // per matrix, -1 until the first load
    std::vector<int> mat_h_out;
    std::vector<int> mat_n_ids;       // per matrix: 1 + largest adapter id ever loaded
    std::vector<int> mat_max_rank;    // per matrix: largest rank ever loaded
    // load staging: a ring of n_slots slots, each a pinned host buffer -> a device
    // buffer -> the scatter kernel and the record copy; a slot is reused once the
    // event recorded after its last copy has completed
    void *h_stage;                    // n_slots x stage_bytes, pinned
    void *d_stage;                    // n_slots x stage_bytes
    size_t stage_bytes;
    int n_slots;
    int next_slot;
    std::vector<cudaEvent_t> slot_done;
    std::vector<char> slot_busy;
    // pages of replaced or unloaded adapters: back to the free list once the
    // event recorded after the table update that retired them has completed
    struct Deferred {
        std::vector<int> pages;
        cudaEvent_t done;
    };
    std::vector<Deferred> deferred;
    std::vector<cudaEvent_t> spare_events;

    lora::PoolView view() const {
        lora::PoolView v;
        v.pages = d_pages;
        v.table = d_table;
        v.status = d_status;
        v.page_elems = page_elems;
        v.n_pages = n_pages;
        v.rec_ints = rec_ints;
        v.n_matrices = n_matrices;
        v.max_adapters = max_adapters;
        v.max_rank = max_rank;
        return v;
    }
};

namespace lora {

// ---------------------------------------------------------------------------
// Host-side argument checks shared by the compute entry points.
// ---------------------------------------------------------------------------
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Checks pool/matrix and returns LORA_OK with h_in/h_out filled in.
inline int matrix_dims(const lora_pool *pool, int matrix, int *h_in, int *h_out) {
    if (!pool || matrix < 0 || matrix >= pool->n_matrices) return LORA_ERR_ARG;
    if (pool->mat_h_in[matrix] < 0) return LORA_ERR_SHAPE;   // nothing loaded on it yet
    *h_in = pool->mat_h_in[matrix];
    *h_out = pool->mat_h_out[matrix];
    return LORA_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag(int *status, int bits) { atomicOr(status, bits); }

// Record of (adapter a, matrix m), or nullptr after flagging an invalid id.
__device__ __forceinline__ const int *lookup(const PoolView &pv, int a, int m) {
    if (a >= pv.max_adapters) {
        flag(pv.status, LORA_DEV_BAD_ADAPTER);
        return nullptr;
    }
    const int *rec = pv.table + ((long long)a * pv.n_matrices + m) * pv.rec_ints;
    if (rec[0] < 0) {
        flag(pv.status, LORA_DEV_BAD_ADAPTER);
        return nullptr;
    }
    return rec;
}

template <typename E>
__device__ __forceinline__ const E *page_row(const PoolView &pv, int page) {
    return reinterpret_cast<const E *>(pv.pages) + (long long)page * pv.page_elems;
}

// Segment containing token t: the last s in [0, S) with seg_starts[s] <= t
// (so empty segments are skipped), clamped into range.
__device__ __forceinline__ int segment_of(const int *seg_starts, int S, int t) {
    int lo = 0, hi = S;   // first index in [0, S] whose start exceeds t
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (__ldg(seg_starts + mid) > t) hi = mid; else lo = mid + 1;
    }
    int s = lo - 1;
    return s < 0 ? 0 : (s >= S ? S - 1 : s);
}

// 8 consecutive elements <-> 8 floats (16-byte aligned for bf16; 32 for f32).
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *o) {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float *p, float *o) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    float4 b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float *o) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void store8(float *p, const float *o) {
    *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The adapter whose term the tensor-core GEMM adds itself for the M-tile of
// rows [r0, r1): the one adapter every non-empty segment overlapping the tile
// uses, or -1 when the tile mixes adapters, has a token without an adapter
// (id < 0), or names an id >= n_ids (never loaded on the matrix).  sb: the S+1
// segment bounds clamped into [0, T]; sa: the S segment adapters.  The caller
// still checks the adapter's rank (1 .. kFuseMaxRank).  Segments are visited
// from the one holding r0 onwards, stopping at the first bound >= r1, 32 at a
// time by one warp (all 32 lanes call it and get the result).  The
// tensor-core shrink (its own tile) and the rows / plan kernels (every tile)
// decide with this one function on the same table, so they agree.
__device__ __forceinline__ int uniform_tile_adapter(const int *sb, const int *sa, int S, int n_ids, int r0, int r1) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = S;                     // first segment bound above r0
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sb[mid] > r0) hi = mid; else lo = mid + 1;
    }
    int a = -1;
    bool have = false, uniform = true;
    for (int base = lo > 0 ? lo - 1 : 0; base < S; base += 32) {
        const int s = base + lane;
        const bool in = s < S;
        const unsigned stopm = __ballot_sync(0xffffffffu, in && sb[s] >= r1);
        const int lim = stopm ? __ffs(stopm) - 1 : 32;   // lanes at or past the first stop are out
        const bool valid = in && lane < lim && sb[s + 1] > sb[s];
        const int val = valid ? ((sa[s] >= 0 && sa[s] < n_ids) ? sa[s] : -1) : 0;
        const unsigned vm = __ballot_sync(0xffffffffu, valid);
        if (vm) {
            const int first = __shfl_sync(0xffffffffu, val, __ffs(vm) - 1);
            if (!have) {
                a = first;
                have = true;
            }
            if (__any_sync(0xffffffffu, valid && val != a)) uniform = false;
        }
        if (stopm || !uniform) break;
    }
    return (have && uniform) ? a : -1;
}

// Checks a device segment table; every thread of the block calls it (the
// starts are read in parallel, then OR-reduced).  Sets LORA_DEV_BAD_SEGMENTS.
__device__ __forceinline__ void check_segments(const int *seg_starts, int S, int T, int *status) {
    bool bad = threadIdx.x == 0 && (seg_starts[0] != 0 || seg_starts[S] != T);
    for (int s = threadIdx.x; s < S; s += blockDim.x) bad |= seg_starts[s + 1] < seg_starts[s];
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag(status, LORA_DEV_BAD_SEGMENTS);
}

// ---------------------------------------------------------------------------
// Launchers implemented in the kernel translation units.
// ---------------------------------------------------------------------------
int launch_shrink(const lora_pool *pool, int matrix, int h_in, const void *x, float *v, int ld_v,
                  const int *seg_starts, const int *seg_adapter, int S, int T, cudaStream_t st);
int launch_expand(const lora_pool *pool, int matrix, int h_out, const float *v, int ld_v, void *y,
                  const int *seg_starts, const int *seg_adapter, int S, int T, cudaStream_t st);
int launch_bgmv(const lora_pool *pool, int matrix, int h_in, int h_out, const void *x, void *y,
                const int *token_adapter, int T, cudaStream_t st);
bool bgmv_cluster_ok(const lora_pool *pool, int h_in, int h_out, int T, int n_ids);
int launch_bgmv_cluster(const lora_pool *pool, int matrix, int h_in, int h_out, const void *x, void *y,
                        const int *token_adapter, int T, int n_ids, cudaStream_t st);
bool sgmv_shrink_ok(const lora_pool *pool, int h_in, int S);
bool sgmv_expand_ok(const lora_pool *pool, int h_out, int S);
// plan: nullptr (items from the segment table) or a plan from launch_sgmv_plan
// skip_fused (with a layer plan that fuses M-tiles into the GEMM): the plan's shrink units, which
// leave out the rows of those tiles (the tensor-core shrink computes their v), by persistent
// clusters; the expand takes the plan's expand units when given tile_ad.  tc_min_rows > 0
// (segment tables): items of
// segments the tensor-core shrink takes (that many rows or more, rank kShrinkTcSegMinRank..kFuseMaxRank)
// are skipped.
int launch_sgmv_shrink(const lora_pool *pool, int matrix, int h_in, const void *x, float *v, int ld_v,
                       const int *seg_starts, const int *seg_adapter, int S, int T, const int *plan,
                       cudaStream_t st, bool skip_fused = false, int tc_min_rows = 0);
int launch_sgmv_expand(const lora_pool *pool, int matrix, int h_out, const float *v, int ld_v, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T, const int *plan,
                       cudaStream_t st, const int *tile_ad = nullptr);
// Groups a batch's tokens by adapter into kM-token items (counting sort).
// units: the plan also lists the persistent shrink / expand units (layer plans with GEMM-fused tiles)
bool sgmv_plan_ok(const lora_pool *pool, int matrix, int S, int T, bool units);
size_t sgmv_plan_bytes(const lora_pool *pool, int matrix, int T);
// The plan's per-M-tile array (after its items).
int *sgmv_plan_tiles(const lora_pool *pool, int matrix, int T, int *plan);
// units: a layer plan -- the plan also classifies the GEMM M-tiles (uniform_tile_adapter, as
// the tensor-core shrink does), masks the fused rows and lists the shrink and expand units.
int launch_sgmv_plan(const lora_pool *pool, int matrix, const int *seg_starts, const int *seg_adapter, int S, int T,
                     int *plan, cudaStream_t st, bool units = false);
int num_sms();   // SMs of the current device (cached per device)
// Opts kernel `func` in to `bytes` of dynamic shared memory on the current
// device (raising the attribute only when a launch needs more than before,
// once per device and kernel; thread safe).  occupancy (optional): resident
// CTAs per SM of `threads` threads at that size.  LORA_OK or LORA_ERR_CUDA.
int smem_optin(const void *func, size_t bytes, int threads = 0, int *occupancy = nullptr);
// The FP8 base product: x quantised per row (codes xq [T x h_in], scales sx [T]) against
// W given as e4m3 codes with one scale w_scale; see lora_layer_forward_fp8.
struct Fp8Base {
    const void *xq;
    const float *sx;
    float w_scale;
    bool quantize;      // the layer call writes xq and sx from x itself (before its GEMM)
};
// Per-row e4m3 codes and scales of x (see lora_quantize_e4m3).
int launch_quantize(const void *x, int T, int h, void *q, float *sx, cudaStream_t st);
bool gemm_tc_ok(const lora_pool *pool, int h_in, int h_out, int T, bool fp8 = false);
// tile_ad != nullptr: M-tiles with tile_ad[m] >= 0 also get that adapter's term
// s * v . B (v: T x ld_v fp32) inside the GEMM.  f8 != nullptr: W holds e4m3 codes and
// the base product is the FP8 one.
int launch_gemm_tc(const lora_pool *pool, int h_in, int h_out, const void *x, const void *W, void *y, int T,
                   cudaStream_t st, int matrix = 0, const int *tile_ad = nullptr, const float *v = nullptr,
                   int ld_v = 0, const Fp8Base *f8 = nullptr);
// Tensor-core shrink (tcgen05) of 128-row tiles that share one adapter of
// rank 1..kFuseMaxRank: the fused layer's uniform M-tiles (tile_ad), or, for
// a segment table, 128-row pieces of the segments with at least
// kShrinkTcMinRows rows and rank at least kShrinkTcSegMinRank (measured: at
// lower ranks the warp-MMA shrink is as fast, both being bound by reading x,
// and a second launch only adds latency; the warp-MMA SGMV shrink skips the
// segments taken here).  K is split over up to
// kShrinkTcSplits CTAs of a cluster.
constexpr int kShrinkTcSplits = 4;
constexpr int kShrinkTcMinRows = 64;
constexpr int kShrinkTcSegMinRank = 65;
constexpr int kShrinkTcMaxS = 8192;
bool shrink_tc_ok(const lora_pool *pool, int h_in, int S);
int launch_shrink_tc(const lora_pool *pool, int matrix, int h_in, const void *x, int T, int *tile_ad,
                     const int *seg_starts, const int *seg_adapter, int S, float *v, int ld_v, cudaStream_t st);
// f8 != nullptr: the base product is the FP8 one (W holds e4m3 codes; tensor cores required).
int layer_forward_impl(const lora_pool *p, int matrix, int h_in, int h_out, const void *x, const void *W, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T, float *v, cudaStream_t st,
                       const Fp8Base *f8 = nullptr);
int launch_base_gemm(const lora_pool *pool, int h_in, int h_out, const void *x, const void *W, void *y,
                     int T, cudaStream_t st);

}  // namespace lora
