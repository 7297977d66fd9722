// SGMV for prefill: the gathered low-rank product over runs of consecutive
// tokens that share one adapter ("Multi-LoRA Serving", section "The kernel
// trick: gather, do not merge"), with per-adapter ranks (S-LoRA slide 10, MBGMM).
//
//   shrink:  v[t][j]  = sum_k x[t][k] * A_T_a[j][k]            j < r_a
//   expand:  y[t][n] += s_a * sum_j v[t][j] * B_a[j][n]
//
// Work items are one adapter and up to kM of its tokens.  They come either
// from the segment table (each segment cut into kM-token chunks; a CTA finds
// each of its items with a block-wide scan of chunk counts and a binary search,
// so Zipf-skewed segment lengths spread over as many CTAs as they have
// chunks), or from a plan built by sgmv_plan_kernel, which groups the tokens
// of a batch by adapter with a counting sort (so a decode batch whose tokens
// are one-token segments still gets items of up to kM tokens).
//
// For the adapted layer the plan also marks the GEMM M-tiles whose rows share
// one adapter (the GEMM adds their term itself) and lists, for the items that
// keep other rows, work units ordered by cost: shrink units (a 16-row half x
// a 32-rank chunk) and expand units (a range of column blocks, sized so that
// the batch's units fill the resident CTAs about once).  Persistent kernels
// walk these lists in snake order, the
// shrink as clusters of two CTAs that split K and add their partial sums
// through distributed shared memory.
//
// Adapter pages, x and y move with 16-byte asynchronous copies through
// multi-stage shared-memory pipelines; the products run on the tensor cores
// as warp-level mma.sync m16n8k16 (bf16 -> fp32) -- tiles here are 32
// tokens by at most a few dozen ranks, and the kernels are bound by HBM
// traffic, not MMA rate.  In the expand, v enters the MMA as a bf16 high part
// plus a bf16 residual, which keeps the product within fp32-level error.
#include <cooperative_groups.h>

#include <algorithm>

#include "internal.cuh"

namespace lora {
namespace {

namespace cg = cooperative_groups;

constexpr int kM = 32;            // tokens per item (one per lane where a warp collects an item's tokens)
static_assert(kM == 32, "an item's tokens are collected one per lane of a warp");
constexpr int kKs = 128;          // k per shrink pipeline stage
constexpr int kRowsS = 16;        // rows per 128-thread shrink CTA (half an item)
constexpr int kStagesS = 4;
constexpr int kNb = 128;          // output columns per expand block
constexpr int kMaxBlocksPerUnit = 8; // column blocks per expand unit (up to 1024 columns)
constexpr int kStagesE = 2;      // expand ring depth: shallow rings leave room for more CTAs per SM
constexpr int kMaxS = 8192;       // segments the segment-mode kernels take
constexpr int kPlanThreads = 1024;
constexpr int kTileRows = kFuseTileRows;   // M-tile rows of the tensor-core GEMM

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int clamp_page(const PoolView &pv, int id) {
    return id < 0 ? 0 : (id >= pv.n_pages ? pv.n_pages - 1 : id);
}

// Exclusive scan of v[0..n) in place by a block of NT threads; returns the total.
template <int NT>
__device__ int block_scan(int *v, int n, int *wtot) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + NT - 1) / NT;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += v[i];
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) wtot[warp] = inc;
    __syncthreads();
    if (warp == 0) {      // exclusive scan of the warp totals (NW <= 32)
        const int t = lane < NW ? wtot[lane] : 0;
        int run = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run += u;
        }
        if (lane < NW) wtot[lane] = run - t;
        if (lane == NW - 1) wtot[NW] = run;
    }
    __syncthreads();
    int run = wtot[warp] + inc - sum;
    for (int i = lo; i < hi; ++i) {
        const int t = v[i];
        v[i] = run;
        run += t;
    }
    const int total = wtot[NW];
    __syncthreads();
    return total;
}

__device__ __forceinline__ int4 add4(int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

// Exclusive scan of four counts per element (v[0..n)) in place; returns the four totals.
// wtot: NT/32 + 1 int4 of shared memory.
template <int NT>
__device__ int4 block_scan4(int4 *v, int n, int4 *wtot) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + NT - 1) / NT;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int4 sum = make_int4(0, 0, 0, 0);
    for (int i = lo; i < hi; ++i) sum = add4(sum, v[i]);
    int4 inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int4 t = make_int4(__shfl_up_sync(0xffffffffu, inc.x, o), __shfl_up_sync(0xffffffffu, inc.y, o),
                                 __shfl_up_sync(0xffffffffu, inc.z, o), __shfl_up_sync(0xffffffffu, inc.w, o));
        if (lane >= o) inc = add4(inc, t);
    }
    if (lane == 31) wtot[warp] = inc;
    __syncthreads();
    if (warp == 0) {      // exclusive scan of the warp totals (NW <= 32)
        const int4 t = lane < NW ? wtot[lane] : make_int4(0, 0, 0, 0);
        int4 run = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int4 u = make_int4(__shfl_up_sync(0xffffffffu, run.x, o), __shfl_up_sync(0xffffffffu, run.y, o),
                                     __shfl_up_sync(0xffffffffu, run.z, o), __shfl_up_sync(0xffffffffu, run.w, o));
            if (lane >= o) run = add4(run, u);
        }
        if (lane < NW) wtot[lane] = make_int4(run.x - t.x, run.y - t.y, run.z - t.z, run.w - t.w);
        if (lane == NW - 1) wtot[NW] = run;
    }
    __syncthreads();
    int4 run = wtot[warp];
    run = make_int4(run.x + inc.x - sum.x, run.y + inc.y - sum.y, run.z + inc.z - sum.z, run.w + inc.w - sum.w);
    for (int i = lo; i < hi; ++i) {
        const int4 t = v[i];
        v[i] = run;
        run = add4(run, t);
    }
    const int4 total = wtot[NW];
    __syncthreads();
    return total;
}

// An item: adapter `a` and its tokens; row i of the item is token
// perm ? perm[off + i] : off + i.
struct Item {
    int a;
    int off;
    int nt;
    int pad;    // segment tables: the segment's length
};

// A unit of the persistent shrink and expand kernels of a layer plan: one
// work item's rows with one rank chunk (shrink) or a range of column blocks
// (expand).  The plan lists the costly units first.
struct Unit {
    int a;
    int off;
    int info;   // bits 0-5: the item's token count; shrink: bit 6 the 16-row half, bits 8+ the rank
                // chunk; expand: bits 6-9 the unit's column blocks, bits 10+ its first column block
    int pad;    // the item's mask of rows whose term the GEMM adds
};

// Item `idx` among the (segment, kM-token chunk) pairs of a segment table.
// scan: S + 1 ints of shared memory; wtot: NT/32 + 4 ints.  All threads return it.
template <int NT>
__device__ int segment_scan(const int *seg_starts, int S, int T, int *scan, int *wtot) {
    for (int s = threadIdx.x; s < S; s += NT) {
        const int a = min(max(seg_starts[s], 0), T), b = min(max(seg_starts[s + 1], 0), T);
        scan[s] = b > a ? (b - a + kM - 1) / kM : 0;
    }
    __syncthreads();
    return block_scan<NT>(scan, S, wtot);
}

// Item idx from a chunk scan made by segment_scan (total: its chunk count).
// All threads call it and return the item.
template <int NT>
__device__ Item segment_lookup(const int *seg_starts, const int *seg_adapter, int S, int T, int idx,
                               const int *scan, int total, int *wtot) {
    if (threadIdx.x == 0) {
        Item it{-1, 0, 0, 0};
        if (idx < total) {
            int lo = 0, hi = S - 1;               // last segment whose first chunk index <= idx
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (scan[mid] <= idx) lo = mid; else hi = mid - 1;
            }
            const int c = idx - scan[lo];
            const int beg = min(max(seg_starts[lo], 0), T), end = min(max(seg_starts[lo + 1], 0), T);
            it.a = seg_adapter[lo];
            it.off = beg + c * kM;
            it.nt = min(kM, end - it.off);
            it.pad = end - beg;           // segment tables: the segment's length
        }
        reinterpret_cast<Item *>(wtot)[0] = it;
    }
    __syncthreads();
    const Item it = reinterpret_cast<Item *>(wtot)[0];
    __syncthreads();
    return it;
}

template <int NT>
__device__ Item segment_item(const int *seg_starts, const int *seg_adapter, int S, int T, int idx, int *scan,
                             int *wtot) {
    const int total = segment_scan<NT>(seg_starts, S, T, scan, wtot);
    return segment_lookup<NT>(seg_starts, seg_adapter, S, T, idx, scan, total, wtot);
}

// The work items of one launch: from a plan (if given) or from the segment table.
struct ItemSource {
    const int *seg_starts, *seg_adapter;
    int S, T;
    const int *plan;     // nullptr, or a plan (see plan_layout): perm[T] and items[...] as Item
};

__device__ __forceinline__ const int *plan_perm(const int *plan) { return plan + 4; }
__device__ __forceinline__ const Item *plan_items(const int *plan, int T) {
    return reinterpret_cast<const Item *>(plan + 4 + ((T + 3) & ~3));
}

// Entry i of a plan's token permutation, i clamped into [0, T) (a plan is
// read only after its kernel wrote it; the clamp keeps a damaged workspace
// from sending a read outside the plan).
__device__ __forceinline__ int perm_at(const ItemSource &src, int i) {
    return plan_perm(src.plan)[min(max(i, 0), src.T - 1)];
}

template <int NT>
__device__ Item get_item(const ItemSource &src, int idx, int *scan, int *wtot) {
    if (src.plan) return plan_items(src.plan, src.T)[idx];   // idx < the plan's item bound; unused items have a = -1
    return segment_item<NT>(src.seg_starts, src.seg_adapter, src.S, src.T, idx, scan, wtot);
}

// Record of adapter a on matrix m into smem; false (after flagging) when invalid.
template <int NT>
__device__ bool load_record(const PoolView &pv, int a, int m, int *rec, bool report) {
    if (a >= pv.max_adapters) {
        if (report) flag(pv.status, LORA_DEV_BAD_ADAPTER);
        return false;
    }
    for (int i = threadIdx.x; i < pv.rec_ints; i += NT)
        rec[i] = pv.table[((long long)a * pv.n_matrices + m) * pv.rec_ints + i];
    __syncthreads();
    if (rec[0] < 0) {
        if (report) flag(pv.status, LORA_DEV_BAD_ADAPTER);
        return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// Plan: tokens grouped by adapter (counting sort), cut into kM-token items.
// ---------------------------------------------------------------------------
struct PlanParams {
    const int *seg_starts, *seg_adapter;
    int S, T;
    int n_ids;          // adapter ids below this may be loaded on the matrix
    int *status;
    int *plan;          // output, see ItemSource
    int max_items;
    PoolView pv;        // for ranks of the tile classification
    int m;
    bool units;         // layer plan: classify the GEMM M-tiles (as the tensor-core shrink does) and list units
    int n_tiles;
    Unit *su, *eu;      // with units: shrink and expand units of the work items (counts plan[2], plan[3])
    int npc_s;          // ranks per shrink unit
    int nb_total;       // column blocks of kNb in h_out
    int e_ctas;         // resident CTAs of the expand-units kernel
    int rank_cap;       // ranks beyond this are not computed (the v row length)
    int body;           // ints of the counting-sort area of shared memory
};

// An item's expand cost per column block, in 256-byte rows: its y rows, read
// and written once per pass of up to 32 ranks, plus its B rows.
__device__ __forceinline__ int expand_cost(int nt, int r) { return 2 * nt * ((r + 31) / 32) + r; }

__global__ void __launch_bounds__(kPlanThreads) sgmv_plan_kernel(PlanParams p) {
    extern __shared__ __align__(16) int sm[];
    int *cnt = sm;                       // [n_ids] tokens per adapter
    int *base = cnt + p.n_ids;           // [n_ids] token offset of each adapter
    int *ibase = base + p.n_ids;         // [n_ids] item offset of each adapter
    int *segoff = ibase + p.n_ids;       // [S] offset of each segment within its adapter's tokens
    int *sb = segoff + p.S;              // [S + 1] segment bounds, clamped into [0, T]
    int *sa = sb + p.S + 1;              // [S] segment adapters (-1: none or invalid)
    int *arank = sa + p.S;               // with units: [n_ids] each adapter's rank on the matrix
    int *sperm = arank + p.n_ids;        // with units: [T] copy of the token permutation
    int *tflag = sperm + p.T;            // with units: [n_tiles] the adapter of each GEMM-fused M-tile, or -1
    int *wtot = sm + p.body;             // [kPlanThreads / 32 + 1], then the work count
    // with units: [max_items] int4 work items, int4 unit counts and ranks, after the counters
    int4 *sitem = reinterpret_cast<int4 *>(sm + p.body + ((kPlanThreads / 32 + 2 + 3) & ~3));
    int4 *ucnt = sitem + p.max_items;
    int4 *wtot4 = ucnt + p.max_items;    // [kPlanThreads / 32 + 1]
    int *srank = reinterpret_cast<int *>(wtot4 + kPlanThreads / 32 + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = kPlanThreads / 32;
    // one round of global loads: segment bounds (checked as they arrive), segment
    // adapters and, with units, every adapter's rank
    bool bad = false;
    for (int i = tid; i < p.n_ids; i += kPlanThreads) {
        cnt[i] = 0;
        if (p.units) arank[i] = p.pv.table[((long long)i * p.pv.n_matrices + p.m) * p.pv.rec_ints];
    }
    for (int s = tid; s <= p.S; s += kPlanThreads) {
        const int b0 = p.seg_starts[s];
        if (s < p.S) bad |= p.seg_starts[s + 1] < b0;
        if (s == 0) bad |= b0 != 0;
        if (s == p.S) bad |= b0 != p.T;
        sb[s] = min(max(b0, 0), p.T);
    }
    for (int s = tid; s < p.S; s += kPlanThreads) {
        const int a = p.seg_adapter[s];
        sa[s] = a < p.n_ids ? a : -1;
        if (a >= p.n_ids) flag(p.status, LORA_DEV_BAD_ADAPTER);      // never loaded on this matrix
    }
    if (__syncthreads_or(bad) && tid == 0) flag(p.status, LORA_DEV_BAD_SEGMENTS);
    // one atomic per segment: its tokens stay contiguous and in order
    for (int s = tid; s < p.S; s += kPlanThreads) {
        const int n = sb[s + 1] - sb[s];
        segoff[s] = (sa[s] >= 0 && n > 0) ? atomicAdd(&cnt[sa[s]], n) : -1;
    }
    __syncthreads();
    for (int i = tid; i < p.n_ids; i += kPlanThreads) {
        base[i] = cnt[i];
        ibase[i] = (cnt[i] + kM - 1) / kM;
    }
    __syncthreads();
    block_scan<kPlanThreads>(base, p.n_ids, wtot);
    const int n_items = block_scan<kPlanThreads>(ibase, p.n_ids, wtot);
    int *perm = p.plan + 4;
    Item *items = reinterpret_cast<Item *>(p.plan + 4 + ((p.T + 3) & ~3));
    // one thread per item: its adapter is the last whose first item index is <= it
    Item first_item{-1, 0, 0, 0};        // this thread's item of the first round (reused below)
    for (int i = tid; i < min(n_items, p.max_items); i += kPlanThreads) {
        int lo = 0, hi = p.n_ids - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ibase[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int a = lo, c = i - ibase[a], n = cnt[a];
        // an invalid (overlapping) segment table can count more than T tokens: never point past T
        const int off = base[a] + c * kM;
        const int nt = max(0, min(min(kM, n - c * kM), p.T - off));
        items[i] = Item{nt > 0 ? a : -1, off, nt, 0};
        if (i == tid) first_item = items[i];
    }
    if (tid == 0) p.plan[0] = min(n_items, p.max_items);
    for (int i = n_items + tid; i < p.max_items; i += kPlanThreads) items[i] = Item{-1, 0, 0, 0};
    // token permutation: short segments one per thread, long ones one per warp
    for (int s = tid; s < p.S; s += kPlanThreads) {
        const int n = sb[s + 1] - sb[s];
        if (segoff[s] < 0 || n > 32) continue;
        const int dst = base[sa[s]] + segoff[s];
        for (int i = 0; i < n; ++i)
            if (dst + i < p.T) {
                perm[dst + i] = sb[s] + i;
                if (p.units) sperm[dst + i] = sb[s] + i;
            }
    }
    for (int s = warp; s < p.S; s += nwarps) {
        const int n = sb[s + 1] - sb[s];
        if (segoff[s] < 0 || n <= 32) continue;
        const int dst = base[sa[s]] + segoff[s];
        for (int i = lane; i < n; i += 32)
            if (dst + i < p.T) {
                perm[dst + i] = sb[s] + i;
                if (p.units) sperm[dst + i] = sb[s] + i;
            }
    }
    if (!p.units) return;
    int *wcount = wtot + nwarps + 1;        // past block_scan's words
    if (tid == 0) *wcount = 0;
    // the GEMM-fused M-tiles, decided as the tensor-core shrink decides them
    // (same function, same table; a warp per tile): the adapter of a tile
    // whose rows all use it, when its rank is 1..kFuseMaxRank
    for (int mb = warp; mb < p.n_tiles; mb += nwarps) {
        const int r0 = mb * kTileRows, r1 = min(p.T, r0 + kTileRows);
        const int a = uniform_tile_adapter(sb, sa, p.S, p.n_ids, r0, r1);
        if (lane == 0)
            tflag[mb] = (a >= 0 && arank[a] >= 1 && arank[a] <= kFuseMaxRank && arank[a] <= p.rank_cap) ? a : -1;
    }
    __syncthreads();
    // each item's mask of rows that sit in such tiles (the expand skips them;
    // the item's perm entries are read with independent loads); items that keep
    // other rows get a work slot (one atomic per warp) and their unit counts
    const int nitems = min(n_items, p.max_items);
    for (int i0 = 0; i0 < nitems; i0 += kPlanThreads) {
        const int i = i0 + tid;
        bool want = false;
        Item w{-1, 0, 0, 0};
        int rank = 0;
        if (i < nitems) {
            const Item it = i0 == 0 ? first_item : items[i];
            if (it.a >= 0) {
                rank = arank[it.a];
                int tk[kM];
#pragma unroll
                for (int k = 0; k < kM; ++k) tk[k] = k < it.nt ? sperm[it.off + k] : -1;
                unsigned mask = 0;
#pragma unroll
                for (int k = 0; k < kM; ++k)
                    if (tk[k] >= 0 && tk[k] < p.T && tflag[tk[k] / kTileRows] >= 0)
                        mask |= 1u << k;
                const unsigned all = it.nt >= 32 ? 0xffffffffu : ((1u << it.nt) - 1u);
                want = (mask & all) != all;        // rows left for the SGMV kernels (slot order is immaterial)
                w = it;
                w.pad = (int)mask;
            }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, want);
        int slot = 0;
        if (lane == 0 && bal) slot = atomicAdd(wcount, __popc(bal));
        slot = __shfl_sync(0xffffffffu, slot, 0);
        if (want) {
            const int k = slot + __popc(bal & ((1u << lane) - 1u));
            if (p.su) {
                // units of this item: 16-row halves that keep rows x rank chunks (shrink), column
                // block ranges (expand); counted in the costly class or the cheap one
                if (rank < 0) flag(p.status, LORA_DEV_BAD_ADAPTER);
                const int r = min(rank, p.rank_cap);
                int4 c = make_int4(0, 0, 0, 0);
                if (r > 0) {
                    const unsigned all = w.nt >= 32 ? 0xffffffffu : ((1u << w.nt) - 1u);
                    const unsigned left = ~(unsigned)w.pad & all;
                    const int nh = ((left & 0xffffu) != 0u) + ((left >> 16) != 0u);
                    const int nch = (r + p.npc_s - 1) / p.npc_s;
                    const bool costly_s = min(w.nt, kRowsS) + min(r, p.npc_s) >= 32;
                    c = make_int4(costly_s ? nh * nch : 0, costly_s ? 0 : nh * nch, 0, 0);   // expand: below
                }
                sitem[k] = make_int4(w.a, w.off, w.nt, w.pad);
                ucnt[k] = c;
                srank[k] = max(r, 0);
            }
        }
    }
    __syncthreads();
    const int n_work = *wcount;
    if (tid == 0) p.plan[1] = n_work;
    if (!p.su) return;
    // Expand units: column-block ranges sized so that the units of the whole
    // batch fill the expand kernel's resident CTAs about once (each unit pays a
    // few dependent global round trips before its copies start, so many small
    // units cost more than the data they move).  Item k gets
    // max(1, floor(C_k / target)) units, C_k its cost over all column blocks and
    // target the batch's total cost per CTA; units whose cost reaches the target
    // are listed first.  Integer sums keep the choice deterministic.
    {
        unsigned long long part = 0;
        for (int k = tid; k < n_work; k += kPlanThreads)
            if (srank[k] > 0) part += (unsigned long long)p.nb_total * expand_cost(sitem[k].z, srank[k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        unsigned long long *wsum = reinterpret_cast<unsigned long long *>(wtot4);
        if (lane == 0) wsum[warp] = part;
        __syncthreads();
        unsigned long long total = 0;
#pragma unroll
        for (int w = 0; w < nwarps; ++w) total += wsum[w];
        const unsigned long long target = max(1ull, total / (unsigned long long)max(1, p.e_ctas));
        for (int k = tid; k < n_work; k += kPlanThreads) {
            const int r = srank[k];
            if (r <= 0) continue;
            const int cost = expand_cost(sitem[k].z, r);
            const unsigned long long ck = (unsigned long long)p.nb_total * cost;
            const int units = (int)max(1ull, min((unsigned long long)p.nb_total, ck / target));
            const int passes = (r + 31) / 32;
            // an item of 2..kStagesE rank passes takes single-block units, so that
            // every one of its rows gets the single rounding of y of that path,
            // whichever item the row falls in (the grouping follows atomics)
            const int bpu = passes > 1 && passes <= kStagesE ? 1 : min(kMaxBlocksPerUnit, (p.nb_total + units - 1) / units);
            const int ne = (p.nb_total + bpu - 1) / bpu;
            const bool costly = (unsigned long long)bpu * cost >= target;
            ucnt[k].z = costly ? ne : 0;
            ucnt[k].w = costly ? 0 : ne;
            srank[k] = r | (costly ? 1 << 12 : 0) | (bpu << 16);     // r <= 1024
        }
        __syncthreads();                 // wsum (over the scan's scratch) is read; the counts are written
    }
    const int4 tot = block_scan4<kPlanThreads>(ucnt, n_work, wtot4);
    for (int k = tid; k < n_work; k += kPlanThreads) {
        const int r = srank[k] & 0xfff, bpu = srank[k] >> 16;
        const bool costly = (srank[k] >> 12) & 1;
        if (r <= 0) continue;
        const int4 w = sitem[k], c = ucnt[k];
        const unsigned all = w.z >= 32 ? 0xffffffffu : ((1u << w.z) - 1u);
        const unsigned left = ~(unsigned)w.w & all;
        const int nch = (r + p.npc_s - 1) / p.npc_s;
        const bool costly_s = min(w.z, kRowsS) + min(r, p.npc_s) >= 32;
        int u = costly_s ? c.x : tot.x + c.y;
        for (int h = 0; h < 2; ++h) {
            if (!((left >> (16 * h)) & 0xffffu)) continue;
            for (int ch = 0; ch < nch; ++ch) p.su[u++] = Unit{w.x, w.y, w.z | (h << 6) | (ch << 8), w.w};
        }
        u = costly ? c.z : tot.z + c.w;
        for (int b = 0; b < p.nb_total; b += bpu)
            p.eu[u++] = Unit{w.x, w.y, w.z | (min(bpu, p.nb_total - b) << 6) | (b << 10), w.w};
    }
    if (tid == 0) {
        p.plan[2] = tot.x + tot.y;
        p.plan[3] = tot.z + tot.w;
    }
}

// ---------------------------------------------------------------------------
// Shrink: 128 threads, one half (16 tokens) of an item x one chunk of npc
// ranks; K in 128-wide stages, warp w takes k 32w .. 32w+31 of every stage and
// the four partial sums are added at the end.  Two kernels share the core:
// one CTA per (item, chunk, half) from the grid, or (layer plans) persistent
// clusters that walk the plan's unit list and split K over the cluster's CTAs.
// ---------------------------------------------------------------------------
constexpr int kThreadsS = 128;

struct ShrinkParams {
    PoolView pv;
    ItemSource src;
    int m, h_in;
    int tc_min_rows;   // > 0: skip segments of at least this many rows the tensor-core shrink takes
    int npc;       // ranks per CTA: max_rank rounded up to 16, at most 32 (64 in the wide kernel); grid.y covers the rest
    int alias_bytes;   // wide kernel: shared bytes of the ring / segment scan / partial sums (they alias)
    const __nv_bfloat16 *x;
    float *v;
    int ld_v;
    const Unit *units;   // unit kernel: the plan's shrink units (count plan[2])
    int max_units;       // unit kernel: the plan's room for shrink units
    int n_work, n_chunks;   // wide kernel: (item, rank chunk) work entries; rank chunks per item
};

// Rows tok[0 .. nt) of x, K stages kc0 .. kc1-1, times ranks j0 .. j0+np-1 of the
// adapter whose record is in rec.  On return warp 0's d holds the CTA's sums
// (fragment rows g and g + 8, rank pairs t * 8 + 2q); the other warps' d are spent.
__device__ __forceinline__ void shrink_core(const ShrinkParams &p, const int *tok, int nt, const int *rec, int j0,
                                            int np, int kc0, int kc1, __nv_bfloat16 *sx, __nv_bfloat16 *sa,
                                            float *red, float (&d)[4][4]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int pitch = kKs + 8;                                        // bf16 per smem row
    const int npc = p.npc;
    const int npad = (np + 15) & ~15;
    // rows that never receive copies stay zero
    for (int i = tid; i < kStagesS * kRowsS * (pitch / 8); i += kThreadsS)
        if ((i / (pitch / 8)) % kRowsS >= nt) reinterpret_cast<uint4 *>(sx)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < kStagesS * npc * (pitch / 8); i += kThreadsS)
        if ((i / (pitch / 8)) % npc >= np) reinterpret_cast<uint4 *>(sa)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    const int g = lane >> 2, q = lane & 3;
    const int nk = kc1 - kc0;
    // this thread's 16-byte copy slots, fixed for the whole K loop: element
    // tid + 128 k of the 16 rows x 16 chunks of x (k < 2) and of the npc rows
    // x 16 chunks of A_T (k < 4)
    const __nv_bfloat16 *xs[2], *as[4];
    uint32_t xd[2], ad[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = tid + k * kThreadsS, row = i >> 4, kv = i & 15;
        xs[k] = row < nt ? p.x + (long long)tok[row] * p.h_in + kc0 * kKs + kv * 8 : nullptr;
        xd[k] = (uint32_t)(row * pitch + kv * 8);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = tid + k * kThreadsS, row = i >> 4, kv = i & 15;
        as[k] = row < np ? page_row<__nv_bfloat16>(p.pv, clamp_page(p.pv, rec[kRecHeader + j0 + row])) + kc0 * kKs +
                               kv * 8
                         : nullptr;
        ad[k] = (uint32_t)(row * pitch + kv * 8);
    }
    auto issue = [&](int kc) {
        const int st = kc % kStagesS;
        __nv_bfloat16 *dx = sx + st * kRowsS * pitch;
        __nv_bfloat16 *da = sa + st * npc * pitch;
        const int ko = kc * kKs;
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (xs[k]) cp_async16(dx + xd[k], xs[k] + ko);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (as[k]) cp_async16(da + ad[k], as[k] + ko);
    };
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[t][e] = 0.f;
#pragma unroll
    for (int kc = 0; kc < kStagesS - 1; ++kc) {
        if (kc < nk) issue(kc);
        cp_commit();
    }
    for (int kc = 0; kc < nk; ++kc) {
        cp_wait<kStagesS - 2>();
        __syncthreads();
        if (kc + kStagesS - 1 < nk) issue(kc + kStagesS - 1);
        cp_commit();
        const int st = kc % kStagesS;
        const __nv_bfloat16 *bx = sx + st * kRowsS * pitch;
        const __nv_bfloat16 *ba = sa + st * npc * pitch;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {                   // this warp's quarter of the stage
            const int k = warp * 32 + ks * 16;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(bx + (lane & 15) * pitch + k + (lane >> 4) * 8, a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < 4; t += 2) {
                if (t * 8 >= npad) break;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(ba + (t * 8 + (lane & 7) + ((lane >> 4) << 3)) * pitch + k + ((lane >> 3) & 1) * 8, b0, b1,
                        b2, b3);
                mma16816(d[t], a0, a1, a2, a3, b0, b1);
                mma16816(d[t + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    cp_wait<0>();
    // add the four k-quarter partials into warp 0's fragment
    if (warp > 0) {
        float *rw = red + (warp - 1) * 16 * npc;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t * 8 >= npad) break;
            rw[g * npc + t * 8 + 2 * q] = d[t][0];
            rw[g * npc + t * 8 + 2 * q + 1] = d[t][1];
            rw[(g + 8) * npc + t * 8 + 2 * q] = d[t][2];
            rw[(g + 8) * npc + t * 8 + 2 * q + 1] = d[t][3];
        }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t * 8 >= npad) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g + 8 * h, j = t * 8 + 2 * q;
#pragma unroll
                for (int w = 0; w < 3; ++w) {
                    d[t][2 * h] += red[w * 16 * npc + row * npc + j];
                    d[t][2 * h + 1] += red[w * 16 * npc + row * npc + j + 1];
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreadsS, 4) sgmv_shrink_kernel(ShrinkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int pitch = kKs + 8;                                        // bf16 per smem row
    const int npc = p.npc;
    __nv_bfloat16 *sx = reinterpret_cast<__nv_bfloat16 *>(smem_raw);     // [stages][16][pitch]
    __nv_bfloat16 *sa = sx + kStagesS * kRowsS * pitch;                  // [stages][npc][pitch]
    float *red = reinterpret_cast<float *>(sa + kStagesS * npc * pitch);  // [3][16][npc] partials of warps 1..3
    int *tok = reinterpret_cast<int *>(red + 3 * 16 * npc);              // [16]
    int *wtot = tok + kRowsS;                                            // [8]
    int *rec = wtot + 8;                                                 // [rec_ints]
    int *scan = rec + p.pv.rec_ints;                                     // [S + 1]

    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && !p.src.plan) check_segments(p.src.seg_starts, p.src.S, p.src.T, p.pv.status);
    const Item it = get_item<kThreadsS>(p.src, blockIdx.x, scan, wtot);
    const int row0 = blockIdx.z * kRowsS;
    const int nt = min(kRowsS, it.nt - row0);
    if (it.a < 0 || nt <= 0) return;
    // the item's tokens load together with the record (load_record's barrier publishes both)
    if (tid < kRowsS)
        tok[tid] = tid < nt ? min(max(p.src.plan ? perm_at(p.src, it.off + row0 + tid) : it.off + row0 + tid, 0),
                                  p.src.T - 1)
                            : 0;
    if (!load_record<kThreadsS>(p.pv, it.a, p.m, rec, tid == 0 && blockIdx.y == 0 && blockIdx.z == 0)) return;
    if (p.tc_min_rows > 0 && !p.src.plan && it.pad >= p.tc_min_rows && rec[0] >= kShrinkTcSegMinRank &&
        rec[0] <= kFuseMaxRank && rec[0] <= p.ld_v)
        return;                                  // the tensor-core shrink computed this segment
    const int r = min(rec[0], min(p.pv.max_rank, p.ld_v));
    const int j0 = blockIdx.y * npc;
    if (j0 >= r) return;
    const int np = min(npc, r - j0);
    float d[4][4];
    shrink_core(p, tok, nt, rec, j0, np, 0, p.h_in / kKs, sx, sa, red, d);
    if (warp == 0) {
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t * 8 >= np) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g + 8 * h, j = t * 8 + 2 * q;
                if (row >= nt) continue;
                float *vrow = p.v + (long long)tok[row] * p.ld_v + j0;
                if (j < np) vrow[j] = d[t][2 * h];
                if (j + 1 < np) vrow[j + 1] = d[t][2 * h + 1];
            }
        }
    }
}

// Layer plans: each cluster of ks CTAs (grid (ks, clusters)) walks the plan's
// shrink units, CTA c of the cluster taking the c-th of ks equal K ranges.  The
// ks partial sums meet in distributed shared memory; CTA c adds, in cluster
// rank order, the rows congruent to c mod ks and writes them to v.  Rows whose
// tile the tensor-core shrink covers keep that kernel's v.
__global__ void __launch_bounds__(kThreadsS, 3) sgmv_shrink_units_kernel(ShrinkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int pitch = kKs + 8;
    const int npc = p.npc;
    __nv_bfloat16 *sx = reinterpret_cast<__nv_bfloat16 *>(smem_raw);     // [stages][16][pitch]
    __nv_bfloat16 *sa = sx + kStagesS * kRowsS * pitch;                  // [stages][npc][pitch]
    float *red = reinterpret_cast<float *>(sa + kStagesS * npc * pitch);  // [3][16][npc] partials of warps 1..3
    float *part = red + 3 * 16 * npc;                                    // [16][npc] this CTA's sums
    int *tok = reinterpret_cast<int *>(part + 16 * npc);                 // [16]
    int *rec = tok + kRowsS;                                             // [rec_ints]

    cg::cluster_group cl = cg::this_cluster();
    const int ks = (int)cl.num_blocks(), kpart = (int)cl.block_rank();
    const int n_units = min(max(p.src.plan[2], 0), p.max_units);
    const int G = gridDim.y, c = blockIdx.y;
    const int nk = p.h_in / kKs;
    const int kc0 = kpart * nk / ks, kc1 = (kpart + 1) * nk / ks;
    const int g = lane >> 2, q = lane & 3;
    for (int k = 0;; ++k) {
        // snake order over the cost-sorted list: cluster c takes units c, 2G - 1 - c, 2G + c, ...
        const int u = k * G + ((k & 1) ? G - 1 - c : c);
        if (u >= n_units) break;                  // the same for every CTA of the cluster
        const Unit un = p.units[u];
        const int row0 = ((un.info >> 6) & 1) * kRowsS, chunk = (int)((unsigned)un.info >> 8);
        const int nt = min(kRowsS, (un.info & 63) - row0);
        __syncthreads();                          // the previous unit's readers of tok and rec are done
        if (tid < kRowsS)
            tok[tid] = tid < nt ? min(max(perm_at(p.src, un.off + row0 + tid), 0), p.src.T - 1) : 0;
        if (!load_record<kThreadsS>(p.pv, un.a, p.m, rec, false)) continue;
        const int r = min(rec[0], min(p.pv.max_rank, p.ld_v));
        const int j0 = chunk * npc;
        if (j0 >= r || nt <= 0) continue;
        const int np = min(npc, r - j0);
        float d[4][4];
        shrink_core(p, tok, nt, rec, j0, np, kc0, kc1, sx, sa, red, d);
        if (warp == 0) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t * 8 >= np) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = g + 8 * h, j = t * 8 + 2 * q;
                    part[row * npc + j] = d[t][2 * h];
                    part[row * npc + j + 1] = d[t][2 * h + 1];
                }
            }
        }
        cl.sync();                                // every CTA's part is written
        const int own = nt > kpart ? (nt - 1 - kpart) / ks + 1 : 0;
        for (int i = tid; i < own * np; i += kThreadsS) {
            const int row = kpart + (i / np) * ks, j = i % np;
            if (((unsigned)un.pad >> (row0 + row)) & 1u) continue;
            float sum = 0.f;
            for (int qq = 0; qq < ks; ++qq) sum += *cl.map_shared_rank(part + row * npc + j, qq);
            p.v[(long long)tok[row] * p.ld_v + j0 + j] = sum;
        }
        cl.sync();                                // no CTA reuses or leaves part while a peer reads it
    }
}

// ---------------------------------------------------------------------------
// Shrink for pools with ranks above 32: 256 threads, one whole item (up to 32
// tokens) x one chunk of up to 64 ranks per CTA, so an item's rows share one
// pass over A_T and a rank-64 adapter needs one chunk.  Warp w takes rows
// 16 (w & 1) .. +16 and k 32 (w >> 1) .. +32 of every 128-wide stage; the
// four K-quarter partial sums are added at the end.  The item's x rows are
// requested before its page-table record arrives.
// ---------------------------------------------------------------------------
constexpr int kThreadsW = 256;
constexpr int kRowsW = kM;
constexpr int kStagesW = 4;

// One work entry of the wide shrink: item it, rank chunk by.
__device__ __forceinline__ void shrink_wide_item(const ShrinkParams &p, const Item &it, const int by, uint8_t *smem_raw) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int pitch = kKs + 8;                                        // bf16 per smem row
    const int npc = p.npc;
    __nv_bfloat16 *sx = reinterpret_cast<__nv_bfloat16 *>(smem_raw);     // [stages][32][pitch]
    __nv_bfloat16 *sa = sx + kStagesW * kRowsW * pitch;                   // [stages][npc][pitch]
    int *tok = reinterpret_cast<int *>(smem_raw + p.alias_bytes);         // [32]
    int *wtot = tok + kRowsW;                                            // [kThreadsW / 32 + 4]
    int *rec = wtot + kThreadsW / 32 + 4;                                // [rec_ints]
    float *red = reinterpret_cast<float *>(smem_raw);                    // [3][32][npc], after it ends

    const int nt = min(kRowsW, it.nt);
    if (it.a < 0 || nt <= 0) return;
    if (tid < kRowsW)
        tok[tid] = tid < nt ? min(max(p.src.plan ? perm_at(p.src, it.off + tid) : it.off + tid, 0), p.src.T - 1)
                            : 0;
    // x rows past the item stay zero
    for (int i = tid; i < kStagesW * kRowsW * (pitch / 8); i += kThreadsW)
        if ((i / (pitch / 8)) % kRowsW >= nt) reinterpret_cast<uint4 *>(sx)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    const int nk = p.h_in / kKs;
    // this thread's 16-byte copy slots, fixed for the whole K loop: element
    // tid + 256 k of the 32 rows x 16 chunks of x (k < 2) and of the npc (<= 64)
    // rows x 16 chunks of A_T (k < 4)
    const __nv_bfloat16 *xs[2], *as[4];
    uint32_t xd[2], ad[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = tid + k * kThreadsW, row = i >> 4, kv = i & 15;
        xs[k] = row < nt ? p.x + (long long)tok[row] * p.h_in + kv * 8 : nullptr;
        xd[k] = (uint32_t)(row * pitch + kv * 8);
    }
    auto issue_x = [&](int kc) {
        __nv_bfloat16 *dx = sx + (kc % kStagesW) * kRowsW * pitch;
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (xs[k]) cp_async16(dx + xd[k], xs[k] + kc * kKs);
    };
    // x of the first stages is on its way while the page-table record loads
#pragma unroll
    for (int kc = 0; kc < kStagesW - 1; ++kc)
        if (kc < nk) issue_x(kc);

    const bool ok = load_record<kThreadsW>(p.pv, it.a, p.m, rec, tid == 0 && by == 0);
    bool skip = !ok;
    if (ok && p.tc_min_rows > 0 && !p.src.plan && it.pad >= p.tc_min_rows && rec[0] >= kShrinkTcSegMinRank &&
        rec[0] <= kFuseMaxRank && rec[0] <= p.ld_v)
        skip = true;                             // the tensor-core shrink computed this segment
    const int r = ok ? min(rec[0], min(p.pv.max_rank, p.ld_v)) : 0;
    const int j0 = by * npc;
    if (skip || j0 >= r) {
        cp_commit();       // nothing may be in flight into shared memory when the CTA exits
        cp_wait<0>();
        return;
    }
    const int np = min(npc, r - j0);
    const int npad = (np + 15) & ~15;
    // A rows np .. npc-1 receive no copies: zero them in every stage
    for (int i = tid; i < kStagesW * npc * (pitch / 8); i += kThreadsW)
        if ((i / (pitch / 8)) % npc >= np) reinterpret_cast<uint4 *>(sa)[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = tid + k * kThreadsW, row = i >> 4, kv = i & 15;
        as[k] = row < np ? page_row<__nv_bfloat16>(p.pv, clamp_page(p.pv, rec[kRecHeader + j0 + row])) + kv * 8 : nullptr;
        ad[k] = (uint32_t)(row * pitch + kv * 8);
    }
    auto issue_a = [&](int kc) {
        __nv_bfloat16 *da = sa + (kc % kStagesW) * npc * pitch;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (as[k]) cp_async16(da + ad[k], as[k] + kc * kKs);
    };
#pragma unroll
    for (int kc = 0; kc < kStagesW - 1; ++kc)
        if (kc < nk) issue_a(kc);
    cp_commit();            // one group holds stages 0 .. kStagesW-2

    const int mh = warp & 1, kq = warp >> 1;
    const int g = lane >> 2, q = lane & 3;
    float d[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[t][e] = 0.f;
    for (int kc = 0; kc < nk; ++kc) {
        if (kc == 0) cp_wait<0>();
        else cp_wait<kStagesW - 2>();
        __syncthreads();
        if (kc + kStagesW - 1 < nk) {
            issue_x(kc + kStagesW - 1);
            issue_a(kc + kStagesW - 1);
        }
        cp_commit();
        const int st = kc % kStagesW;
        const __nv_bfloat16 *bx = sx + st * kRowsW * pitch;
        const __nv_bfloat16 *ba = sa + st * npc * pitch;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {                   // this warp's quarter of the stage
            const int k = kq * 32 + ks * 16;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(bx + (mh * 16 + (lane & 15)) * pitch + k + (lane >> 4) * 8, a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
                if (t * 8 >= npad) break;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(ba + (t * 8 + (lane & 7) + ((lane >> 4) << 3)) * pitch + k + ((lane >> 3) & 1) * 8, b0, b1,
                        b2, b3);
                mma16816(d[t], a0, a1, a2, a3, b0, b1);
                mma16816(d[t + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    cp_wait<0>();
    __syncthreads();        // the pipeline buffers are free: red aliases them
    // add the four K-quarter partials and write v
    if (kq > 0) {
        float *rw = red + (kq - 1) * kRowsW * npc;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t * 8 >= npad) break;
            const int r0 = mh * 16 + g;
            rw[r0 * npc + t * 8 + 2 * q] = d[t][0];
            rw[r0 * npc + t * 8 + 2 * q + 1] = d[t][1];
            rw[(r0 + 8) * npc + t * 8 + 2 * q] = d[t][2];
            rw[(r0 + 8) * npc + t * 8 + 2 * q + 1] = d[t][3];
        }
    }
    __syncthreads();
    if (kq == 0) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t * 8 >= npad) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mh * 16 + g + 8 * h;
                const int j = t * 8 + 2 * q;
                if (row >= nt) continue;
                float v0 = d[t][2 * h], v1 = d[t][2 * h + 1];
#pragma unroll
                for (int w = 0; w < 3; ++w) {
                    v0 += red[w * kRowsW * npc + row * npc + j];
                    v1 += red[w * kRowsW * npc + row * npc + j + 1];
                }
                float *vrow = p.v + (long long)tok[row] * p.ld_v + j0;
                if (j < np) vrow[j] = v0;
                if (j + 1 < np) vrow[j + 1] = v1;
            }
        }
    }
}

// Persistent over (item, rank chunk) work entries: CTA c takes c, c + G, ...
__global__ void __launch_bounds__(kThreadsW, 2) sgmv_shrink_wide_kernel(ShrinkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    if (blockIdx.x == 0 && !p.src.plan) check_segments(p.src.seg_starts, p.src.S, p.src.T, p.pv.status);
    // a segment table's chunk scan, made once (it is the same for every item), after the rest
    int *wtot = reinterpret_cast<int *>(smem_raw + p.alias_bytes) + kRowsW;
    int *scan = wtot + kThreadsW / 32 + 4 + p.pv.rec_ints;
    const int total = p.src.plan ? 0 : segment_scan<kThreadsW>(p.src.seg_starts, p.src.S, p.src.T, scan, wtot);
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
        __syncthreads();                          // the previous entry's readers of shared memory are done
        const int idx = w / p.n_chunks;
        const Item it = p.src.plan ? plan_items(p.src.plan, p.src.T)[idx]
                                   : segment_lookup<kThreadsW>(p.src.seg_starts, p.src.seg_adapter, p.src.S, p.src.T,
                                                               idx, scan, total, wtot);
        shrink_wide_item(p, it, w % p.n_chunks, smem_raw);
    }
}

// ---------------------------------------------------------------------------
// Expand: 128 threads, unit = (item, up to bpu <= kMaxBlocksPerUnit column blocks of
// kNb).  warp w: rows 16*(w & 1) .. +16, columns 64*(w >> 1) .. +64 of the
// block.  y tiles and B chunks stream through a kStagesE-stage pipeline; y is read
// and written with coalesced 16-byte accesses staged in shared memory.
// ---------------------------------------------------------------------------
constexpr int kThreadsE = 128;

struct ExpandParams {
    PoolView pv;
    ItemSource src;
    int m, h_out;
    int kpc;       // ranks per pass: max_rank rounded up to 16, at most 64
    const float *v;
    int ld_v;
    __nv_bfloat16 *y;
    int ncg;       // column groups per item
    int n_work;    // segment tables: items (upper bound) x column groups
    int bpu;       // column blocks per unit (1 .. kMaxBlocksPerUnit)
    const Unit *units;    // unit kernel: the plan's expand units (count plan[3])
    int max_units;        // unit kernel: the plan's room for expand units
};

// Rows of item `it` outside `fused` x column blocks b_first .. b_first + nb_req - 1.
// report: this CTA flags an invalid adapter.
__device__ __forceinline__ void expand_unit(const ExpandParams &p, const Item &it, unsigned fused, int b_first,
                                            int nb_req, bool report, uint8_t *smem_raw) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int yp = kNb + 8;                  // bf16 per smem row of y and B tiles
    const int kpc = p.kpc, vp = p.kpc + 8;
    __nv_bfloat16 *sy = reinterpret_cast<__nv_bfloat16 *>(smem_raw);      // [stages][kM][yp]
    __nv_bfloat16 *sb = sy + kStagesE * kM * yp;                          // [stages][kpc][yp]
    __nv_bfloat16 *svh = sb + kStagesE * kpc * yp;                        // [kM][vp]
    __nv_bfloat16 *svl = svh + kM * vp;                                   // [kM][vp]
    int *tok = reinterpret_cast<int *>(svl + kM * vp);                    // [kM]
    int *wtot = tok + kM;                                                 // [8]
    int *rec = wtot + 8;

    const unsigned all = it.nt >= 32 ? 0xffffffffu : ((1u << it.nt) - 1u);
    if ((fused & all) == all) return;            // the GEMM added every row's term
    if (it.a >= p.pv.max_adapters) {
        if (tid == 0 && report) flag(p.pv.status, LORA_DEV_BAD_ADAPTER);
        return;
    }
    // the record and the item's tokens load together
    for (int i = tid; i < p.pv.rec_ints; i += kThreadsE)
        rec[i] = p.pv.table[((long long)it.a * p.pv.n_matrices + p.m) * p.pv.rec_ints + i];
    if (warp == 0) {   // the item's tokens, minus rows whose term the GEMM already added (one per lane)
        const bool keep = lane < it.nt && !((fused >> lane) & 1u);
        const int t = keep ? min(max(p.src.plan ? perm_at(p.src, it.off + lane) : it.off + lane, 0),
                                 p.src.T - 1)
                           : 0;
        const unsigned kept = __ballot_sync(0xffffffffu, keep);
        const int n = __popc(kept);
        if (keep) tok[__popc(kept & ((1u << lane) - 1u))] = t;
        if (lane >= n) tok[lane] = 0;
        if (lane == 0) wtot[0] = n;
    }
    __syncthreads();
    if (rec[0] < 0) {
        if (tid == 0 && report) flag(p.pv.status, LORA_DEV_BAD_ADAPTER);
        return;
    }
    const int nt = wtot[0];
    if (nt == 0) return;
    const int r_rec = min(rec[0], p.pv.max_rank);
    const int r = min(r_rec, p.ld_v);
    const float scale = __int_as_float(rec[1]);
    const int nb_total = (p.h_out + kNb - 1) / kNb;
    const int nb = min(nb_req, nb_total - b_first);
    if (nb <= 0 || r <= 0) return;
    const int mg = warp & 1, nh = warp >> 1;
    const int g = lane >> 2, q = lane & 3;

    const int passes = (r + kpc - 1) / kpc;
    if (nb == 1 && passes > 1 && passes <= kStagesE && 2 * vp <= yp) {
        // One column block and several rank passes (the costly units of high-rank
        // adapters): y is read and written once, the B chunks of every pass are
        // copied at once into the ring's B slots (pass j -> stage j), the scaled v
        // of pass 0 goes to svh/svl and that of pass j >= 1 to stage j's unused y
        // slot (both parts fit there: 2 vp <= yp), and the passes' products
        // accumulate in registers before the one rounding of y.
        const int n0 = b_first * kNb;
        const int ncv = min(kNb, p.h_out - n0) / 8;
        for (int i = tid; i < nt * 16; i += kThreadsE) {
            const int row = i >> 4, cv = i & 15;
            if (cv < ncv) cp_async16(sy + row * yp + cv * 8, p.y + (long long)tok[row] * p.h_out + n0 + cv * 8);
        }
        for (int j = 0; j < passes; ++j) {
            const int jj0 = j * kpc, rn = min(kpc, r - jj0), kpad = (rn + 15) & ~15;
            __nv_bfloat16 *db = sb + j * kpc * yp;
            for (int i = tid; i < kpad * 16; i += kThreadsE) {
                const int row = i >> 4, cv = i & 15;
                if (row < rn) {
                    if (cv < ncv)
                        cp_async16(db + row * yp + cv * 8,
                                   page_row<__nv_bfloat16>(p.pv, clamp_page(p.pv, rec[kRecHeader + r_rec + jj0 + row])) +
                                       n0 + cv * 8);
                } else {
                    *reinterpret_cast<uint4 *>(db + row * yp + cv * 8) = make_uint4(0, 0, 0, 0);   // MMA K padding
                }
            }
        }
        cp_commit();
        const bool vec = (p.ld_v & 3) == 0;
        for (int j = 0; j < passes; ++j) {
            const int jj0 = j * kpc, rn = min(kpc, r - jj0), kpad = (rn + 15) & ~15;
            __nv_bfloat16 *vh = j == 0 ? svh : sy + j * kM * yp;
            __nv_bfloat16 *vl = j == 0 ? svl : vh + kM * vp;
            for (int i = tid; i < kM * (kpad >> 2); i += kThreadsE) {
                const int row = i / (kpad >> 2), jl = 4 * (i % (kpad >> 2));
                float e4[4] = {0.f, 0.f, 0.f, 0.f};
                if (row < nt && jl < rn) {
                    const float *src = p.v + (long long)tok[row] * p.ld_v + jj0 + jl;
                    if (vec) {       // ld_v % 4 == 0 and jj0 % 4 == 0: the group stays in the row
                        const float4 f = *reinterpret_cast<const float4 *>(src);
                        e4[0] = f.x; e4[1] = f.y; e4[2] = f.z; e4[3] = f.w;
                    } else {
                        for (int e = 0; e < 4; ++e)
                            if (jl + e < rn) e4[e] = src[e];
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float val = jl + e < rn ? scale * e4[e] : 0.f;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(val);
                    vh[row * vp + jl + e] = hi;
                    vl[row * vp + jl + e] = __float2bfloat16_rn(val - __bfloat162float(hi));
                }
            }
        }
        cp_wait<0>();
        __syncthreads();
        float d[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[t][e] = 0.f;
        for (int j = 0; j < passes; ++j) {
            const int rn = min(kpc, r - j * kpc), kpad = (rn + 15) & ~15;
            const __nv_bfloat16 *vh = j == 0 ? svh : sy + j * kM * yp;
            const __nv_bfloat16 *vl = j == 0 ? svl : vh + kM * vp;
            const __nv_bfloat16 *tb = sb + j * kpc * yp;
            for (int kk = 0; kk < kpad; kk += 16) {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                ldsm_x4(vh + (mg * 16 + (lane & 15)) * vp + kk + (lane >> 4) * 8, h0, h1, h2, h3);
                ldsm_x4(vl + (mg * 16 + (lane & 15)) * vp + kk + (lane >> 4) * 8, l0, l1, l2, l3);
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(tb + (kk + (lane & 7) + ((lane >> 3) & 1) * 8) * yp + nh * 64 + (t + (lane >> 4)) * 8,
                              b0, b1, b2, b3);
                    mma16816(d[t], h0, h1, h2, h3, b0, b1);
                    mma16816(d[t], l0, l1, l2, l3, b0, b1);
                    mma16816(d[t + 1], h0, h1, h2, h3, b2, b3);
                    mma16816(d[t + 1], l0, l1, l2, l3, b2, b3);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mg * 16 + g + 8 * h;
                __nv_bfloat162 *yy = reinterpret_cast<__nv_bfloat162 *>(sy + row * yp + nh * 64 + t * 8 + 2 * q);
                const float2 f = __bfloat1622float2(*yy);
                *yy = __floats2bfloat162_rn(f.x + d[t][2 * h], f.y + d[t][2 * h + 1]);
            }
        __syncthreads();
        for (int i = tid; i < nt * (kNb / 8); i += kThreadsE) {
            const int row = i >> 4, cv = i & 15;
            if (cv < ncv)
                *reinterpret_cast<uint4 *>(p.y + (long long)tok[row] * p.h_out + n0 + cv * 8) =
                    *reinterpret_cast<const uint4 *>(sy + row * yp + cv * 8);
        }
        __syncthreads();   // shared memory is read before the next unit reuses it
        return;
    }

    // ranks in passes of kpc; each pass streams the unit's y blocks once
    for (int j0 = 0; j0 < r; j0 += kpc) {
        const int rn = min(kpc, r - j0);
        const int kpad = (rn + 15) & ~15;
        // this thread's 16-byte copy slots for the pass (fixed across column blocks):
        // element tid + 128 k of the 32 rows x 16 chunks of y (k < 4) and of the
        // kpc rows x 16 chunks of B (k < 8)
        const __nv_bfloat16 *ysrc[4], *bsrc[8];
        uint32_t ydst[4], bdst[8];
        int ycv[4], bcv[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = tid + k * kThreadsE, row = i >> 4, cv = i & 15;
            ysrc[k] = row < nt ? p.y + (long long)tok[row] * p.h_out + cv * 8 : nullptr;
            ydst[k] = (uint32_t)(row * yp + cv * 8);
            ycv[k] = cv;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * kThreadsE, row = i >> 4, cv = i & 15;
            bsrc[k] = row < rn ? page_row<__nv_bfloat16>(p.pv, clamp_page(p.pv, rec[kRecHeader + r_rec + j0 + row])) +
                                     cv * 8
                               : nullptr;
            bdst[k] = (uint32_t)(row * yp + cv * 8);
            bcv[k] = cv;
        }
        // B rows rn .. kpad-1 (MMA K padding) get no copies in this pass: zero them in every stage
        for (int i = tid; i < kStagesE * (kpad - rn) * (kNb / 8); i += kThreadsE) {
            const int st = i / ((kpad - rn) * (kNb / 8)), rem = i % ((kpad - rn) * (kNb / 8));
            *reinterpret_cast<uint4 *>(sb + st * kpc * yp + (rn + (rem >> 4)) * yp + (rem & 15) * 8) =
                make_uint4(0, 0, 0, 0);
        }
        auto issue = [&](int bi) {
            const int st = bi % kStagesE;
            const int n0 = (b_first + bi) * kNb;
            const int ncv = min(kNb, p.h_out - n0) / 8;
            __nv_bfloat16 *dy = sy + st * kM * yp;
            __nv_bfloat16 *db = sb + st * kpc * yp;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (ysrc[k] && ycv[k] < ncv) cp_async16(dy + ydst[k], ysrc[k] + n0);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (bsrc[k] && bcv[k] < ncv) cp_async16(db + bdst[k], bsrc[k] + n0);
        };
#pragma unroll
        for (int bi = 0; bi < kStagesE - 1; ++bi) {
            if (bi < nb) issue(bi);
            cp_commit();
        }
        // v of the item's tokens for this pass, scaled, as two bf16 parts (rows past the item are
        // zero).  Groups of 4 ranks; a thread's loads are all issued before any is used.
        {
            constexpr int kMaxG = kM * 64 / 4 / kThreadsE;          // groups per thread at kpc = 64
            const int g4 = kpad >> 2, total = kM * g4;
            const bool vec = (p.ld_v & 3) == 0;
            float4 f[kMaxG];
#pragma unroll
            for (int u = 0; u < kMaxG; ++u) {
                const int i = tid + u * kThreadsE, row = i / max(g4, 1), j = 4 * (i % max(g4, 1));
                f[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < total && row < nt && j < rn) {
                    const float *src = p.v + (long long)tok[row] * p.ld_v + j0 + j;
                    if (vec) {       // ld_v % 4 == 0 and j0 % 4 == 0: the group stays in the row
                        f[u] = *reinterpret_cast<const float4 *>(src);
                    } else {
                        f[u].x = src[0];
                        if (j + 1 < rn) f[u].y = src[1];
                        if (j + 2 < rn) f[u].z = src[2];
                        if (j + 3 < rn) f[u].w = src[3];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kMaxG; ++u) {
                const int i = tid + u * kThreadsE, row = i / max(g4, 1), j = 4 * (i % max(g4, 1));
                if (i >= total) continue;
                const float e4[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float val = j + e < rn ? scale * e4[e] : 0.f;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(val);
                    svh[row * vp + j + e] = hi;
                    svl[row * vp + j + e] = __float2bfloat16_rn(val - __bfloat162float(hi));
                }
            }
        }

        for (int bi = 0; bi < nb; ++bi) {
            cp_wait<kStagesE - 2>();
            __syncthreads();
            if (bi + kStagesE - 1 < nb) issue(bi + kStagesE - 1);
            cp_commit();
            const int st = bi % kStagesE;
            __nv_bfloat16 *ty = sy + st * kM * yp;
            const __nv_bfloat16 *tb = sb + st * kpc * yp;
            float d[8][4];
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[t][e] = 0.f;
            for (int kk = 0; kk < kpad; kk += 16) {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                ldsm_x4(svh + (mg * 16 + (lane & 15)) * vp + kk + (lane >> 4) * 8, h0, h1, h2, h3);
                ldsm_x4(svl + (mg * 16 + (lane & 15)) * vp + kk + (lane >> 4) * 8, l0, l1, l2, l3);
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(tb + (kk + (lane & 7) + ((lane >> 3) & 1) * 8) * yp + nh * 64 + (t + (lane >> 4)) * 8,
                              b0, b1, b2, b3);
                    mma16816(d[t], h0, h1, h2, h3, b0, b1);
                    mma16816(d[t], l0, l1, l2, l3, b0, b1);
                    mma16816(d[t + 1], h0, h1, h2, h3, b2, b3);
                    mma16816(d[t + 1], l0, l1, l2, l3, b2, b3);
                }
            }
            // y tile += delta in shared memory, then coalesced stores
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = mg * 16 + g + 8 * h;
                    __nv_bfloat162 *yy =
                        reinterpret_cast<__nv_bfloat162 *>(ty + row * yp + nh * 64 + t * 8 + 2 * q);
                    const float2 f = __bfloat1622float2(*yy);
                    *yy = __floats2bfloat162_rn(f.x + d[t][2 * h], f.y + d[t][2 * h + 1]);
                }
            __syncthreads();
            const int n0 = (b_first + bi) * kNb;
            const int ncv = min(kNb, p.h_out - n0) / 8;
            for (int i = tid; i < nt * (kNb / 8); i += kThreadsE) {
                const int row = i >> 4, cv = i & 15;
                if (cv < ncv)
                    *reinterpret_cast<uint4 *>(p.y + (long long)tok[row] * p.h_out + n0 + cv * 8) =
                        *reinterpret_cast<const uint4 *>(ty + row * yp + cv * 8);
            }
        }
        cp_wait<0>();
        __syncthreads();   // this pass's stores are issued before the next pass reloads y
    }
}

__global__ void __launch_bounds__(kThreadsE, 4) sgmv_expand_kernel(ExpandParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int kpc = p.kpc, vp = p.kpc + 8;
    constexpr int yp = kNb + 8;
    int *wtot = reinterpret_cast<int *>(reinterpret_cast<__nv_bfloat16 *>(smem_raw) + kStagesE * kM * yp +
                                        kStagesE * kpc * yp + 2 * kM * vp) + kM;
    int *scan = wtot + 8 + p.pv.rec_ints;
    if (blockIdx.x == 0 && !p.src.plan) check_segments(p.src.seg_starts, p.src.S, p.src.T, p.pv.status);
    // persistent: CTA c takes work c, c + G, ... (work = item x column group); a
    // segment table's chunk scan is made once and kept (it is the same for every item)
    const int total = p.src.plan ? 0 : segment_scan<kThreadsE>(p.src.seg_starts, p.src.S, p.src.T, scan, wtot);
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
        __syncthreads();                          // the previous unit's readers of shared memory are done
        const int cg = w % p.ncg;
        const Item it = p.src.plan ? plan_items(p.src.plan, p.src.T)[w / p.ncg]
                                   : segment_lookup<kThreadsE>(p.src.seg_starts, p.src.seg_adapter, p.src.S, p.src.T,
                                                               w / p.ncg, scan, total, wtot);
        if (it.a < 0 || it.nt <= 0) continue;
        expand_unit(p, it, 0u, cg * p.bpu, p.bpu, cg == 0, smem_raw);
    }
}

// Layer plans: persistent CTAs walk the plan's expand units (costly ones first,
// snake order: CTA c takes units c, 2G - 1 - c, 2G + c, ...).
__global__ void __launch_bounds__(kThreadsE, 4) sgmv_expand_units_kernel(ExpandParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int n_units = min(max(p.src.plan[3], 0), p.max_units);
    const int G = gridDim.x, c = blockIdx.x;
    for (int k = 0;; ++k) {
        const int u = k * G + ((k & 1) ? G - 1 - c : c);
        if (u >= n_units) break;
        const Unit un = p.units[u];
        __syncthreads();                          // the previous unit's readers of shared memory are done
        const Item it{un.a, un.off, un.info & 63, un.pad};
        expand_unit(p, it, (unsigned)un.pad, (int)((unsigned)un.info >> 10), (un.info >> 6) & 15, false, smem_raw);
    }
}

// The units kernel's ranks per pass, shared memory and grid (one CTA per
// resident slot: the SMs times the CTAs one SM holds); grid 0 on error.
int expand_units_kpc(const lora_pool *pool) { return std::min(32, (pool->max_rank + 15) / 16 * 16); }
size_t expand_units_smem(const lora_pool *pool) {
    const int kpc = expand_units_kpc(pool);
    return (size_t)kStagesE * (kM + kpc) * (kNb + 8) * 2 + (size_t)2 * kM * (kpc + 8) * 2 +
           (size_t)(kM + 8 + pool->view().rec_ints) * 4 + 16;
}
int expand_units_grid(const lora_pool *pool) {
    int occ = 0;
    if (smem_optin(reinterpret_cast<const void *>(sgmv_expand_units_kernel), expand_units_smem(pool), kThreadsE, &occ))
        return 0;
    return num_sms() * std::max(1, occ);
}

// Upper bound on items: every non-empty segment (or adapter) has at least
// one chunk, and the chunks together cover T tokens.
int item_bound(int groups, int T) { return std::min(groups, T) + (T + kM - 1) / kM; }

}  // namespace

bool sgmv_shrink_ok(const lora_pool *pool, int h_in, int S) {
    return pool->dtype == LORA_BF16 && h_in % kKs == 0 && S <= kMaxS;
}

bool sgmv_expand_ok(const lora_pool *pool, int h_out, int S) {
    return pool->dtype == LORA_BF16 && h_out % 8 == 0 && S <= kMaxS;
}

// Plan layout in ints from its start: header [n_items, n_work, n_shrink_units,
// n_expand_units], perm[T], items, M-tile adapters, then (layer plans) shrink
// and expand units.  Every array starts 16-byte aligned.
struct PlanLayout {
    int max_items, max_su, max_eu;
    size_t tiles, su, eu, total;   // offsets in ints; total bytes
};

// Ranks per shrink CTA of the 128-thread kernels.
static int shrink_npc(const lora_pool *pool) { return std::min(32, (pool->max_rank + 15) / 16 * 16); }

static PlanLayout plan_layout(const lora_pool *pool, int matrix, int T) {
    PlanLayout L;
    const int n_ids = std::max(1, pool->mat_n_ids[matrix]);
    const int n_tiles = (T + kTileRows - 1) / kTileRows;
    const int item_ints = (int)(sizeof(Item) / sizeof(int));
    L.max_items = item_bound(n_ids, T);
    L.max_su = L.max_items * 2 * ((pool->max_rank + shrink_npc(pool) - 1) / shrink_npc(pool));
    L.max_eu = L.max_items * ((std::max(0, pool->mat_h_out[matrix]) + kNb - 1) / kNb);
    L.tiles = 4 + (size_t)((T + 3) & ~3) + (size_t)L.max_items * item_ints;
    L.su = L.tiles + (size_t)((n_tiles + 3) & ~3);
    L.eu = L.su + (size_t)L.max_su * item_ints;
    L.total = (L.eu + (size_t)L.max_eu * item_ints) * 4 + 64;
    return L;
}

size_t sgmv_plan_bytes(const lora_pool *pool, int matrix, int T) { return plan_layout(pool, matrix, T).total; }

int *sgmv_plan_tiles(const lora_pool *pool, int matrix, int T, int *plan) {
    return plan + plan_layout(pool, matrix, T).tiles;
}


// Shared memory of the plan kernel: the counting-sort area, the scan words and,
// for layer plans, the unit-building arrays.
static size_t plan_smem(const lora_pool *pool, int matrix, int S, int T, bool units, int *body) {
    const int n_ids = pool->mat_n_ids[matrix];
    const int n_tiles = (T + kTileRows - 1) / kTileRows;
    *body = (3 * n_ids + 3 * S + 1 + (units ? n_ids + T + n_tiles : 0) + 3) & ~3;
    size_t ints = (size_t)*body + ((kPlanThreads / 32 + 2 + 3) & ~3);
    if (units) ints += (size_t)9 * plan_layout(pool, matrix, T).max_items + 4 * (kPlanThreads / 32 + 1);
    return ints * 4;
}

bool sgmv_plan_ok(const lora_pool *pool, int matrix, int S, int T, bool units) {
    int body;
    return pool->mat_n_ids[matrix] > 0 && S <= kMaxS && plan_smem(pool, matrix, S, T, units, &body) <= 160 * 1024;
}

int launch_sgmv_plan(const lora_pool *pool, int matrix, const int *seg_starts, const int *seg_adapter, int S, int T,
                     int *plan, cudaStream_t st, bool units) {
    const PlanLayout L = plan_layout(pool, matrix, T);
    PlanParams p;
    p.seg_starts = seg_starts;
    p.seg_adapter = seg_adapter;
    p.S = S;
    p.T = T;
    p.n_ids = pool->mat_n_ids[matrix];
    p.status = pool->d_status;
    p.plan = plan;
    p.max_items = L.max_items;
    p.pv = pool->view();
    p.m = matrix;
    p.units = units;
    p.n_tiles = (T + kTileRows - 1) / kTileRows;
    p.su = units ? reinterpret_cast<Unit *>(plan + L.su) : nullptr;
    p.eu = units ? reinterpret_cast<Unit *>(plan + L.eu) : nullptr;
    p.npc_s = shrink_npc(pool);
    p.nb_total = (std::max(0, pool->mat_h_out[matrix]) + kNb - 1) / kNb;
    p.e_ctas = units ? expand_units_grid(pool) : 1;
    if (units && p.e_ctas <= 0) return LORA_ERR_CUDA;
    p.rank_cap = pool->max_rank;
    const size_t smem = plan_smem(pool, matrix, S, T, units, &p.body);
    if (smem_optin(reinterpret_cast<const void *>(sgmv_plan_kernel), smem)) return LORA_ERR_CUDA;
    sgmv_plan_kernel<<<1, kPlanThreads, smem, st>>>(p);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int launch_sgmv_shrink(const lora_pool *pool, int matrix, int h_in, const void *x, float *v, int ld_v,
                       const int *seg_starts, const int *seg_adapter, int S, int T, const int *plan,
                       cudaStream_t st, bool skip_fused, int tc_min_rows) {
    ShrinkParams p;
    p.tc_min_rows = tc_min_rows;
    p.pv = pool->view();
    p.src = ItemSource{seg_starts, seg_adapter, S, T, plan};
    p.m = matrix;
    p.h_in = h_in;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.v = v;
    p.ld_v = ld_v;
    const int groups = plan ? std::max(1, pool->mat_n_ids[matrix]) : S;
    if (skip_fused && plan) {
        // layer plan: persistent clusters over the plan's shrink units, K split over the cluster
        p.npc = shrink_npc(pool);
        p.alias_bytes = 0;
        p.units = reinterpret_cast<const Unit *>(plan + plan_layout(pool, matrix, T).su);
        p.max_units = plan_layout(pool, matrix, T).max_su;
        const size_t smem = (size_t)kStagesS * (kRowsS + p.npc) * (kKs + 8) * 2 + (size_t)4 * 16 * p.npc * 4 +
                            (size_t)(kRowsS + p.pv.rec_ints) * 4 + 16;
        int occ = 0;
        if (smem_optin(reinterpret_cast<const void *>(sgmv_shrink_units_kernel), smem, kThreadsS, &occ))
            return LORA_ERR_CUDA;
        const int nk = h_in / kKs;
        const int ks = nk >= 16 ? 2 : 1;       // measured: 2 beats 1 and 4 (4 leaves too few clusters)
        const int clusters = std::max(1, num_sms() * std::max(1, occ) / ks);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ks, clusters, 1);
        cfg.blockDim = dim3(kThreadsS, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ks;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, sgmv_shrink_units_kernel, p);
        count_launch();
        return cuda_status(e != cudaSuccess ? e : cudaGetLastError());
    }
    p.units = nullptr;
    if (pool->max_rank > 32 && !plan) {
        // ranks above 32 in a segment table: whole items and 64-rank chunks per CTA
        p.npc = std::min(64, (pool->max_rank + 15) / 16 * 16);
        constexpr int pitch = kKs + 8;
        const size_t pipe = (size_t)kStagesW * (kRowsW + p.npc) * pitch * 2;
        const size_t alias = (std::max(pipe, (size_t)3 * kRowsW * p.npc * 4) + 15) & ~(size_t)15;
        p.alias_bytes = (int)alias;
        const size_t smem_w = alias + (size_t)(kRowsW + kThreadsW / 32 + 4 + p.pv.rec_ints + S + 1) * 4;
        int occ = 0;
        if (smem_optin(reinterpret_cast<const void *>(sgmv_shrink_wide_kernel), smem_w, kThreadsW, &occ))
            return LORA_ERR_CUDA;
        p.n_chunks = (pool->max_rank + p.npc - 1) / p.npc;
        p.n_work = item_bound(groups, T) * p.n_chunks;
        const int grid_w = std::max(1, std::min(p.n_work, num_sms() * std::max(1, occ)));
        sgmv_shrink_wide_kernel<<<grid_w, kThreadsW, smem_w, st>>>(p);
        count_launch();
        return cuda_status(cudaGetLastError());
    }
    p.npc = std::min(32, (pool->max_rank + 15) / 16 * 16);
    p.alias_bytes = 0;
    const size_t smem = (size_t)kStagesS * (kRowsS + p.npc) * (kKs + 8) * 2 + (size_t)3 * 16 * p.npc * 4 +
                        (size_t)(kRowsS + 8 + p.pv.rec_ints + (plan ? 0 : S + 1)) * 4 + 16;
    if (smem_optin(reinterpret_cast<const void *>(sgmv_shrink_kernel), smem)) return LORA_ERR_CUDA;
    const dim3 grid(item_bound(groups, T), (pool->max_rank + p.npc - 1) / p.npc, kM / kRowsS);
    sgmv_shrink_kernel<<<grid, kThreadsS, smem, st>>>(p);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int launch_sgmv_expand(const lora_pool *pool, int matrix, int h_out, const float *v, int ld_v, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T, const int *plan,
                       cudaStream_t st, const int *tile_ad) {
    ExpandParams p;
    p.pv = pool->view();
    p.src = ItemSource{seg_starts, seg_adapter, S, T, plan};
    p.m = matrix;
    p.h_out = h_out;
    p.kpc = std::min(64, (pool->max_rank + 15) / 16 * 16);
    p.v = v;
    p.ld_v = ld_v;
    p.y = static_cast<__nv_bfloat16 *>(y);
    const int nb_total = (h_out + kNb - 1) / kNb;
    // wide units amortise each unit's start-up latency (measured: fewer, longer
    // CTAs win even when the grid is below the resident-CTA count)
    p.bpu = kMaxBlocksPerUnit;
    p.ncg = (nb_total + p.bpu - 1) / p.bpu;
    const size_t smem = (size_t)kStagesE * (kM + p.kpc) * (kNb + 8) * 2 + (size_t)2 * kM * (p.kpc + 8) * 2 +
                        (size_t)(kM + 8 + p.pv.rec_ints + (plan ? 0 : S + 1)) * 4 + 16;
    if (smem_optin(reinterpret_cast<const void *>(sgmv_expand_kernel), smem)) return LORA_ERR_CUDA;
    if (tile_ad && plan) {
        // layer plan: persistent CTAs over the plan's expand units, in passes of at most 32
        // ranks (a smaller CTA, so more fit per SM; only units of ranks above 32 take more passes)
        p.units = reinterpret_cast<const Unit *>(plan + plan_layout(pool, matrix, T).eu);
        p.max_units = plan_layout(pool, matrix, T).max_eu;
        p.kpc = expand_units_kpc(pool);
        const int grid = expand_units_grid(pool);
        if (grid <= 0) return LORA_ERR_CUDA;
        sgmv_expand_units_kernel<<<grid, kThreadsE, expand_units_smem(pool), st>>>(p);
        count_launch();
        return cuda_status(cudaGetLastError());
    }
    p.units = nullptr;
    const int groups = plan ? std::max(1, pool->mat_n_ids[matrix]) : S;
    p.n_work = item_bound(groups, T) * p.ncg;
    int occ = 0;
    if (smem_optin(reinterpret_cast<const void *>(sgmv_expand_kernel), smem, kThreadsE, &occ)) return LORA_ERR_CUDA;
    const int grid = std::max(1, std::min(p.n_work, num_sms() * std::max(1, occ)));
    sgmv_expand_kernel<<<grid, kThreadsE, smem, st>>>(p);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace lora
