// BGMV for decode batches: every decode token gathers the low-rank factors of
// its own adapter ("Multi-LoRA Serving", section "The kernel trick: gather, do
// not merge"), with per-adapter ranks as in S-LoRA's MBGMV (slide 10).
//
//   y[t][n] += s_a * sum_j (sum_k x[t][k] * A_T_a[j][k]) * B_a[j][n],  a = token_adapter[t]
//
// Design (GB300).  Tokens are grouped by adapter inside the kernel, so every
// adapter page is read from HBM once per launch however many tokens use it.
// A work item is one adapter and up to kTok of its tokens; one thread-block
// cluster of kC CTAs serves one item.  CTA c of the cluster owns the c-th
// slice of h_in for the shrink and the c-th slice of h_out for the expand:
//   1. every CTA loads the id list and (for the adapter its cluster index
//      names) the page-table record, and starts 16-byte asynchronous copies
//      of its slice of that adapter's A_T and B pages into shared memory;
//   2. the item's token list is the ordered set of tokens with that id;
//      every CTA of the cluster derives it from the same ids and table, so
//      all take the same branches (the exchange waits are bounded anyway);
//   3. x slices of the item's tokens arrive by 16-byte async copies; each
//      CTA forms partial v over its h_in slice on the tensor cores
//      (mma.sync m16n8k16, bf16 -> fp32: 16 tokens x 16 ranks x 64 k per
//      warp), the partials are summed across the cluster through DSMEM, and
//      each CTA applies y += s * v . B on its h_out slice, again on the
//      tensor cores, with v split into a bf16 high part and a bf16 residual
//      so the product keeps fp32-level accuracy.
// The per-cluster products (16 x 16 x 512 and 16 x 512 x 16) are below the
// 64-row minimum of tcgen05.mma, so the warp-level MMA is the right unit
// here; the kernel is bound by HBM traffic and latency, not by MMA rate.
// Adapters with more than kTok tokens in the batch get extra items
// ("overflow" clusters) located by an in-kernel histogram and scan.  Ranks
// above kJ are processed kJ rows at a time.
//
// Page ids read from the table are clamped into the pool and every loop is
// bounded, so a corrupt table can give wrong numbers but never an
// out-of-bounds access or a barrier that some CTA skips.
#include <cooperative_groups.h>

#include <algorithm>

#include "internal.cuh"

namespace cg = cooperative_groups;

namespace lora {
namespace {

constexpr int kC = 8;           // CTAs per cluster
constexpr int kTok = 16;        // tokens per work item (MMA M)
constexpr int kJ = 16;          // ranks per chunk (MMA N of the shrink, K of the expand)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxT = 2048;     // largest batch this path takes
constexpr int kMaxIds = 4096;   // largest adapter-id range this path takes
constexpr int kMaxSliceOut = 512;
constexpr int kMaxSliceIn = 1024;
constexpr int kVPitch = 24;     // bf16 elements per row of the v tiles (48 B: conflict-free ldmatrix)

struct Item {
    int a;          // adapter (-1: nothing to do)
    int c;          // chunk of that adapter's tokens
    int ntok;
    int rank;
    float scale;
    int tok[kTok];
};

// Byte sizes of the shared regions that two buffers share (see the kernel).
struct BgmvLayout {
    int a_bytes;    // A_T chunk / warp partials
    int xy_bytes;   // x and y tiles / id list and histogram
};
__host__ __device__ inline BgmvLayout bgmv_layout(int slice_in, int slice_out, int T, int n_ids) {
    const int a = kJ * (slice_in + 8) * 2, red = kWarps * kTok * kJ * 4;
    const int xy = kTok * (slice_in + 8) * 2 + kTok * (slice_out + 8) * 2, ids = ((T + n_ids + 1) * 4 + 15) & ~15;
    return BgmvLayout{a > red ? a : red, xy > ids ? xy : ids};
}

struct BgmvParams {
    PoolView pv;
    int m;
    int h_in, h_out;
    int slice_in, slice_out;    // elements per CTA (multiples of 16 and 128)
    int n_ids;                  // adapter ids < n_ids may be loaded on this matrix
    int T;
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    const int *ids;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ int clamp_page(const PoolView &pv, int id) {
    return id < 0 ? 0 : (id >= pv.n_pages ? pv.n_pages - 1 : id);
}

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

// D (16x8 fp32) += A (16x16 bf16, row) . B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Arrive (release, cluster scope) on the barrier at the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ void remote_arrive(uint64_t *bar, int rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(ra) : "memory");
}

// Store `v` into the float at the same offset as `dst` in CTA `rank` of the
// cluster; the store completes as a transaction of 4 bytes on that CTA's
// barrier at the offset of `bar`.
__device__ __forceinline__ void store_async_remote(float *dst, float v, uint64_t *bar, int rank) {
    uint32_t rd, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(rd) : "r"(smem_u32(dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n" ::"r"(rd),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Bounded wait (acquire, cluster scope) for the phase of `parity`; false after 2 s.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity) {
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t0));
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 63u) == 63u) {
            asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
            if (t - t0 > 2000000000ull) return false;
        }
    }
}

// Exclusive scan of n ints in place (block-wide, kThreads threads); returns the total.
__device__ int block_exclusive_scan(int *v, int n, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = tid * per, hi = min(n, lo + per);
    int s = 0;
    for (int i = lo; i < hi; ++i) s += v[i];
    int inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            int t = warp_tot[w];
            warp_tot[w] = run;
            run += t;
        }
        warp_tot[kWarps] = run;
    }
    __syncthreads();
    int run = warp_tot[warp] + inc - s;
    for (int i = lo; i < hi; ++i) {
        int t = v[i];
        v[i] = run;
        run += t;
    }
    const int total = warp_tot[kWarps];
    __syncthreads();
    return total;
}

// Ordered compaction: tokens t with ids[t] == a whose rank among them lies in
// [c*kTok, (c+1)*kTok) go to tok[rank - c*kTok].  Returns that count.
__device__ int collect_tokens(const int *ids, int T, int a, int c, int *tok, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int run = 0;
    for (int base = 0; base < T; base += kThreads) {
        const int t = base + tid;
        const bool hit = t < T && ids[t] == a;
        const unsigned mask = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) warp_tot[warp] = __popc(mask);
        __syncthreads();
        int off = run;
        for (int w = 0; w < warp; ++w) off += warp_tot[w];
        int round_total = 0;
        for (int w = 0; w < kWarps; ++w) round_total += warp_tot[w];
        if (hit) {
            const int pos = off + __popc(mask & ((1u << lane) - 1u)) - c * kTok;
            if (pos >= 0 && pos < kTok) tok[pos] = t;
        }
        run += round_total;
        __syncthreads();
    }
    const int n = run - c * kTok;
    return n < 0 ? 0 : (n > kTok ? kTok : n);
}

__global__ void __launch_bounds__(kThreads, 3) bgmv_cluster_kernel(BgmvParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int item_idx = blockIdx.x / kC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const PoolView &pv = p.pv;
    // the next kernel on the stream may start once every CTA of this one has:
    // its CTAs only read the pool before they wait for this grid to finish,
    // so their page prefetch overlaps this launch's compute and exchange
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- shared memory carve-up (row pitches padded by 16 B for conflict-free
    //      ldmatrix).  Regions whose lifetimes do not overlap share space: the
    //      warps' partial sums live over A_T's chunk once the shrink has read it,
    //      and the id list / histogram over the x and y tiles, which are loaded
    //      only after the item's tokens are known.
    const int pin = p.slice_in + 8, pout = p.slice_out + 8;
    const BgmvLayout L = bgmv_layout(p.slice_in, p.slice_out, p.T, p.n_ids);
    __nv_bfloat16 *sA = reinterpret_cast<__nv_bfloat16 *>(smem_raw);   // [kJ][pin]   rows of A_T
    float *red = reinterpret_cast<float *>(smem_raw);                    // [kWarps][kTok*kJ] (over sA)
    __nv_bfloat16 *sB = reinterpret_cast<__nv_bfloat16 *>(smem_raw + L.a_bytes);   // [kJ][pout] rows of B
    __nv_bfloat16 *sX = sB + kJ * pout;                                  // [kTok][pin] rows of x
    __nv_bfloat16 *sY = sX + kTok * pin;                                 // [kTok][pout] rows of y
    int *sids = reinterpret_cast<int *>(sX);                             // [T] (over sX, sY)
    int *hist = sids + p.T;                                              // [n_ids + 1]
    __nv_bfloat16 *sVh = reinterpret_cast<__nv_bfloat16 *>(reinterpret_cast<uint8_t *>(sX) + L.xy_bytes);
    __nv_bfloat16 *sVl = sVh + kTok * kVPitch;                           // [kTok][kVPitch] v residual
    float *recv = reinterpret_cast<float *>(sVl + kTok * kVPitch);       // [kC][kTok*kJ] partials of every CTA
    uint64_t *bars = reinterpret_cast<uint64_t *>(recv + kC * kTok * kJ); // [0] partials in, [1] partials consumed
    int *rec = reinterpret_cast<int *>(bars + 2);                        // [rec_ints]
    int *warp_tot = rec + pv.rec_ints;                                   // [kWarps + 2]
    Item *mine = reinterpret_cast<Item *>(warp_tot + kWarps + 2);
    const Item *item;

    // ---- 1. before the previous kernel on the stream has finished: this
    //         cluster's page-table record and its first rows of pages.  Only
    //         the pool's load path writes these, and it ends in an event
    //         record, which orders it fully before this launch.
    int a = item_idx < p.n_ids ? item_idx : -1;
    int c = 0;
    if (a >= 0)
        for (int i = tid; i < pv.rec_ints; i += kThreads)
            rec[i] = pv.table[((long long)a * pv.n_matrices + p.m) * pv.rec_ints + i];
    __syncthreads();

    const int k0 = crank * p.slice_in;
    const int nkv = max(0, min(p.slice_in, p.h_in - k0)) / 8;      // valid 16-byte vectors of x / A_T
    const int n0 = crank * p.slice_out;
    const int ncv = max(0, min(p.slice_out, p.h_out - n0)) / 8;    // valid 16-byte vectors of y / B
    const int kvpow = 31 - __clz(max(p.slice_in / 8, 1));          // slice sizes are powers of two
    const int cvpow = 31 - __clz(max(p.slice_out / 8, 1));

    auto prefetch_pages = [&](int r_own, int jc) {
        const int jn = min(kJ, r_own - jc * kJ);
        const int sv_in = p.slice_in / 8, sv_out = p.slice_out / 8;
        for (int i = tid; i < kJ * sv_in; i += kThreads) {
            const int jj = i >> kvpow, kv = i & (sv_in - 1);
            __nv_bfloat16 *dst = sA + jj * pin + kv * 8;
            if (jj < jn && kv < nkv) {
                const int page = clamp_page(pv, rec[kRecHeader + jc * kJ + jj]);
                cp_async16(dst, page_row<__nv_bfloat16>(pv, page) + k0 + kv * 8);
            } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
        }
        for (int i = tid; i < kJ * sv_out; i += kThreads) {
            const int jj = i >> cvpow, cv = i & (sv_out - 1);
            __nv_bfloat16 *dst = sB + jj * pout + cv * 8;
            if (jj < jn && cv < ncv) {
                const int page = clamp_page(pv, rec[kRecHeader + r_own + jc * kJ + jj]);
                cp_async16(dst, page_row<__nv_bfloat16>(pv, page) + n0 + cv * 8);
            } else {
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
        }
    };

    int r_own = 0;
    if (a >= 0) {
        r_own = min(max(rec[0], 0), pv.max_rank);
        prefetch_pages(r_own, 0);
    }
    // the exchange barriers, published to the cluster before any CTA touches a peer
    // (the matching wait comes right before the first remote access)
    if (tid == 0) {
        mbar_init(&bars[0], 1);        // own arrival with the expected bytes; the partials come as transactions
        mbar_init(&bars[1], kC);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");

    // ---- 2. inputs that earlier stream work may produce: wait for it
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    for (int t = tid; t < p.T; t += kThreads) {
        const int id = p.ids[t];
        sids[t] = id;
        if (blockIdx.x == 0 && id >= p.n_ids) flag(pv.status, LORA_DEV_BAD_ADAPTER);
    }
    __syncthreads();
    if (a < 0) {
        // overflow item: find (adapter, chunk >= 1) from a histogram of the ids
        for (int i = tid; i <= p.n_ids; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int t = tid; t < p.T; t += kThreads) {
            const int id = sids[t];
            if (id >= 0 && id < p.n_ids) atomicAdd(&hist[id], 1);
        }
        __syncthreads();
        for (int i = tid; i < p.n_ids; i += kThreads) hist[i] = max(0, (hist[i] + kTok - 1) / kTok - 1);
        __syncthreads();
        const int total = block_exclusive_scan(hist, p.n_ids, warp_tot);
        const int o = item_idx - p.n_ids;
        if (tid == 0) {
            int found = -1;
            if (o < total) {
                int lo = 0, hi = p.n_ids - 1;     // last adapter whose start <= o
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (hist[mid] <= o) lo = mid; else hi = mid - 1;
                }
                found = lo;
                warp_tot[0] = 1 + (o - hist[lo]);
            }
            warp_tot[1] = found;
        }
        __syncthreads();
        a = warp_tot[1];
        c = warp_tot[0];
        __syncthreads();
        if (a >= 0) {
            for (int i = tid; i < pv.rec_ints; i += kThreads)
                rec[i] = pv.table[((long long)a * pv.n_matrices + p.m) * pv.rec_ints + i];
            __syncthreads();
            r_own = min(max(rec[0], 0), pv.max_rank);
            prefetch_pages(r_own, 0);
        }
    }

    // ---- 3. the item: every CTA of the cluster derives the same one from the
    //         same ids and table, so all take the same branches; start its x
    //         and y loads at once
    int ntok = 0;
    if (a >= 0) ntok = collect_tokens(sids, p.T, a, c, mine->tok, warp_tot);
    if (tid == 0) {
        mine->a = a;
        mine->c = c;
        mine->ntok = ntok;
        mine->rank = (a >= 0) ? rec[0] : -1;
        mine->scale = (a >= 0) ? __int_as_float(rec[1]) : 0.f;
    }
    __syncthreads();
    auto load_x = [&](const Item *it_, int nt) {
        const int sv_in = p.slice_in / 8;
        for (int i = tid; i < kTok * sv_in; i += kThreads) {
            const int tl = i >> kvpow, kv = i & (sv_in - 1);
            __nv_bfloat16 *dst = sX + tl * pin + kv * 8;
            if (tl < nt && kv < nkv)
                cp_async16(dst, p.x + (long long)it_->tok[tl] * p.h_in + k0 + kv * 8);
            else
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
    };
    // MMA fragment coordinates: g = row group, q = thread in group
    const int g = lane >> 2, q = lane & 3;
    // Expand output tile of this warp: columns [wc0, wc0 + cw) of the CTA slice, n-tiles of 8
    const int cw = p.slice_out / kWarps;             // multiple of 16
    const int wc0 = warp * cw;
    const int ntiles = cw / 8;                       // <= kMaxSliceOut / kWarps / 8 = 8
    auto load_y = [&](const Item *it_, int nt) {
        const int sv_out = p.slice_out / 8;
        for (int i = tid; i < nt * sv_out; i += kThreads) {
            const int tl = i >> cvpow, cv = i & (sv_out - 1);
            if (cv < ncv) cp_async16(sY + tl * pout + cv * 8, p.y + (long long)it_->tok[tl] * p.h_out + n0 + cv * 8);
        }
    };
    if (ntok > 0) {
        load_x(mine, ntok);
        load_y(mine, ntok);
    }
    item = mine;
    const int ia = item->a, intok = min(max(item->ntok, 0), kTok);
    // nothing to add: no adapter, no tokens, or rank 0 (y stays as it is; an
    // unloaded adapter is also flagged)
    if (ia < 0 || intok == 0 || item->rank <= 0) {
        if (ia >= 0 && intok > 0 && item->rank < 0 && crank == 0 && tid == 0) flag(pv.status, LORA_DEV_BAD_ADAPTER);
        asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
        cp_async_wait_all();   // no copy may still be landing when the CTA exits
        return;
    }
    const int rank = min(item->rank, pv.max_rank);
    const float scale = item->scale;

    float dacc[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) dacc[t][e] = 0.f;

    const int n_jc = (rank + kJ - 1) / kJ;
    bool failed = false;
    for (int jc = 0; jc < n_jc; ++jc) {
        const int jn = max(0, min(kJ, min(rank, r_own) - jc * kJ));
        if (jc > 0) prefetch_pages(r_own, jc);
        cp_async_wait_all();
        __syncthreads();

        // partial shrink over this CTA's h_in slice: warp w takes k-steps w, w+8, ...
        {
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            const int ksteps = p.slice_in / 16;
            for (int ks = warp; ks < ksteps; ks += kWarps) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                // x tile 16 x 16: lane l -> row (l & 15), column half (l >> 4)
                ldsm_x4(sX + (lane & 15) * pin + ks * 16 + (lane >> 4) * 8, a0, a1, a2, a3);
                // A_T rows as B operand: matrices (j 0-7,k 0-7) (j 0-7,k 8-15) (j 8-15,k 0-7) (j 8-15,k 8-15)
                ldsm_x4(sA + ((lane & 7) + ((lane >> 4) << 3)) * pin + ks * 16 + ((lane >> 3) & 1) * 8, b0, b1, b2,
                        b3);
                mma16816(d0, a0, a1, a2, a3, b0, b1);
                mma16816(d1, a0, a1, a2, a3, b2, b3);
            }
            __syncthreads();     // every warp is done with sA: the partials overwrite it
            float *rw = red + warp * kTok * kJ;
            rw[g * kJ + 2 * q] = d0[0];
            rw[g * kJ + 2 * q + 1] = d0[1];
            rw[(g + 8) * kJ + 2 * q] = d0[2];
            rw[(g + 8) * kJ + 2 * q + 1] = d0[3];
            rw[g * kJ + 8 + 2 * q] = d1[0];
            rw[g * kJ + 8 + 2 * q + 1] = d1[1];
            rw[(g + 8) * kJ + 8 + 2 * q] = d1[2];
            rw[(g + 8) * kJ + 8 + 2 * q + 1] = d1[3];
        }
        __syncthreads();
        {
            float part = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) part += red[w * kTok * kJ + tid];   // kThreads == kTok * kJ
            // push this CTA's partial into every CTA's receive slot, then signal them
            if (jc == 0) asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");   // peers' barriers exist
            if (jc > 0 && !wait_bar(&bars[1], (uint32_t)(jc - 1) & 1u)) failed = true;
            // asynchronous remote stores that count their bytes on the receiver's barrier
            if (!failed) {
#pragma unroll
                for (int r = 0; r < kC; ++r) store_async_remote(recv + crank * kTok * kJ + tid, part, &bars[0], r);
            }
            // this CTA's own phase: it expects every CTA's partial (kC x kTok x kJ floats)
            if (tid == 0) mbar_arrive_expect_tx(&bars[0], (uint32_t)(kC * kTok * kJ * sizeof(float)));
        }
        if (!failed && !wait_bar(&bars[0], (uint32_t)jc & 1u)) failed = true;
        if (__syncthreads_or(failed)) {
            // Leaving while a peer could still store its partial here would let
            // that store land in a finished CTA: give this round's partials a
            // second bounded window first (a peer that gave up itself sends no
            // more; one that is only late lands within it).
            if (tid == 0) flag(pv.status, LORA_DEV_WAIT_TIMEOUT);
            wait_bar(&bars[0], (uint32_t)jc & 1u);
            cp_async_wait_all();
            return;
        }
        {
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < kC; ++r) sum += recv[r * kTok * kJ + tid];
            const int tl = tid >> 4, jj = tid & 15;
            const float val = jj < jn ? scale * sum : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(val);
            sVh[tl * kVPitch + jj] = hi;
            sVl[tl * kVPitch + jj] = __float2bfloat16_rn(val - __bfloat162float(hi));
        }
        __syncthreads();     // receive slots read; sA and sB may be refilled
        if (tid == 0 && jc + 1 < n_jc)
            for (int r = 0; r < kC; ++r) remote_arrive(&bars[1], r);

        // expand on this CTA's h_out slice: D[16 tok x 8 cols] per n-tile, K = 16 ranks
        {
            uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
            ldsm_x4(sVh + (lane & 15) * kVPitch + (lane >> 4) * 8, h0, h1, h2, h3);
            ldsm_x4(sVl + (lane & 15) * kVPitch + (lane >> 4) * 8, l0, l1, l2, l3);
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
                if (t >= ntiles) break;
                uint32_t b0, b1, b2, b3;
                // B rows (k = rank) n-contiguous, transposed into col fragments:
                // matrices (k 0-7, n t) (k 8-15, n t) (k 0-7, n t+1) (k 8-15, n t+1)
                ldsm_x4_t(sB + ((lane & 7) + ((lane >> 3) & 1) * 8) * pout + wc0 + (t + (lane >> 4)) * 8, b0, b1,
                          b2, b3);
                mma16816(dacc[t], h0, h1, h2, h3, b0, b1);
                mma16816(dacc[t], l0, l1, l2, l3, b0, b1);
                mma16816(dacc[t + 1], h0, h1, h2, h3, b2, b3);
                mma16816(dacc[t + 1], l0, l1, l2, l3, b2, b3);
            }
        }
        __syncthreads();
    }

    // ---- y += delta: add into the y tile in shared memory, then coalesced stores
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        if (t >= ntiles) break;
        const int col = wc0 + t * 8 + 2 * q;               // within the CTA slice
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            __nv_bfloat162 *yy = reinterpret_cast<__nv_bfloat162 *>(sY + (g + 8 * h) * pout + col);
            const float2 f = __bfloat1622float2(*yy);
            *yy = __floats2bfloat162_rn(f.x + dacc[t][2 * h], f.y + dacc[t][2 * h + 1]);
        }
    }
    __syncthreads();
    {
        const int sv_out = p.slice_out / 8;
        for (int i = tid; i < intok * sv_out; i += kThreads) {
            const int tl = i >> cvpow, cv = i & (sv_out - 1);
            if (cv < ncv)
                *reinterpret_cast<uint4 *>(p.y + (long long)item->tok[tl] * p.h_out + n0 + cv * 8) =
                    *reinterpret_cast<const uint4 *>(sY + tl * pout + cv * 8);
        }
    }
}

// ---------------------------------------------------------------------------
// Compacted mode, for adapter-id ranges large next to the batch (a pool of
// thousands of adapters serving a few hundred decode tokens).  The grid no
// longer has a cluster per id: G persistent clusters (as many as the GPU holds,
// at most the item bound min(T, n_ids) + T / kTok) walk the batch's items.
// After the wait on the previous kernel every CTA reads the ids, counts the
// tokens of each adapter and scans ceil(count / kTok), which numbers the items
// (adapter, chunk) of the adapters present in the batch; cluster c takes items
// c, 2G-1-c, 2G+c, ... (snake order).  No page is read for an adapter the batch
// does not use (measured: 2048 adapters loaded, 256 decode tokens over about
// 245 of them, 4096 x 4096: 74 us per launch).  Each item runs as in
// bgmv_cluster_kernel; the exchange
// barriers' phases run on across items: round R (every 16-rank chunk of every
// item the cluster takes) completes phase R of bars[0] and, when another
// round follows, of bars[1].  All CTAs of a cluster derive the same items and
// ranks from the same ids and table, so they agree on every phase and none
// signals a peer after its last round.
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t bgmv_compact_smem(int slice_in, int slice_out, int T, int n_ids, int rec_ints) {
    const int pin = slice_in + 8, pout = slice_out + 8;
    const int a = kJ * pin * 2, red = kWarps * kTok * kJ * 4;
    return (size_t)(a > red ? a : red) + (size_t)kJ * pout * 2 + (size_t)kTok * pin * 2 + (size_t)kTok * pout * 2 +
           (size_t)2 * kTok * kVPitch * 2 + (size_t)kC * kTok * kJ * 4 + 16 +
           (size_t)(rec_ints + kWarps + 2 + kTok + T + n_ids + 1) * 4 + 16;
}

// collect_tokens with one barrier: warp w scans its contiguous slice of the ids
// and counts the tokens of adapter a; after the warps' counts are published
// each warp writes its matches whose rank among all of a's tokens (index order)
// falls in chunk c.  The same ordered list as collect_tokens.
__device__ int collect_tokens_sliced(const int *ids, int T, int a, int c, int *tok, int *wcnt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (T + kWarps - 1) / kWarps, lo = min(T, warp * per), hi = min(T, lo + per);
    int n = 0;
    for (int t0 = lo; t0 < hi; t0 += 32) {
        const int t = t0 + lane;
        n += __popc(__ballot_sync(0xffffffffu, t < hi && ids[t] == a));
    }
    if (lane == 0) wcnt[warp] = n;
    __syncthreads();
    int run = 0, total = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) run += wcnt[w];
        total += wcnt[w];
    }
    const int first = c * kTok;
    if (run < first + kTok && run + n > first) {
        for (int t0 = lo; t0 < hi; t0 += 32) {
            const int t = t0 + lane;
            const bool hit = t < hi && ids[t] == a;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            const int pos = run + __popc(m & ((1u << lane) - 1u)) - first;
            if (hit && pos >= 0 && pos < kTok) tok[pos] = t;
            run += __popc(m);
        }
    }
    __syncthreads();
    const int cnt = total - first;
    return cnt < 0 ? 0 : (cnt > kTok ? kTok : cnt);
}

__global__ void __launch_bounds__(kThreads, 2) bgmv_compact_kernel(BgmvParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int G = gridDim.x / kC, cid = blockIdx.x / kC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const PoolView &pv = p.pv;
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    const int pin = p.slice_in + 8, pout = p.slice_out + 8;
    const int a_bytes = max(kJ * pin * 2, kWarps * kTok * kJ * 4);
    __nv_bfloat16 *sA = reinterpret_cast<__nv_bfloat16 *>(smem_raw);   // [kJ][pin]   rows of A_T
    float *red = reinterpret_cast<float *>(smem_raw);                    // [kWarps][kTok*kJ] (over sA)
    __nv_bfloat16 *sB = reinterpret_cast<__nv_bfloat16 *>(smem_raw + a_bytes);   // [kJ][pout] rows of B
    __nv_bfloat16 *sX = sB + kJ * pout;                                  // [kTok][pin] rows of x
    __nv_bfloat16 *sY = sX + kTok * pin;                                 // [kTok][pout] rows of y
    __nv_bfloat16 *sVh = sY + kTok * pout;                               // [kTok][kVPitch] s v, high part
    __nv_bfloat16 *sVl = sVh + kTok * kVPitch;                           // [kTok][kVPitch] residual
    float *recv = reinterpret_cast<float *>(sVl + kTok * kVPitch);       // [kC][kTok*kJ] partials of every CTA
    uint64_t *bars = reinterpret_cast<uint64_t *>(recv + kC * kTok * kJ); // [0] partials in, [1] consumed
    int *rec = reinterpret_cast<int *>(bars + 2);                        // [rec_ints]
    int *warp_tot = rec + pv.rec_ints;                                   // [kWarps + 2]
    int *tok = warp_tot + kWarps + 2;                                    // [kTok]
    int *sids = tok + kTok;                                              // [T]
    int *hist = sids + p.T;                                              // [n_ids + 1]

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], kC);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    for (int i = tid; i <= p.n_ids; i += kThreads) hist[i] = 0;
    __syncthreads();
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");

    // ---- the batch's items: every CTA numbers them the same way
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    for (int t = tid; t < p.T; t += kThreads) {
        const int id = p.ids[t];
        sids[t] = id;
        if (id >= 0 && id < p.n_ids) atomicAdd(&hist[id], 1);
        else if (blockIdx.x == 0 && id >= p.n_ids) flag(pv.status, LORA_DEV_BAD_ADAPTER);
    }
    __syncthreads();
    for (int i = tid; i < p.n_ids; i += kThreads) hist[i] = (hist[i] + kTok - 1) / kTok;
    __syncthreads();
    const int n_items = block_exclusive_scan(hist, p.n_ids, warp_tot);
    auto item_at = [&](int k) { return k * G + ((k & 1) ? G - 1 - cid : cid); };
    auto adapter_of_item = [&](int i) {   // last adapter whose first item index is <= i
        int lo = 0, hi = p.n_ids - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (hist[mid] <= i) lo = mid; else hi = mid - 1;
        }
        return lo;
    };
    auto rank_in_table = [&](int a) {
        return pv.table[((long long)a * pv.n_matrices + p.m) * pv.rec_ints];
    };
    int total_rounds = 0;
    for (int k = 0;; ++k) {
        const int i = item_at(k);
        if (i >= n_items) break;
        const int r = min(max(rank_in_table(adapter_of_item(i)), 0), pv.max_rank);
        total_rounds += (r + kJ - 1) / kJ;
    }

    const int k0 = crank * p.slice_in;
    const int nkv = max(0, min(p.slice_in, p.h_in - k0)) / 8;
    const int n0 = crank * p.slice_out;
    const int ncv = max(0, min(p.slice_out, p.h_out - n0)) / 8;
    const int kvpow = 31 - __clz(max(p.slice_in / 8, 1));
    const int cvpow = 31 - __clz(max(p.slice_out / 8, 1));
    const int g = lane >> 2, q = lane & 3;
    const int cw = p.slice_out / kWarps;
    const int wc0 = warp * cw;
    const int ntiles = cw / 8;
    int R = 0;

    for (int k = 0;; ++k) {
        const int ii = item_at(k);
        if (ii >= n_items) break;
        const int a = adapter_of_item(ii), c = ii - hist[a];
        __syncthreads();                        // the previous item's readers of rec, tok and the tiles are done
        for (int i = tid; i < pv.rec_ints; i += kThreads)
            rec[i] = pv.table[((long long)a * pv.n_matrices + p.m) * pv.rec_ints + i];
        const int ntok = collect_tokens_sliced(sids, p.T, a, c, tok, warp_tot);   // ends with a barrier
        const int rank = min(max(rec[0], 0), pv.max_rank);
        if (rec[0] < 0) {
            if (crank == 0 && tid == 0) flag(pv.status, LORA_DEV_BAD_ADAPTER);
            continue;
        }
        const int n_jc = (rank + kJ - 1) / kJ;
        if (n_jc == 0) continue;               // rank 0: y stays as it is (counted as no round above)
        const float scale = __int_as_float(rec[1]);
        auto prefetch_pages = [&](int jc) {
            const int jn = min(kJ, rank - jc * kJ);
            const int sv_in = p.slice_in / 8, sv_out = p.slice_out / 8;
            for (int i = tid; i < kJ * sv_in; i += kThreads) {
                const int jj = i >> kvpow, kv = i & (sv_in - 1);
                __nv_bfloat16 *dst = sA + jj * pin + kv * 8;
                if (jj < jn && kv < nkv)
                    cp_async16(dst, page_row<__nv_bfloat16>(pv, clamp_page(pv, rec[kRecHeader + jc * kJ + jj])) + k0 +
                                        kv * 8);
                else
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
            for (int i = tid; i < kJ * sv_out; i += kThreads) {
                const int jj = i >> cvpow, cv = i & (sv_out - 1);
                __nv_bfloat16 *dst = sB + jj * pout + cv * 8;
                if (jj < jn && cv < ncv)
                    cp_async16(dst, page_row<__nv_bfloat16>(pv, clamp_page(pv, rec[kRecHeader + rank + jc * kJ + jj])) +
                                        n0 + cv * 8);
                else
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
        };
        prefetch_pages(0);
        {
            const int sv_in = p.slice_in / 8, sv_out = p.slice_out / 8;
            for (int i = tid; i < kTok * sv_in; i += kThreads) {
                const int tl = i >> kvpow, kv = i & (sv_in - 1);
                __nv_bfloat16 *dst = sX + tl * pin + kv * 8;
                if (tl < ntok && kv < nkv)
                    cp_async16(dst, p.x + (long long)tok[tl] * p.h_in + k0 + kv * 8);
                else
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
            }
            for (int i = tid; i < ntok * sv_out; i += kThreads) {
                const int tl = i >> cvpow, cv = i & (sv_out - 1);
                if (cv < ncv) cp_async16(sY + tl * pout + cv * 8, p.y + (long long)tok[tl] * p.h_out + n0 + cv * 8);
            }
        }
        float dacc[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) dacc[t][e] = 0.f;
        for (int jc = 0; jc < n_jc; ++jc, ++R) {
            const int jn = min(kJ, rank - jc * kJ);
            if (jc > 0) prefetch_pages(jc);
            cp_async_wait_all();
            __syncthreads();
            {
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                const int ksteps = p.slice_in / 16;
                for (int ks = warp; ks < ksteps; ks += kWarps) {
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldsm_x4(sX + (lane & 15) * pin + ks * 16 + (lane >> 4) * 8, a0, a1, a2, a3);
                    ldsm_x4(sA + ((lane & 7) + ((lane >> 4) << 3)) * pin + ks * 16 + ((lane >> 3) & 1) * 8, b0, b1,
                            b2, b3);
                    mma16816(d0, a0, a1, a2, a3, b0, b1);
                    mma16816(d1, a0, a1, a2, a3, b2, b3);
                }
                __syncthreads();     // every warp is done with sA: the partials overwrite it
                float *rw = red + warp * kTok * kJ;
                rw[g * kJ + 2 * q] = d0[0];
                rw[g * kJ + 2 * q + 1] = d0[1];
                rw[(g + 8) * kJ + 2 * q] = d0[2];
                rw[(g + 8) * kJ + 2 * q + 1] = d0[3];
                rw[g * kJ + 8 + 2 * q] = d1[0];
                rw[g * kJ + 8 + 2 * q + 1] = d1[1];
                rw[(g + 8) * kJ + 8 + 2 * q] = d1[2];
                rw[(g + 8) * kJ + 8 + 2 * q + 1] = d1[3];
            }
            __syncthreads();
            bool failed = false;
            {
                float part = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) part += red[w * kTok * kJ + tid];   // kThreads == kTok * kJ
                if (R == 0) asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");   // peers' barriers exist
                if (R > 0 && !wait_bar(&bars[1], (uint32_t)(R - 1) & 1u)) failed = true;
                if (!failed) {
#pragma unroll
                    for (int r = 0; r < kC; ++r) store_async_remote(recv + crank * kTok * kJ + tid, part, &bars[0], r);
                }
                if (tid == 0) mbar_arrive_expect_tx(&bars[0], (uint32_t)(kC * kTok * kJ * sizeof(float)));
            }
            if (!failed && !wait_bar(&bars[0], (uint32_t)R & 1u)) failed = true;
            if (__syncthreads_or(failed)) {
                // a second bounded window for peers' late partials before the CTA leaves
                if (tid == 0) flag(pv.status, LORA_DEV_WAIT_TIMEOUT);
                wait_bar(&bars[0], (uint32_t)R & 1u);
                cp_async_wait_all();
                return;
            }
            {
                float sum = 0.f;
#pragma unroll
                for (int r = 0; r < kC; ++r) sum += recv[r * kTok * kJ + tid];
                const int tl = tid >> 4, jj = tid & 15;
                const float val = jj < jn ? scale * sum : 0.f;
                const __nv_bfloat16 hi = __float2bfloat16_rn(val);
                sVh[tl * kVPitch + jj] = hi;
                sVl[tl * kVPitch + jj] = __float2bfloat16_rn(val - __bfloat162float(hi));
            }
            __syncthreads();     // receive slots read; sA and sB may be refilled
            if (tid == 0 && R + 1 < total_rounds)
                for (int r = 0; r < kC; ++r) remote_arrive(&bars[1], r);
            {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                ldsm_x4(sVh + (lane & 15) * kVPitch + (lane >> 4) * 8, h0, h1, h2, h3);
                ldsm_x4(sVl + (lane & 15) * kVPitch + (lane >> 4) * 8, l0, l1, l2, l3);
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    if (t >= ntiles) break;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(sB + ((lane & 7) + ((lane >> 3) & 1) * 8) * pout + wc0 + (t + (lane >> 4)) * 8, b0, b1,
                              b2, b3);
                    mma16816(dacc[t], h0, h1, h2, h3, b0, b1);
                    mma16816(dacc[t], l0, l1, l2, l3, b0, b1);
                    mma16816(dacc[t + 1], h0, h1, h2, h3, b2, b3);
                    mma16816(dacc[t + 1], l0, l1, l2, l3, b2, b3);
                }
            }
            __syncthreads();
        }
        // y += delta in the shared y tile, then coalesced stores
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t >= ntiles) break;
            const int col = wc0 + t * 8 + 2 * q;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                __nv_bfloat162 *yy = reinterpret_cast<__nv_bfloat162 *>(sY + (g + 8 * h) * pout + col);
                const float2 f = __bfloat1622float2(*yy);
                *yy = __floats2bfloat162_rn(f.x + dacc[t][2 * h], f.y + dacc[t][2 * h + 1]);
            }
        }
        __syncthreads();
        {
            const int sv_out = p.slice_out / 8;
            for (int i = tid; i < ntok * sv_out; i += kThreads) {
                const int tl = i >> cvpow, cv = i & (sv_out - 1);
                if (cv < ncv)
                    *reinterpret_cast<uint4 *>(p.y + (long long)tok[tl] * p.h_out + n0 + cv * 8) =
                        *reinterpret_cast<const uint4 *>(sY + tl * pout + cv * 8);
            }
        }
    }
    if (R == 0) asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
    cp_async_wait_all();
}

int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

// Slices per CTA: powers of two, h_in slices a multiple of 16 elements, h_out
// slices a multiple of 128 (8 warps x 16 columns).
static int slice_in_of(int h_in) { return pow2_at_least(std::max(16, (h_in + kC - 1) / kC)); }
static int slice_out_of(int h_out) { return pow2_at_least(std::max(128, (h_out + kC - 1) / kC)); }

// Whether the clustered kernels take this problem (else the per-token kernel
// does): bf16, a batch of at most kMaxT tokens, and an id range the compacted
// mode's histogram holds.  (Measured: for a 16384-token batch of 128-token
// runs over 1024 mixed-rank adapters, 768 wide, consecutive kMaxT-token chunks
// of the compacted kernel took 412 us per call and the per-token kernel 103
// us, so larger batches stay on the per-token kernel.)
constexpr int kMaxCompactIds = 8192;
bool bgmv_cluster_ok(const lora_pool *pool, int h_in, int h_out, int T, int n_ids) {
    return pool->dtype == LORA_BF16 && T <= kMaxT && n_ids > 0 && n_ids <= kMaxCompactIds && h_in % 16 == 0 &&
           slice_in_of(h_in) <= kMaxSliceIn && slice_out_of(h_out) <= kMaxSliceOut;
}

// A batch of at most kMaxT tokens.  Id-indexed mode (a cluster per adapter id,
// pages prefetched before the wait on the previous kernel) while the id range is
// small next to the batch; compacted persistent mode otherwise, so the grid and
// the page reads follow the batch, not the id range.
static int launch_bgmv_chunk(const lora_pool *pool, int matrix, int h_in, int h_out, const __nv_bfloat16 *x,
                             __nv_bfloat16 *y, const int *ids, int T, int n_ids, cudaStream_t st) {
    BgmvParams p;
    p.pv = pool->view();
    p.m = matrix;
    p.h_in = h_in;
    p.h_out = h_out;
    p.slice_in = slice_in_of(h_in);
    p.slice_out = slice_out_of(h_out);
    p.n_ids = n_ids;
    p.T = T;
    p.x = x;
    p.y = y;
    p.ids = ids;
    const bool compact = n_ids > std::max(64, T / 8) || n_ids > kMaxIds;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may overlap the previous kernel's tail
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    if (!compact) {
        const BgmvLayout lay = bgmv_layout(p.slice_in, p.slice_out, T, n_ids);
        const size_t smem = (size_t)lay.a_bytes + (size_t)kJ * (p.slice_out + 8) * 2 + (size_t)lay.xy_bytes +
                            (size_t)2 * kTok * kVPitch * 2 + (size_t)kC * kTok * kJ * 4 + 16 +
                            (size_t)(p.pv.rec_ints + kWarps + 2) * 4 + sizeof(Item) + 16;
        if (smem_optin(reinterpret_cast<const void *>(bgmv_cluster_kernel), smem)) return LORA_ERR_CUDA;
        cfg.gridDim = dim3((n_ids + (T + kTok - 1) / kTok) * kC);
        cfg.dynamicSmemBytes = smem;
        e = cudaLaunchKernelEx(&cfg, bgmv_cluster_kernel, p);
    } else {
        const size_t smem = bgmv_compact_smem(p.slice_in, p.slice_out, T, n_ids, p.pv.rec_ints);
        if (smem_optin(reinterpret_cast<const void *>(bgmv_compact_kernel), smem)) return LORA_ERR_CUDA;
        cfg.dynamicSmemBytes = smem;
        cfg.gridDim = dim3(kC);
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, bgmv_compact_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            active = 0;
        }
        const int bound = std::min(T, n_ids) + (T + kTok - 1) / kTok;
        const int clusters = std::max(1, std::min(bound, active > 0 ? active : num_sms() / kC));
        cfg.gridDim = dim3(clusters * kC);
        e = cudaLaunchKernelEx(&cfg, bgmv_compact_kernel, p);
    }
    count_launch();
    return cuda_status(e);
}

int launch_bgmv_cluster(const lora_pool *pool, int matrix, int h_in, int h_out, const void *x, void *y,
                        const int *token_adapter, int T, int n_ids, cudaStream_t st) {
    return launch_bgmv_chunk(pool, matrix, h_in, h_out, static_cast<const __nv_bfloat16 *>(x),
                             static_cast<__nv_bfloat16 *>(y), token_adapter, T, n_ids, st);
}

}  // namespace lora
