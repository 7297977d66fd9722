// Paged adapter pool and the C-ABI entry points.
//
// The pool follows S-LoRA's unified paging (slide 8: memory is cut into pages
// of H elements and a rank-R adapter takes R of them; "Multi-LoRA Serving",
// question ladder: mixed ranks in fixed-size slots would fragment memory,
// one paged pool avoids that): one device array of equal pages and a free
// list, so adapters of any rank take exactly the pages they need.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.cuh"

namespace lora {

namespace {
// Per-device launch facts, looked up under one mutex: SM counts, and for each
// (device, kernel) the dynamic shared memory it has been opted in to and the
// resident CTAs per SM measured at given sizes.
struct FuncEntry {
    int device;
    const void *func;
    size_t optin;           // bytes the attribute was last raised to on this device
};
struct OccEntry {
    int device;
    const void *func;
    size_t bytes;
    int threads;
    int occ;
};
std::mutex g_launch_mu;
std::vector<FuncEntry> g_funcs;
std::vector<OccEntry> g_occ;
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(g_launch_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

int smem_optin(const void *func, size_t bytes, int threads, int *occupancy) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_launch_mu);
    FuncEntry *fe = nullptr;
    for (FuncEntry &e : g_funcs)
        if (e.device == dev && e.func == func) fe = &e;
    if (!fe) {
        g_funcs.push_back(FuncEntry{dev, func, 0});
        fe = &g_funcs.back();
    }
    if (bytes > fe->optin) {
        if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
            cudaGetLastError();
            return LORA_ERR_CUDA;
        }
        fe->optin = bytes;
    }
    if (occupancy) {
        for (const OccEntry &e : g_occ)
            if (e.device == dev && e.func == func && e.bytes == bytes && e.threads == threads) {
                *occupancy = e.occ;
                return LORA_OK;
            }
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, func, threads, bytes) != cudaSuccess) {
            cudaGetLastError();
            return LORA_ERR_CUDA;
        }
        g_occ.push_back(OccEntry{dev, func, bytes, threads, occ});
        *occupancy = occ;
    }
    return LORA_OK;
}

std::atomic<unsigned long long> g_launches{0};

// Copies one staged row per block into its page.  Staged layout: rows of A_T
// then rows of B, each `row_bytes[...]` long, packed back to back at 16-byte
// multiples.  The record that points at the pages is copied after this kernel
// (a plain host-to-device copy, see enqueue_load), so a kernel that reads it
// finds the pages written.
struct LoadArgs {
    int rec_index;
    int rank;
    float scale;
    int row_bytes_a;
    int row_bytes_b;
    int ids[2 * 1024];
};

__global__ void load_scatter_kernel(const uint8_t *__restrict__ stage, uint8_t *__restrict__ pages,
                                    long long page_bytes, const LoadArgs *__restrict__ args) {
    const int row = blockIdx.x;
    const int r = args->rank;
    if (row < 2 * r) {
        const bool is_a = row < r;
        const int bytes = is_a ? args->row_bytes_a : args->row_bytes_b;
        const long long src_off = is_a ? (long long)row * args->row_bytes_a
                                       : (long long)r * args->row_bytes_a + (long long)(row - r) * args->row_bytes_b;
        const uint4 *src = reinterpret_cast<const uint4 *>(stage + src_off);
        uint4 *dst = reinterpret_cast<uint4 *>(pages + (long long)args->ids[row] * page_bytes);
        for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) dst[i] = src[i];
    }
}

// One staging slot: the adapter's rows (A_T then B), its LoadArgs, and the
// table record the load publishes.
struct StageLayout {
    size_t args, rec, total;
};
constexpr int kStageSlots = 8;
constexpr size_t kStageRingBytes = (size_t)64 << 20;

StageLayout stage_layout(const lora_pool *p, int rank) {
    const size_t data = (size_t)2 * rank * p->page_elems * p->esize;
    StageLayout L;
    L.args = (data + 255) & ~(size_t)255;
    L.rec = (L.args + sizeof(LoadArgs) + 255) & ~(size_t)255;
    L.total = (L.rec + (size_t)p->rec_ints * sizeof(int) + 255) & ~(size_t)255;
    return L;
}

}  // namespace lora

namespace lora {
// Streams for the parts of a layer call that may run beside the caller's
// stream, with the events that fork them from it and join them back.  One set
// per host thread, device and caller stream (up to kSideSets caller streams per
// thread and device; further ones share the last set made), so that calls issued
// at once on different streams do not queue behind one another's side work.
// Under stream capture the forks and joins become graph edges.
struct SideStream {
    int device = -1;
    cudaStream_t caller = nullptr;
    cudaStream_t s = nullptr, s2 = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
};
constexpr int kSideSets = 16;

static SideStream *side_stream(cudaStream_t caller) {
    thread_local SideStream sets[kSideSets];
    thread_local int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    SideStream *last = nullptr;
    for (int i = 0; i < used; ++i) {
        if (sets[i].device != dev) continue;
        if (sets[i].caller == caller) return &sets[i];
        last = &sets[i];
    }
    if (used == kSideSets) return last;
    // the side streams take the device's highest priority: their kernels are short
    // and the caller's stream waits for them, so when an SM frees up their CTAs
    // should go before the waiting CTAs of long kernels (another call's GEMM)
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) {
        cudaGetLastError();
        greatest = 0;
    }
    SideStream n;
    if (cudaStreamCreateWithPriority(&n.s, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&n.s2, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join2, cudaEventDisableTiming) != cudaSuccess)
        return last;
    n.device = dev;
    n.caller = caller;
    sets[used] = n;
    return &sets[used++];
}

// The adapted layer given scratch for v (T x max_rank fp32): base product for
// the whole batch (tensor cores when the shape allows), then each token's own
// low-rank term: shrink into v, expand into y.
int layer_forward_impl(const lora_pool *p, int matrix, int h_in, int h_out, const void *x, const void *W, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T, float *v, cudaStream_t st,
                       const Fp8Base *f8) {
    int rc;
    const bool tc = gemm_tc_ok(p, h_in, h_out, T, f8 != nullptr);
    if (f8 && !tc) return LORA_ERR_SHAPE;      // the FP8 base product runs on the tensor cores only
    // FP8: x's codes and scales, before the GEMM -- on the call's stream, or (tensor-core
    // tiles, below) on a second side stream beside the tensor-core shrink
    const bool q_side = f8 && f8->quantize && shrink_tc_ok(p, h_in, S) &&
                        sgmv_plan_ok(p, matrix, S, T, true) && sgmv_shrink_ok(p, h_in, S) && sgmv_expand_ok(p, h_out, S);
    if (f8 && f8->quantize && !q_side && (rc = launch_quantize(x, T, h_in, const_cast<void *>(f8->xq),
                                                               const_cast<float *>(f8->sx), st)))
        return rc;
    const bool tcs = tc && shrink_tc_ok(p, h_in, S);
    if (sgmv_plan_ok(p, matrix, S, T, tcs) && sgmv_shrink_ok(p, h_in, S) && sgmv_expand_ok(p, h_out, S)) {
        // With tensor-core tiles (tcs):
        //   main stream: (1) the tensor-core shrink, whose CTAs also decide which
        //     128-row GEMM M-tiles have one adapter for all their rows (tile_ad),
        //     computes v of those tiles; (2) the GEMM adds their low-rank term
        //     itself; after the join, (3) the expand of the remaining rows.
        //   side stream, forked at the start: the plan (the other rows' tokens
        //     grouped by adapter as cost-ordered work units; it classifies the
        //     M-tiles itself with the same function) and the warp-MMA shrink of
        //     those rows.  They read only the segment table, the pool's ranks
        //     and x, and write only the plan and v rows outside fused tiles,
        //     which (1) and (2) never touch.
        // Without tensor-core tiles everything runs on the one stream: plan,
        // shrink, base product, expand.
        int *plan = reinterpret_cast<int *>((reinterpret_cast<uintptr_t>(v + (size_t)T * p->max_rank) + 255) &
                                            ~uintptr_t(255));
        if (!tcs) {
            if ((rc = launch_sgmv_plan(p, matrix, seg_starts, seg_adapter, S, T, plan, st))) return rc;
            if ((rc = launch_sgmv_shrink(p, matrix, h_in, x, v, p->max_rank, seg_starts, seg_adapter, S, T, plan, st)))
                return rc;
            rc = tc ? launch_gemm_tc(p, h_in, h_out, x, W, y, T, st, 0, nullptr, nullptr, 0, f8)
                    : launch_base_gemm(p, h_in, h_out, x, W, y, T, st);
            if (rc) return rc;
            return launch_sgmv_expand(p, matrix, h_out, v, p->max_rank, y, seg_starts, seg_adapter, S, T, plan, st);
        }
        int *tile_ad = sgmv_plan_tiles(p, matrix, T, plan);
        SideStream *side = side_stream(st);
        cudaStream_t st3 = st;
        if (side && cudaEventRecord(side->fork, st) != cudaSuccess) return LORA_ERR_CUDA;
        if (q_side) {   // FP8: x quantised on the second side stream, joined before the GEMM
            cudaStream_t sq = side ? side->s2 : st;
            if (side && cudaStreamWaitEvent(sq, side->fork, 0) != cudaSuccess) return LORA_ERR_CUDA;
            rc = launch_quantize(x, T, h_in, const_cast<void *>(f8->xq), const_cast<float *>(f8->sx), sq);
            if (side && cudaEventRecord(side->join2, sq) != cudaSuccess) {
                cudaStreamWaitEvent(st, side->join2, 0);
                return LORA_ERR_CUDA;
            }
            if (rc) {
                if (side) cudaStreamWaitEvent(st, side->join2, 0);   // no side work is left unjoined
                return rc;
            }
        }
        // the tensor-core shrink is enqueued first, so its CTAs take the SMs first
        rc = launch_shrink_tc(p, matrix, h_in, x, T, tile_ad, seg_starts, seg_adapter, S, v, p->max_rank, st);
        if (side) {
            if (cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess) return LORA_ERR_CUDA;
            st3 = side->s;
        }
        if (!rc) rc = launch_sgmv_plan(p, matrix, seg_starts, seg_adapter, S, T, plan, st3, true);
        if (!rc)
            rc = launch_sgmv_shrink(p, matrix, h_in, x, v, p->max_rank, seg_starts, seg_adapter, S, T, plan, st3, true);
        if (side && cudaEventRecord(side->join, side->s) != cudaSuccess) return LORA_ERR_CUDA;
        if (q_side && side && cudaStreamWaitEvent(st, side->join2, 0) != cudaSuccess) return LORA_ERR_CUDA;
        if (!rc) rc = launch_gemm_tc(p, h_in, h_out, x, W, y, T, st, matrix, tile_ad, v, p->max_rank, f8);
        // no side work is left unjoined, error or not
        if (side && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return LORA_ERR_CUDA;
        if (rc) return rc;
        return launch_sgmv_expand(p, matrix, h_out, v, p->max_rank, y, seg_starts, seg_adapter, S, T, plan, st,
                                  tile_ad);
    }
    rc = tc ? launch_gemm_tc(p, h_in, h_out, x, W, y, T, st, 0, nullptr, nullptr, 0, f8)
            : launch_base_gemm(p, h_in, h_out, x, W, y, T, st);
    if (rc) return rc;
    if ((rc = launch_shrink(p, matrix, h_in, x, v, p->max_rank, seg_starts, seg_adapter, S, T, st))) return rc;
    return launch_expand(p, matrix, h_out, v, p->max_rank, y, seg_starts, seg_adapter, S, T, st);
}
}  // namespace lora

using namespace lora;

extern "C" {

const char *lora_strerror(int status) {
    switch (status) {
        case LORA_OK: return "ok";
        case LORA_ERR_ARG: return "invalid argument";
        case LORA_ERR_POOL_FULL: return "adapter pool has too few free pages";
        case LORA_ERR_RANK: return "rank out of range (or ld_v below the pool's max_rank)";
        case LORA_ERR_NOT_LOADED: return "no adapter loaded in that entry";
        case LORA_ERR_CUDA: return "CUDA runtime error";
        case LORA_ERR_DEVICE_INDEX: return "device reported an invalid adapter id, segment table or wait timeout";
        case LORA_ERR_SHAPE: return "h_in/h_out mismatch with the matrix, or larger than a page";
        default: return "unknown status";
    }
}

unsigned long long lora_launch_count(void) { return g_launches.load(); }

int lora_pool_create(lora_pool **out, int dtype, int page_elems, int n_pages, int max_rank,
                     int n_matrices, int max_adapters) {
    if (!out) return LORA_ERR_ARG;
    *out = nullptr;
    if ((dtype != LORA_F32 && dtype != LORA_BF16) || page_elems <= 0 || page_elems % 8 != 0 ||
        n_pages <= 0 || max_rank <= 0 || max_rank > 1024 || n_matrices <= 0 || max_adapters <= 0)
        return LORA_ERR_ARG;
    lora_pool *p = new (std::nothrow) lora_pool();
    if (!p) return LORA_ERR_ARG;
    p->dtype = dtype;
    p->esize = dtype == LORA_F32 ? 4 : 2;
    p->page_elems = page_elems;
    p->n_pages = n_pages;
    p->max_rank = max_rank;
    p->n_matrices = n_matrices;
    p->max_adapters = max_adapters;
    p->rec_ints = (kRecHeader + 2 * max_rank + 3) & ~3;
    p->d_pages = p->d_table = nullptr;
    p->d_status = nullptr;
    p->h_stage = p->d_stage = nullptr;
    const size_t n_rec = (size_t)max_adapters * n_matrices;
    p->stage_bytes = stage_layout(p, max_rank).total;
    // a ring of up to kStageSlots slots, at most about kStageRingBytes of pinned memory (at least 2 slots)
    p->n_slots = (int)std::max<size_t>(2, std::min<size_t>(kStageSlots, kStageRingBytes / p->stage_bytes));
    p->next_slot = 0;
    int rc = LORA_OK;
    try {
        p->slot_done.assign(p->n_slots, nullptr);
    } catch (...) {
        delete p;
        return LORA_ERR_ARG;
    }
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaMalloc(&p->d_pages, (size_t)n_pages * page_elems * p->esize) != cudaSuccess ||
        cudaMalloc((void **)&p->d_table, n_rec * p->rec_ints * sizeof(int)) != cudaSuccess ||
        cudaMalloc((void **)&p->d_status, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&p->d_stage, p->stage_bytes * p->n_slots) != cudaSuccess ||
        cudaMallocHost(&p->h_stage, p->stage_bytes * p->n_slots) != cudaSuccess ||
        cudaMemset(p->d_table, 0xFF, n_rec * p->rec_ints * sizeof(int)) != cudaSuccess ||   // rank -1
        cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess)
        rc = LORA_ERR_CUDA;
    for (int i = 0; rc == LORA_OK && i < p->n_slots; ++i)
        if (cudaEventCreateWithFlags(&p->slot_done[i], cudaEventDisableTiming) != cudaSuccess) rc = LORA_ERR_CUDA;
    if (rc == LORA_OK && cudaDeviceSynchronize() != cudaSuccess) rc = LORA_ERR_CUDA;
    if (rc != LORA_OK) {
        cudaGetLastError();
        lora_pool_destroy(p);
        return rc;
    }
    try {
        p->free_pages.resize(n_pages);
        for (int i = 0; i < n_pages; ++i) p->free_pages[i] = n_pages - 1 - i;   // pop gives 0,1,2...
        p->host_table.assign(n_rec * p->rec_ints, -1);
        p->mat_h_in.assign(n_matrices, -1);
        p->mat_h_out.assign(n_matrices, -1);
        p->mat_n_ids.assign(n_matrices, 0);
        p->mat_max_rank.assign(n_matrices, 0);
    } catch (...) {
        lora_pool_destroy(p);
        return LORA_ERR_ARG;
    }
    *out = p;
    return LORA_OK;
}

int lora_pool_destroy(lora_pool *p) {
    if (!p) return LORA_OK;
    cudaDeviceSynchronize();
    if (p->d_pages) cudaFree(p->d_pages);
    if (p->d_table) cudaFree(p->d_table);
    if (p->d_status) cudaFree(p->d_status);
    if (p->d_stage) cudaFree(p->d_stage);
    if (p->h_stage) cudaFreeHost(p->h_stage);
    for (cudaEvent_t e : p->slot_done)
        if (e) cudaEventDestroy(e);
    for (auto &d : p->deferred)
        if (d.done) cudaEventDestroy(d.done);
    for (cudaEvent_t e : p->spare_events) cudaEventDestroy(e);
    cudaGetLastError();
    delete p;
    return LORA_OK;
}


// Pages of retired records whose event has completed go back to the free list.
static void reclaim(lora_pool *p) {
    size_t keep = 0;
    for (size_t i = 0; i < p->deferred.size(); ++i) {
        auto &d = p->deferred[i];
        if (cudaEventQuery(d.done) == cudaSuccess) {
            for (int pg : d.pages) p->free_pages.push_back(pg);
            p->spare_events.push_back(d.done);
        } else {
            cudaGetLastError();    // cudaErrorNotReady is not an error here
            if (keep != i) p->deferred[keep] = std::move(d);
            ++keep;
        }
    }
    p->deferred.resize(keep);
}

// Frees at least `need` pages if the retired ones allow it, waiting for their
// events oldest first; false if even all of them would not be enough.
static bool ensure_free(lora_pool *p, size_t need) {
    reclaim(p);
    size_t pending = 0;
    for (auto &d : p->deferred) pending += d.pages.size();
    if (p->free_pages.size() + pending < need) return false;
    while (p->free_pages.size() < need && !p->deferred.empty()) {
        cudaEventSynchronize(p->deferred.front().done);
        cudaGetLastError();
        reclaim(p);
    }
    return p->free_pages.size() >= need;
}

static cudaEvent_t take_event(lora_pool *p) {
    if (!p->spare_events.empty()) {
        cudaEvent_t e = p->spare_events.back();
        p->spare_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}

// Retires the pages of record `ri` (host mirror marked unloaded).  immediate:
// straight back to the free list (no kernel can still read them); else they
// wait for an event recorded now on `st`, after the table update that retired
// them.
static int retire_pages(lora_pool *p, size_t ri, bool immediate, cudaStream_t st) {
    int *rec = &p->host_table[ri * p->rec_ints];
    const int r = rec[0];
    rec[0] = -1;
    if (r <= 0) return LORA_OK;
    if (immediate) {
        for (int i = 0; i < 2 * r; ++i) p->free_pages.push_back(rec[kRecHeader + i]);
        return LORA_OK;
    }
    lora_pool::Deferred d;
    d.done = take_event(p);
    if (!d.done) return LORA_ERR_CUDA;
    try {
        d.pages.assign(rec + kRecHeader, rec + kRecHeader + 2 * r);
        if (cudaEventRecord(d.done, st) != cudaSuccess) throw 0;
        p->deferred.push_back(std::move(d));
    } catch (...) {
        cudaGetLastError();
        // the event could not be recorded: wait for the stream instead
        cudaStreamSynchronize(st);
        for (int i = 0; i < 2 * r; ++i) p->free_pages.push_back(rec[kRecHeader + i]);
        p->spare_events.push_back(d.done);
    }
    return LORA_OK;
}

// The next staging slot, once its previous copies have completed.
static int take_slot(lora_pool *p) {
    const int slot = p->next_slot;
    p->next_slot = (slot + 1) % p->n_slots;
    cudaEventSynchronize(p->slot_done[slot]);   // returns at once for an event never recorded
    cudaGetLastError();
    return slot;
}

static int check_load(const lora_pool *p, int adapter, int matrix, int rank, int h_in, int h_out, const void *A_T,
                      const void *B) {
    if (!p || adapter < 0 || adapter >= p->max_adapters || matrix < 0 || matrix >= p->n_matrices)
        return LORA_ERR_ARG;
    if (rank < 0 || rank > p->max_rank) return LORA_ERR_RANK;
    if (h_in <= 0 || h_out <= 0 || h_in % 8 || h_out % 8) return LORA_ERR_ARG;
    if (h_in > p->page_elems || h_out > p->page_elems) return LORA_ERR_SHAPE;
    if (p->mat_h_in[matrix] >= 0 && (p->mat_h_in[matrix] != h_in || p->mat_h_out[matrix] != h_out))
        return LORA_ERR_SHAPE;
    if (rank > 0 && (!A_T || !B)) return LORA_ERR_ARG;
    return LORA_OK;
}

// Stages one adapter in a slot and enqueues on `st`: the copy of its rows and
// page ids to the device, the scatter into its pages, the copy of its table
// record, and the slot's event.  The record copy comes last and is a plain
// copy, not a kernel, so a kernel launched after it on `st` -- even one that
// may start before the kernel ahead of it finishes (programmatic dependent
// launch) -- reads the new record, and the record points at written pages.
// Pages come from the free list (the caller made room); the host mirror is
// updated once everything is enqueued.
static int enqueue_load(lora_pool *p, size_t ri, int adapter, int matrix, int rank, float scale, int h_in, int h_out,
                        const void *A_T, const void *B, cudaStream_t st, int *slot_out) {
    const int slot = take_slot(p);
    const StageLayout L = stage_layout(p, p->max_rank);
    uint8_t *hs = (uint8_t *)p->h_stage + (size_t)slot * p->stage_bytes;
    uint8_t *ds = (uint8_t *)p->d_stage + (size_t)slot * p->stage_bytes;
    const int rba = h_in * p->esize, rbb = h_out * p->esize;
    if (rank > 0) {
        std::memcpy(hs, A_T, (size_t)rank * rba);
        std::memcpy(hs + (size_t)rank * rba, B, (size_t)rank * rbb);
    }
    LoadArgs *la = reinterpret_cast<LoadArgs *>(hs + L.args);
    la->rec_index = (int)ri;
    la->rank = rank;
    la->scale = scale;
    la->row_bytes_a = rba;
    la->row_bytes_b = rbb;
    for (int i = 0; i < 2 * rank; ++i) {
        la->ids[i] = p->free_pages.back();
        p->free_pages.pop_back();
    }
    int *hrec_stage = reinterpret_cast<int *>(hs + L.rec);
    for (int i = 0; i < p->rec_ints; ++i) hrec_stage[i] = -1;
    hrec_stage[0] = rank;
    std::memcpy(&hrec_stage[1], &scale, sizeof(int));
    hrec_stage[2] = hrec_stage[3] = 0;
    for (int i = 0; i < 2 * rank; ++i) hrec_stage[kRecHeader + i] = la->ids[i];
    cudaError_t e = cudaSuccess;
    if (rank > 0) {
        const size_t data_bytes = (size_t)rank * (rba + rbb);
        e = cudaMemcpyAsync(ds, hs, data_bytes, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ds + L.args, hs + L.args, offsetof(LoadArgs, ids) + sizeof(int) * 2 * rank,
                                cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) {
            load_scatter_kernel<<<2 * rank, 256, 0, st>>>(ds, (uint8_t *)p->d_pages,
                                                         (long long)p->page_elems * p->esize,
                                                         reinterpret_cast<const LoadArgs *>(ds + L.args));
            count_launch();
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->d_table + ri * p->rec_ints, hrec_stage, (size_t)p->rec_ints * sizeof(int),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(p->slot_done[slot], st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        for (int i = 2 * rank - 1; i >= 0; --i) p->free_pages.push_back(la->ids[i]);
        return LORA_ERR_CUDA;
    }
    int *hrec = &p->host_table[ri * p->rec_ints];
    std::memcpy(hrec, hrec_stage, (size_t)p->rec_ints * sizeof(int));
    p->mat_h_in[matrix] = h_in;
    p->mat_h_out[matrix] = h_out;
    if (adapter + 1 > p->mat_n_ids[matrix]) p->mat_n_ids[matrix] = adapter + 1;
    if (rank > p->mat_max_rank[matrix]) p->mat_max_rank[matrix] = rank;
    if (slot_out) *slot_out = slot;
    return LORA_OK;
}

int lora_pool_free_pages(const lora_pool *p) {
    if (!p) return -1;
    reclaim(const_cast<lora_pool *>(p));
    return (int)p->free_pages.size();
}

int lora_pool_load(lora_pool *p, int adapter, int matrix, int rank, float scale, int h_in, int h_out,
                   const void *A_T, const void *B, lora_stream stream) {
    int rc = check_load(p, adapter, matrix, rank, h_in, h_out, A_T, B);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t ri = (size_t)adapter * p->n_matrices + matrix;
    const int old_rank = p->host_table[ri * p->rec_ints];
    reclaim(p);
    size_t pending = 0;
    for (auto &d : p->deferred) pending += d.pages.size();
    if (p->free_pages.size() + pending + (old_rank > 0 ? 2 * old_rank : 0) < (size_t)2 * rank)
        return LORA_ERR_POOL_FULL;
    if (old_rank >= 0) {
        // Replacing: queued kernels may still read the old pages.
        if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ERR_CUDA;
        retire_pages(p, ri, true, st);
    }
    if (!ensure_free(p, (size_t)2 * rank)) return LORA_ERR_POOL_FULL;
    int slot = 0;
    if ((rc = enqueue_load(p, ri, adapter, matrix, rank, scale, h_in, h_out, A_T, B, st, &slot))) return rc;
    // The call returns with the adapter resident, for kernels on any stream.
    if (cudaEventSynchronize(p->slot_done[slot]) != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    return LORA_OK;
}

int lora_pool_load_async(lora_pool *p, int adapter, int matrix, int rank, float scale, int h_in, int h_out,
                         const void *A_T, const void *B, lora_stream stream) {
    int rc = check_load(p, adapter, matrix, rank, h_in, h_out, A_T, B);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t ri = (size_t)adapter * p->n_matrices + matrix;
    const int old_rank = p->host_table[ri * p->rec_ints];
    reclaim(p);
    size_t pending = 0;
    for (auto &d : p->deferred) pending += d.pages.size();
    // the replaced adapter's pages are retired on `st` after the new record is
    // published, so they cannot serve this load
    if (p->free_pages.size() + pending < (size_t)2 * rank) return LORA_ERR_POOL_FULL;
    if (!ensure_free(p, (size_t)2 * rank)) return LORA_ERR_POOL_FULL;
    std::vector<int> old;
    if (old_rank > 0) {
        const int *hrec = &p->host_table[ri * p->rec_ints];
        old.assign(hrec + kRecHeader, hrec + kRecHeader + 2 * old_rank);
    }
    if ((rc = enqueue_load(p, ri, adapter, matrix, rank, scale, h_in, h_out, A_T, B, st, nullptr))) return rc;
    if (!old.empty()) {
        lora_pool::Deferred d;
        d.done = take_event(p);
        if (!d.done || cudaEventRecord(d.done, st) != cudaSuccess) {
            cudaGetLastError();
            cudaStreamSynchronize(st);
            for (int pg : old) p->free_pages.push_back(pg);
            if (d.done) p->spare_events.push_back(d.done);
        } else {
            d.pages = std::move(old);
            p->deferred.push_back(std::move(d));
        }
    }
    return LORA_OK;
}

int lora_pool_prefetch(lora_pool *p, const lora_adapter_src *list, int n, lora_stream stream) {
    if (!p || n < 0 || (n > 0 && !list)) return LORA_ERR_ARG;
    int enqueued = 0;
    for (int i = 0; i < n; ++i) {
        const lora_adapter_src &e = list[i];
        if (e.adapter < 0 || e.adapter >= p->max_adapters || e.matrix < 0 || e.matrix >= p->n_matrices)
            return LORA_ERR_ARG;
        const size_t ri = (size_t)e.adapter * p->n_matrices + e.matrix;
        if (p->host_table[ri * p->rec_ints] >= 0) continue;      // already resident
        const int rc = lora_pool_load_async(p, e.adapter, e.matrix, e.rank, e.scale, e.h_in, e.h_out, e.A_T, e.B,
                                            stream);
        if (rc) return rc;
        ++enqueued;
    }
    return enqueued;
}

int lora_pool_unload(lora_pool *p, int adapter, int matrix) {
    if (!p || adapter < 0 || adapter >= p->max_adapters || matrix < 0 || matrix >= p->n_matrices)
        return LORA_ERR_ARG;
    const size_t ri = (size_t)adapter * p->n_matrices + matrix;
    if (p->host_table[ri * p->rec_ints] < 0) return LORA_ERR_NOT_LOADED;
    if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ERR_CUDA;
    const int minus1 = -1;
    if (cudaMemcpy(p->d_table + ri * p->rec_ints, &minus1, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    retire_pages(p, ri, true, nullptr);
    reclaim(p);
    return LORA_OK;
}

int lora_pool_unload_async(lora_pool *p, int adapter, int matrix, lora_stream stream) {
    if (!p || adapter < 0 || adapter >= p->max_adapters || matrix < 0 || matrix >= p->n_matrices)
        return LORA_ERR_ARG;
    const size_t ri = (size_t)adapter * p->n_matrices + matrix;
    if (p->host_table[ri * p->rec_ints] < 0) return LORA_ERR_NOT_LOADED;
    cudaStream_t st = (cudaStream_t)stream;
    const int slot = take_slot(p);
    int *hrank = reinterpret_cast<int *>((uint8_t *)p->h_stage + (size_t)slot * p->stage_bytes +
                                         stage_layout(p, p->max_rank).rec);
    *hrank = -1;
    if (cudaMemcpyAsync(p->d_table + ri * p->rec_ints, hrank, sizeof(int), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaEventRecord(p->slot_done[slot], st) != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    return retire_pages(p, ri, false, st);
}

int lora_get_error(lora_pool *p, int *device_status) {
    if (device_status) *device_status = 0;
    if (!p) return LORA_ERR_ARG;
    int word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    if (device_status) *device_status = word;
    return word ? LORA_ERR_DEVICE_INDEX : LORA_OK;
}

// ---------------------------------------------------------------------------
// Compute entry points: argument checks, then the launchers.
// ---------------------------------------------------------------------------
static int check_common(const lora_pool *p, int S, int T) {
    if (!p || T < 0 || S < 0) return LORA_ERR_ARG;
    if (S == 0 && T > 0) return LORA_ERR_ARG;
    return LORA_OK;
}

int lora_sgmv_shrink(lora_pool *p, int matrix, const void *x, float *v, int ld_v, const int *seg_starts,
                     const int *seg_adapter, int S, int T, lora_stream stream) {
    int rc = check_common(p, S, T);
    if (rc) return rc;
    int h_in, h_out;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (ld_v < p->max_rank) return LORA_ERR_RANK;
    if (T == 0) return LORA_OK;
    if (!x || !v || !seg_starts || !seg_adapter || !aligned16(x) || !aligned16(v)) return LORA_ERR_ARG;
    return launch_shrink(p, matrix, h_in, x, v, ld_v, seg_starts, seg_adapter, S, T, (cudaStream_t)stream);
}

int lora_sgmv_expand(lora_pool *p, int matrix, const float *v, int ld_v, void *y, const int *seg_starts,
                     const int *seg_adapter, int S, int T, lora_stream stream) {
    int rc = check_common(p, S, T);
    if (rc) return rc;
    int h_in, h_out;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (ld_v < p->max_rank) return LORA_ERR_RANK;
    if (T == 0) return LORA_OK;
    if (!y || !v || !seg_starts || !seg_adapter || !aligned16(y) || !aligned16(v)) return LORA_ERR_ARG;
    return launch_expand(p, matrix, h_out, v, ld_v, y, seg_starts, seg_adapter, S, T, (cudaStream_t)stream);
}

int lora_bgmv(lora_pool *p, int matrix, const void *x, void *y, const int *token_adapter, int T,
              lora_stream stream) {
    if (!p || T < 0) return LORA_ERR_ARG;
    int h_in, h_out, rc;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (T == 0) return LORA_OK;
    if (!x || !y || !token_adapter || !aligned16(x) || !aligned16(y)) return LORA_ERR_ARG;
    return launch_bgmv(p, matrix, h_in, h_out, x, y, token_adapter, T, (cudaStream_t)stream);
}

size_t lora_layer_forward_workspace_size(const lora_pool *p, int matrix, int S, int T) {
    int h_in, h_out;
    if (!p || T < 0 || S < 0 || matrix_dims(p, matrix, &h_in, &h_out)) return 0;
    return (size_t)T * p->max_rank * sizeof(float) + sgmv_plan_bytes(p, matrix, T) + 256;
}

int lora_layer_forward(lora_pool *p, int matrix, const void *x, const void *W, void *y,
                       const int *seg_starts, const int *seg_adapter, int S, int T, void *workspace,
                       size_t ws_bytes, lora_stream stream) {
    int rc = check_common(p, S, T);
    if (rc) return rc;
    int h_in, h_out;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (T == 0) return LORA_OK;
    if (!x || !W || !y || !seg_starts || !seg_adapter || !workspace || !aligned16(x) || !aligned16(W) ||
        !aligned16(y) || !aligned16(workspace))
        return LORA_ERR_ARG;
    if (ws_bytes < lora_layer_forward_workspace_size(p, matrix, S, T)) return LORA_ERR_ARG;
    return layer_forward_impl(p, matrix, h_in, h_out, x, W, y, seg_starts, seg_adapter, S, T,
                              static_cast<float *>(workspace), (cudaStream_t)stream);
}

}  // extern "C"
