// Shared base product of the adapted layer on the 5th-generation tensor cores:
//
//   y[t][n] = sum_k x[t][k] W[n][k]
//
// The base term is computed once for the whole mixed batch, as a single
// matmul shared by every request ("Multi-LoRA Serving", section "The kernel
// trick: gather, do not merge").
// The fused variant also adds the low-rank term s * v . B_a of every M-tile
// whose 128 rows share one adapter a into the same accumulator (v from the
// tensor-core shrink below); the other rows get theirs from the SGMV expand.
//
// Structure: a persistent kernel, one CTA per SM, 128 x 256 output tiles,
// K in steps of 64.  Warp 0 (one lane) streams x and W tiles into a 4-stage
// shared-memory ring with TMA (128-byte swizzle); warp 1
// (one lane) issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) into one of
// two TMEM accumulators (2 x 256 columns) and commits each ring slot back to
// the producer and each finished accumulator to the epilogue; warps 2-5 read
// the accumulator with tcgen05.ld (each warp its 32-lane TMEM sub-partition,
// one row per thread), round to bf16 and store, and in the fused variant
// stage the next uniform tile's s * v and B operands (32 ranks per round,
// 64-byte swizzle, 32 KB beside the ring).  The two accumulators
// let the epilogue of one tile overlap the main loop of the next.
//
// Every mbarrier wait is bounded (by the global timer); a wait that gives up
// sets LORA_DEV_WAIT_TIMEOUT, makes the other roles stop, waits (bounded)
// for its own copies and MMAs in flight, and the CTA frees its TMEM.
#include <cudaTypedefs.h>

#include <algorithm>

#include "internal.cuh"
#include "tc_common.cuh"

namespace lora {
namespace {

using namespace tc;

constexpr int BM = kFuseTileRows, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreadsTC = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr uint32_t IDESC_F8 = idesc_e4m3_f32(BM, BN);   // FP8 base: K-blocks of 128 e4m3 (the same 128 bytes)

// The fused tile's low-rank term enters the accumulator in rounds of kRound ranks,
// staged K-major with 64-byte swizzling; 32-rank rounds keep the operands at
// 32 KB, which leaves room for a 4-stage ring (4 x 48 KB) in 227 KB.
constexpr int kRound = 32;
constexpr int kMaxRounds = (kFuseMaxRank + kRound - 1) / kRound;
constexpr int A2_BYTES = BM * kRound * 2;   // s * v tile, one round (high or residual part)
constexpr int B2_BYTES = BN * kRound * 2;   // B rows of the tile's columns, transposed to K-major

struct LayerTcParams {
    int T, N, K;
    int num_m, num_n, num_k, num_tiles;
    __nv_bfloat16 *y;
    int *status;
    // adapter term for uniform M-tiles (fused variant only)
    const int *tile_ad;     // per M-tile: adapter whose term is added here, or -1
    PoolView pv;
    int m;
    const float *v;         // [T][ld_v]: x . A_a of the fused tiles' rows
    int ld_v;
    // FP8 base (FP8 variant): the accumulator holds sum_k q[t][k] W8[n][k]; row t is
    // scaled by sx[t] * w_scale, and the fused tiles' low-rank operand enters divided by it
    const float *sx;
    float w_scale;
};

template <int ST>
struct Ctrl {
    uint64_t full[ST];
    uint64_t empty[ST];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t aready;      // one round of a tile's adapter operands is in shared memory
    uint64_t aconsumed;   // the MMAs of that round have read it
    uint32_t tmem_base;
    int abort;
    int akpad;            // K of the staged round (0: the tile has no adapter term)
    int arounds;          // rounds of that tile (set with round 0)
};

// Byte offset of 16-byte chunk c of row `row` in a K-major tile with 128-byte
// swizzling (8-row, 1024-byte atoms; chunk index XOR row-in-atom) -- the
// layout TMA writes and the UMMA descriptor reads.
__device__ __forceinline__ uint32_t swz128(int row, int c) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + (((c ^ row) & 7) << 4));
}

// Epilogue warps (128 threads) stage round `round` (ranks kRound*round ..
// +kRound-1) of the adapter term's operands of a tile in two steps: its global
// loads into registers (load_round), then the bf16 conversion and the
// swizzled shared-memory stores (store_round).  A2hi/A2lo: s * v of the tile's
// rows (bf16 high part / residual), K-major; B2: row n holds B_a[j][n0 + n]
// (the B rows transposed), K-major.  The next round's loads are issued as
// soon as a round is handed to the MMA warp, so they overlap its MMAs.
// What round 0 of a tile looks up for every round of it (one thread's share):
// the adapter's rank and scale and the B page ids of ranks lane + kRound * rd.
struct FillCache {
    int r;
    float s;
    int page[kMaxRounds];
};

// One thread's share of a round: its row's v values and its rank's B columns.
struct RoundRegs {
    float4 v[kRound / 4];
    uint4 b[8];
};

// Rank, scale and page ids of the tile's adapter (round 0 only).
__device__ __forceinline__ void lookup_adapter(const LayerTcParams &p, int tile, int lane, FillCache &fc) {
    const int mb = tile % p.num_m;
    const int a = p.tile_ad[mb];
    fc.r = 0;
    fc.s = 0.f;
    if (a >= 0 && a < p.pv.max_adapters) {
        const int *rec = p.pv.table + ((long long)a * p.pv.n_matrices + p.m) * p.pv.rec_ints;
        int r = rec[0];
        if (r < 1 || r > kFuseMaxRank || r > p.ld_v) r = 0;
        fc.r = r;
        if (r > 0) fc.s = __int_as_float(rec[1]);
#pragma unroll
        for (int rd = 0; rd < kMaxRounds; ++rd) {
            const int j = lane + kRound * rd;
            const int pg = j < r ? rec[kRecHeader + r + j] : 0;
            fc.page[rd] = pg < 0 ? 0 : (pg >= p.pv.n_pages ? p.pv.n_pages - 1 : pg);
        }
    }
}

__device__ __forceinline__ void load_round(const LayerTcParams &p, int tile, int round, const FillCache &fc,
                                           int ethr, RoundRegs &g) {
    static_assert(kRound == 32, "one rank of a round per lane");
    const int mb = tile % p.num_m, nb = tile / p.num_m;
    const int lane = ethr & 31, w = ethr >> 5;
    const int j0 = round * kRound, rn = max(0, min(kRound, fc.r - j0));
    const int kpad = (rn + 15) & ~15;
    // v: row ethr of the tile
    const int row = mb * BM + ethr;
    const bool live = row < p.T;
    const float *vrow = p.v + (long long)(live ? row : 0) * p.ld_v + j0;
    const bool vec = (p.ld_v & 3) == 0;
#pragma unroll
    for (int c = 0; c < kRound / 4; ++c) {
        g.v[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && c * 4 < rn) {
            if (vec) {                       // ranks past rn hold zeros after the conversion (float4 over-read)
                g.v[c] = *reinterpret_cast<const float4 *>(vrow + c * 4);
            } else {
                float e[4] = {0.f, 0.f, 0.f, 0.f};
                for (int u = 0; u < 4; ++u)
                    if (c * 4 + u < rn) e[u] = vrow[c * 4 + u];
                g.v[c] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
    }
    // B: rank `lane` of the round, 8-column groups w, w + 4, ... of the tile's columns
    int page = 0;
#pragma unroll
    for (int rd = 0; rd < kMaxRounds; ++rd)
        if (rd == round) page = fc.page[rd];
    const __nv_bfloat16 *prow = page_row<__nv_bfloat16>(p.pv, page);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int col = nb * BN + (w + 4 * q) * 8;
        g.b[q] = (lane < rn && lane < kpad && col < p.N) ? *reinterpret_cast<const uint4 *>(prow + col)
                                                         : make_uint4(0, 0, 0, 0);
    }
}

// Writes the round's operands; returns the tile's number of rounds.
template <int ST>
__device__ int store_round(const FillCache &fc, int round, const RoundRegs &g, uint8_t *a2hi, uint8_t *a2lo,
                           uint8_t *b2, Ctrl<ST> *ctrl, int ethr, float row_mul) {
    const int lane = ethr & 31, w = ethr >> 5;
    const int rounds = (fc.r + kRound - 1) / kRound;
    const int j0 = round * kRound, rn = max(0, min(kRound, fc.r - j0));
    const int kpad = (rn + 15) & ~15;
    if (ethr == 0) {
        ctrl->akpad = kpad;
        if (round == 0) ctrl->arounds = rounds;
    }
    if (kpad == 0) return rounds;
    const float s = fc.s * row_mul;
#pragma unroll
    for (int c = 0; c < kRound / 8; ++c) {
        if (c * 8 >= kpad) break;
        const float vv[8] = {g.v[2 * c].x, g.v[2 * c].y, g.v[2 * c].z, g.v[2 * c].w,
                             g.v[2 * c + 1].x, g.v[2 * c + 1].y, g.v[2 * c + 1].z, g.v[2 * c + 1].w};
        uint4 hi4, lo4;
        __nv_bfloat16 *hi = reinterpret_cast<__nv_bfloat16 *>(&hi4);
        __nv_bfloat16 *lo = reinterpret_cast<__nv_bfloat16 *>(&lo4);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = c * 8 + e;
            const float val = j < rn ? s * vv[e] : 0.f;
            hi[e] = __float2bfloat16_rn(val);
            lo[e] = __float2bfloat16_rn(val - __bfloat162float(hi[e]));
        }
        *reinterpret_cast<uint4 *>(a2hi + swz64(ethr, c)) = hi4;
        *reinterpret_cast<uint4 *>(a2lo + swz64(ethr, c)) = lo4;
    }
    if (lane < kpad) {
        const int j = lane;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int n0 = (w + 4 * q) * 8;
            const __nv_bfloat16 *e8 = reinterpret_cast<const __nv_bfloat16 *>(&g.b[q]);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                *reinterpret_cast<__nv_bfloat16 *>(b2 + swz64(n0 + e, j >> 3) + (j & 7) * 2) = e8[e];
        }
    }
    return rounds;
}

template <int ST>
__device__ __forceinline__ void give_up(Ctrl<ST> *c, int *status) {
    c->abort = 1;
    __threadfence_block();
    flag(status, LORA_DEV_WAIT_TIMEOUT);
}

template <int STAGES, bool FUSE, bool FP8>
__global__ void __launch_bounds__(kThreadsTC, 1)
    layer_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                         LayerTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *a2hi = smem + STAGES * STAGE_BYTES;          // used when FUSE
    uint8_t *a2lo = a2hi + A2_BYTES;
    uint8_t *b2 = a2lo + A2_BYTES;
    Ctrl<STAGES> *ctrl = reinterpret_cast<Ctrl<STAGES> *>(smem + STAGES * STAGE_BYTES + (FUSE ? 2 * A2_BYTES + B2_BYTES : 0));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort = &ctrl->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctrl->full[s], 1);
            mbar_init(&ctrl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctrl->tfull[b], 1);
            mbar_init(&ctrl->tempty[b], 4);
        }
        mbar_init(&ctrl->drain, 1);
        mbar_init(&ctrl->aready, 4);
        mbar_init(&ctrl->aconsumed, 1);
        ctrl->abort = 0;
        ctrl->akpad = 0;
        ctrl->arounds = 0;
        mbar_fence_init();
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
    }
    if (warp == 1) {
        tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int last_par[STAGES];
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                const int mb = tile % p.num_m, nb = tile / p.num_m;
                for (int kb = 0; kb < p.num_k; ++kb) {
                    if (!wait_phase(&ctrl->empty[stage], phase ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(&ctrl->full[stage], STAGE_BYTES);
                    const int kx = kb * (FP8 ? 2 * BK : BK);      // K-block origin in elements (128 bytes)
                    tma_load_2d(sa, &tmx, kx, mb * BM, &ctrl->full[stage]);
                    tma_load_2d(sa + A_BYTES, &tmw, kx, nb * BN, &ctrl->full[stage]);
                    last_par[stage] = (int)phase;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                give_up(ctrl, p.status);
                for (int s = 0; s < STAGES; ++s)       // copies still landing must land before exit
                    if (last_par[s] >= 0) wait_phase(&ctrl->full[s], (uint32_t)last_par[s], nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            uint32_t n_ready = 0;          // aready phases consumed so far
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++local) {
                const int b = local & 1;
                const uint32_t u = (uint32_t)(local >> 1);
                if (!wait_phase(&ctrl->tempty[b], (u & 1u) ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = 0; kb < p.num_k; ++kb) {
                    if (!wait_phase(&ctrl->full[stage], phase, abort)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t a0 = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {      // 32 bytes of K per MMA: 16 bf16 or 32 e4m3
                        if (FP8)
                            mma_f8(d, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), IDESC_F8,
                                   (kb | k) != 0);
                        else
                            mma_bf16(d, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), IDESC,
                                     (kb | k) != 0);
                    }
                    mma_commit(&ctrl->empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok && FUSE) {
                    // the tile's low-rank term, kRound ranks per round:
                    // acc += (s v)_hi . B + (s v)_lo . B over the round's ranks
                    const uint32_t ah = smem_u32(a2hi), al = smem_u32(a2lo), bb = smem_u32(b2);
                    int rounds = 1;
                    for (int rd = 0; rd < rounds && ok; ++rd) {
                        if (rd > 0) mma_commit(&ctrl->aconsumed);     // round rd-1's operands may be replaced
                        if (!wait_phase(&ctrl->aready, n_ready++ & 1u, abort)) {
                            ok = false;
                            break;
                        }
                        fence_after_sync();
                        if (rd == 0) rounds = ctrl->arounds;
                        const int kpad = ctrl->akpad;
                        for (int kk = 0; kk < kpad / 16; ++kk) {
                            mma_bf16(d, desc_kmajor_sw64(ah + kk * 32), desc_kmajor_sw64(bb + kk * 32), IDESC, 1);
                            mma_bf16(d, desc_kmajor_sw64(al + kk * 32), desc_kmajor_sw64(bb + kk * 32), IDESC, 1);
                        }
                    }
                    if (!ok) break;
                }
                if (ok) mma_commit(&ctrl->tfull[b]);
            }
            if (!ok) give_up(ctrl, p.status);
            mma_commit(&ctrl->drain);                  // all MMAs of this CTA complete before TMEM is freed
            wait_phase(&ctrl->drain, 0, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int sub = warp & 3;                      // TMEM sub-partition this warp may access
        const int ethr = (warp - 2) * 32 + lane;       // 0..127
        uint32_t n_consumed = 0;                       // aconsumed phases waited for so far
        bool staged_ok = true;
        // stage every round of a tile's adapter operands, handing each to the MMA warp
        auto stage_tile = [&](int t) {
            FillCache fc;
            RoundRegs g;
            lookup_adapter(p, t, lane, fc);
            float row_mul = 1.f;       // FP8: the accumulator is in units of sx[row] * w_scale
            if (FP8) {
                const int row = (t % p.num_m) * BM + ethr;
                row_mul = 1.f / ((row < p.T ? p.sx[row] : 1.f) * p.w_scale);
            }
            const int rounds = max(1, (fc.r + kRound - 1) / kRound);
            load_round(p, t, 0, fc, ethr, g);
            for (int rd = 0; rd < rounds; ++rd) {
                if (rd > 0) {
                    const bool okc = wait_phase(&ctrl->aconsumed, n_consumed++ & 1u, abort);
                    if (!__all_sync(0xffffffffu, okc)) {
                        if (lane == 0) give_up(ctrl, p.status);
                        staged_ok = false;
                        return;
                    }
                }
                store_round<STAGES>(fc, rd, g, a2hi, a2lo, b2, ctrl, ethr, row_mul);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->aready);
                if (rd + 1 < rounds) load_round(p, t, rd + 1, fc, ethr, g);   // overlaps round rd's MMAs
            }
        };
        if (FUSE && (int)blockIdx.x < p.num_tiles) stage_tile(blockIdx.x);
        int local = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
            const int b = local & 1;
            const uint32_t u = (uint32_t)(local >> 1);
            const bool ok = wait_phase(&ctrl->tfull[b], u & 1u, abort);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) give_up(ctrl, p.status);
                break;
            }
            fence_after_sync();
            const int mb = tile % p.num_m, nb = tile / p.num_m;
            const int row = mb * BM + sub * 32 + lane;
            const float out_mul = FP8 && row < p.T ? p.sx[row] * p.w_scale : 1.f;

            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = nb * BN + c * 32;
                float f[32];
                __syncwarp();
                tmem_ld32(tmem + (uint32_t)(b * BN + c * 32) + ((uint32_t)(sub * 32) << 16), f);
                if (col0 >= p.N || row >= p.T) continue;
                if (FP8) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] *= out_mul;
                }
                uint4 *dst = reinterpret_cast<uint4 *>(p.y + (long long)row * p.N + col0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 o;
                    __nv_bfloat162 *ho = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                    for (int e = 0; e < 4; ++e) ho[e] = __floats2bfloat162_rn(f[q * 8 + 2 * e], f[q * 8 + 2 * e + 1]);
                    dst[q] = o;
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->tempty[b]);
            // the tile's adapter MMAs are complete (tfull): stage the next tile's operands
            if (FUSE && staged_ok && tile + (int)gridDim.x < p.num_tiles) stage_tile(tile + gridDim.x);
        }
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Shrink on the tensor cores for tiles of up to 128 rows that share one
// adapter: v[rows] = x[rows] . A_a^T, M = 128, N = r (<= kFuseMaxRank),
// K = h_in.  At rank 128 that is 256 flops per x element, more than
// warp-level MMAs sustain at HBM rate.  A tile is either an M-tile of the
// fused layer whose rows all use one adapter (the plan's tile array), or
// 128 consecutive rows of one long segment of a segment table (long
// prefill segments, encoder sequences).
//
// Grid (tiles, K splits); the nsplit CTAs of a tile form a cluster.
// Through a ring of shared-memory stages, warp 0 streams x (one 128 x 64 TMA
// box, 128-byte swizzle) and warps 2-5 the r page rows of A_a (16-byte
// cp.async into the same swizzled K-major layout, each thread's copies
// arriving on the stage's mbarrier as they land); warp 1 issues tcgen05.mma
// into TMEM.  The splits' partial accumulators are then reduce-scattered over
// the cluster: split s owns a quarter of the rank columns, the others read
// that part of their accumulators out of TMEM and send it with asynchronous
// remote stores counted on its mbarrier, and it adds the parts in split order
// and stores its columns of v.  Rows of a tile past its end (another
// segment's, or past T) are computed and dropped.
// ---------------------------------------------------------------------------
constexpr int SK_MAX_STAGES = 8;
constexpr int SK_X_BYTES = BM * BK * 2;
constexpr uint32_t SK_TMEM_COLS = kFuseMaxRank;

struct ShrinkTcParams {
    int T, num_k, nsplit;
    int stages, stage_bytes;   // ring depth; bytes of one stage (x tile + npad_max A rows)
    int *tile_ad;              // fused layer: per M-tile adapter, written here (-1: tile not fused); else nullptr
    const int *seg_starts, *seg_adapter;   // the batch's segment table
    int S, min_rows;           // segment tables: tiles of segments with >= min_rows rows
    int n_ids;                 // fused layer: adapter ids below this may be loaded on the matrix
    PoolView pv;
    int m;
    float *v;
    int ld_v;
    int *status;
};

struct SkCtrl {
    uint64_t full[SK_MAX_STAGES];
    uint64_t empty[SK_MAX_STAGES];
    uint64_t done;    // every MMA of the CTA complete
    uint64_t ready;   // every other CTA of the cluster may receive
    uint64_t recv;    // every other split's share of this CTA's columns has arrived
    uint32_t tmem_base;
    int abort;
    int tile[3];      // adapter, first row, rows
    int wsum[kThreadsTC / 32 + 1];
    int page[kFuseMaxRank];
};

__device__ __forceinline__ void cp_async16_sk(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival was counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_sk(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_wait_all_sk() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_rank_sk() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_sk(const void *p, int rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ void remote_arrive_sk(uint64_t *bar, int rank) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(mapa_sk(bar, rank)) : "memory");
}
// 16 bytes into the first CTA's shared memory, counted on its barrier `bar`.
__device__ __forceinline__ void st_async16_sk(uint32_t dst, uint32_t bar, float a, float b, float c, float d) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(dst),
                 "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
                 "r"(bar)
                 : "memory");
}
// Bounded cluster-scope acquire wait (the remote arrivals and transactions release at cluster scope).
__device__ __forceinline__ bool wait_cluster_sk(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const unsigned long long t0 = now_ns();
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
            if (abort && *abort) return false;
            if (now_ns() - t0 > kTimeoutNs) return false;
        }
    }
}

// Fused layer: the adapter whose term M-tile `mb` gets inside the GEMM (its
// rows all use that adapter, of rank 1..kFuseMaxRank), or -1.  All threads
// call it; the segment table is staged in `stage` (2 S + 1 ints of shared
// memory), then warp 0 decides with uniform_tile_adapter -- the function the
// rows and plan kernels apply to every tile -- and the first CTA of the cluster
// publishes the result in tile_ad for the GEMM and the expand that follow.
__device__ int layer_tile_sk(const ShrinkTcParams &p, int mb, int split, int *stage, SkCtrl *ctrl) {
    int *sb = stage, *sa = stage + p.S + 1;
    for (int s = threadIdx.x; s <= p.S; s += kThreadsTC) sb[s] = min(max(p.seg_starts[s], 0), p.T);
    for (int s = threadIdx.x; s < p.S; s += kThreadsTC) sa[s] = p.seg_adapter[s];
    __syncthreads();
    if (threadIdx.x < 32) {
        const int r0 = mb * BM, r1 = min(p.T, r0 + BM);
        int a = uniform_tile_adapter(sb, sa, p.S, p.n_ids, r0, r1);
        if (threadIdx.x == 0) {
            if (a >= 0) {
                const int r = a < p.pv.max_adapters
                                  ? p.pv.table[((long long)a * p.pv.n_matrices + p.m) * p.pv.rec_ints]
                                  : -1;
                if (r < 1 || r > kFuseMaxRank || r > p.ld_v) a = -1;
            }
            if (split == 0) p.tile_ad[mb] = a;
            ctrl->tile[0] = a;
        }
    }
    __syncthreads();
    const int a = ctrl->tile[0];
    __syncthreads();    // the staged table (aliasing the ring) is no longer read
    return a;
}

// Segment tables: tile `t` among the 128-row pieces of the segments with at
// least min_rows rows.  All threads call it; ctrl->tile gets the result.
__device__ void segment_tile_sk(const ShrinkTcParams &p, int t, int *scan, SkCtrl *ctrl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kThreadsTC / 32;
    const int per = (p.S + kThreadsTC - 1) / kThreadsTC;
    const int lo = min(p.S, tid * per), hi = min(p.S, lo + per);
    int sum = 0;
    for (int s = lo; s < hi; ++s) {
        const int b = min(max(p.seg_starts[s], 0), p.T), e = min(max(p.seg_starts[s + 1], 0), p.T);
        const int n = e - b >= p.min_rows ? (e - b + BM - 1) / BM : 0;
        scan[s] = n;
        sum += n;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) ctrl->wsum[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            const int v = ctrl->wsum[w];
            ctrl->wsum[w] = run;
            run += v;
        }
        ctrl->wsum[NW] = run;
    }
    __syncthreads();
    int run = ctrl->wsum[warp] + inc - sum;
    for (int s = lo; s < hi; ++s) {
        const int v = scan[s];
        scan[s] = run;
        run += v;
    }
    __syncthreads();
    if (tid == 0) {
        int a = -1, row0 = 0, rows = 0;
        if (t < ctrl->wsum[NW]) {
            int l = 0, h = p.S - 1;            // last segment whose first tile index <= t
            while (l < h) {
                const int mid = (l + h + 1) >> 1;
                if (scan[mid] <= t) l = mid; else h = mid - 1;
            }
            const int b = min(max(p.seg_starts[l], 0), p.T), e = min(max(p.seg_starts[l + 1], 0), p.T);
            a = p.seg_adapter[l];
            row0 = b + (t - scan[l]) * BM;
            rows = min(BM, e - row0);
        }
        ctrl->tile[0] = a;
        ctrl->tile[1] = row0;
        ctrl->tile[2] = rows;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreadsTC, 1)
    shrink_tc_kernel(const __grid_constant__ CUtensorMap tmx, ShrinkTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SkCtrl *ctrl = reinterpret_cast<SkCtrl *>(smem + p.stages * p.stage_bytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = p.nsplit > 1 ? (int)cluster_rank_sk() : 0;
    int a, row0, rows;
    if (p.tile_ad) {
        row0 = blockIdx.x * BM;
        rows = min(BM, p.T - row0);
        a = layer_tile_sk(p, blockIdx.x, split, reinterpret_cast<int *>(smem), ctrl);
    } else {
        segment_tile_sk(p, blockIdx.x, reinterpret_cast<int *>(smem), ctrl);
        a = ctrl->tile[0];
        row0 = ctrl->tile[1];
        rows = ctrl->tile[2];
    }
    // every CTA of the cluster resolves the same tile, so they leave together
    if (a < 0 || a >= p.pv.max_adapters || rows <= 0) return;
    const int *rec = p.pv.table + ((long long)a * p.pv.n_matrices + p.m) * p.pv.rec_ints;
    const int r = rec[0];
    if (r < (p.tile_ad ? 1 : kShrinkTcSegMinRank) || r > kFuseMaxRank || r > p.ld_v) return;   // the warp-MMA shrink takes it
    const int npad = (r + 15) & ~15;
    const uint32_t idesc = idesc_bf16_f32(BM, npad);
    const int kb0 = split * p.num_k / p.nsplit, kb1 = (split + 1) * p.num_k / p.nsplit;
    volatile int *abort = &ctrl->abort;
    const int ST = p.stages;

    __syncthreads();                       // the segment scan (aliasing the ring) is done
    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&ctrl->full[s], 129);    // the x TMA (with its bytes) + 128 threads' A copies
            mbar_init(&ctrl->empty[s], 1);
        }
        mbar_init(&ctrl->done, 1);
        mbar_init(&ctrl->ready, p.nsplit > 1 ? p.nsplit - 1 : 1);   // every other split's ring is drained
        mbar_init(&ctrl->recv, 1);
        ctrl->abort = 0;
        mbar_fence_init();
        prefetch_tmap(&tmx);
    }
    for (int j = threadIdx.x; j < r; j += kThreadsTC) {
        const int pg = rec[kRecHeader + j];
        ctrl->page[j] = pg < 0 ? 0 : (pg >= p.pv.n_pages ? p.pv.n_pages - 1 : pg);
    }
    if (warp == 1) {
        tmem_alloc(&ctrl->tmem_base, SK_TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (p.nsplit > 1) asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    const uint32_t tmem = ctrl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ x producer (one lane)
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                const int i = kb - kb0, stage = i % ST;
                const uint32_t phase = (uint32_t)(i / ST) & 1u;
                if (!wait_phase(&ctrl->empty[stage], phase ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&ctrl->full[stage], (uint32_t)SK_X_BYTES);
                tma_load_2d(smem + stage * p.stage_bytes, &tmx, kb * BK, row0, &ctrl->full[stage]);
                ++issued;
            }
            if (!ok) {
                ctrl->abort = 1;
                __threadfence_block();
                flag(p.status, LORA_DEV_WAIT_TIMEOUT);
                // the x copies still landing must land before exit (the A copies arrive by themselves)
                for (int i = issued > ST ? issued - ST : 0; i < issued; ++i)
                    wait_phase(&ctrl->full[i % ST], (uint32_t)(i / ST) & 1u, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                const int i = kb - kb0, stage = i % ST;
                const uint32_t phase = (uint32_t)(i / ST) & 1u;
                if (!wait_phase(&ctrl->full[stage], phase, abort)) {
                    ok = false;
                    break;
                }
                fence_proxy_async();                  // the A rows came through the generic proxy
                fence_after_sync();
                const uint32_t a0 = smem_u32(smem + stage * p.stage_bytes);
                const uint32_t b0 = a0 + SK_X_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    mma_bf16(tmem, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), idesc,
                             (i | k) != 0);
                mma_commit(&ctrl->empty[stage]);
            }
            if (!ok) {
                ctrl->abort = 1;
                __threadfence_block();
                flag(p.status, LORA_DEV_WAIT_TIMEOUT);
            }
            mma_commit(&ctrl->done);                 // every MMA of this CTA complete before TMEM is read or freed
            wait_phase(&ctrl->done, 0, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ warps 2..5: A producers, then epilogue
        // thread t: 16-byte chunk c = t & 7 of rank rows (t >> 3) + 16 q.  Each
        // thread's copies of a stage arrive on the stage's barrier when they land.
        const int t = threadIdx.x - 64, c = t & 7;
        for (int kb = kb0; kb < kb1; ++kb) {
            const int i = kb - kb0, stage = i % ST;
            const uint32_t phase = (uint32_t)(i / ST) & 1u;
            if (!wait_phase(&ctrl->empty[stage], phase ^ 1u, abort)) break;
            const uint32_t sa = smem_u32(smem + stage * p.stage_bytes + SK_X_BYTES);
            for (int j = t >> 3; j < r; j += 16)
                cp_async16_sk(sa + swz128(j, c), page_row<__nv_bfloat16>(p.pv, ctrl->page[j]) + kb * BK + c * 8);
            cp_async_arrive_sk(&ctrl->full[stage]);
        }
        cp_wait_all_sk();                            // nothing lands after the CTA exits

        const int sub = warp & 3;
        const int lrow = sub * 32 + lane;            // row of the tile (TMEM lane)
        bool ok = wait_phase(&ctrl->done, 0, nullptr) && !*abort;
        ok = __all_sync(0xffffffffu, ok);
        if (ok) fence_after_sync();
        // reduce-scatter over the cluster: split s owns columns [s q, (s + 1) q) of the
        // partial sums, receives every other split's share of them and writes that part of v
        const int ns = p.nsplit;
        const int q = ((npad + ns - 1) / ns + 3) & ~3;   // columns per split (multiple of 4)
        const int pitch = q + 4;                         // floats per received row (16-byte aligned)
        auto col_lo = [&](int t) { return min(npad, t * q); };
        float *recvbuf = reinterpret_cast<float *>(smem);   // [ns][BM][pitch] by sender, over the drained ring
        const int my_lo = col_lo(split), my_hi = col_lo(split + 1);
        if (ns > 1) {
            asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
            // this CTA's ring is drained (all MMAs complete, all copies landed): open it to the others
            if (threadIdx.x == 64) {
                mbar_arrive_expect_tx(&ctrl->recv, (uint32_t)((ns - 1) * BM * (my_hi - my_lo) * 4));
                for (int t = 0; t < ns; ++t)
                    if (t != split) remote_arrive_sk(&ctrl->ready, t);
            }
            ok = ok && wait_cluster_sk(&ctrl->ready, 0, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                for (int t = 0; t < ns; ++t) {
                    if (t == split) continue;
                    const int lo = col_lo(t), hi = col_lo(t + 1);
                    if (lo >= hi) continue;
                    const uint32_t rbar = mapa_sk(&ctrl->recv, t);
                    const uint32_t rdst = mapa_sk(recvbuf + ((long long)split * BM + lrow) * pitch, t);
                    for (int c0 = lo & ~31; c0 < hi; c0 += 32) {
                        float f[32];
                        __syncwarp();
                        tmem_ld32(tmem + (uint32_t)c0 + ((uint32_t)(sub * 32) << 16), f);
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            if (c0 + e >= lo && c0 + e < hi)
                                st_async16_sk(rdst + (c0 + e - lo) * 4, rbar, f[e], f[e + 1], f[e + 2], f[e + 3]);
                    }
                }
                ok = wait_cluster_sk(&ctrl->recv, 0, abort);
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) flag(p.status, LORA_DEV_WAIT_TIMEOUT);
        }
        if (ok && my_lo < my_hi) {
            const int row = row0 + lrow;
            float *out = p.v + (long long)row * p.ld_v;
            const bool vec = (p.ld_v & 3) == 0;
            for (int c0 = my_lo & ~31; c0 < my_hi; c0 += 32) {
                float own[32];
                __syncwarp();
                tmem_ld32(tmem + (uint32_t)c0 + ((uint32_t)(sub * 32) << 16), own);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int col = c0 + e;
                    if (col < my_lo || col >= my_hi) continue;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int t = 0; t < ns; ++t) {                 // split order: deterministic
                        float4 f4;
                        if (t == split) {
                            f4 = make_float4(own[e], own[e + 1], own[e + 2], own[e + 3]);
                        } else {
                            f4 = *reinterpret_cast<const float4 *>(recvbuf + ((long long)t * BM + lrow) * pitch +
                                                                   (col - my_lo));
                        }
                        acc.x += f4.x;
                        acc.y += f4.y;
                        acc.z += f4.z;
                        acc.w += f4.w;
                    }
                    if (lrow < rows) {
                        if (vec) {
                            if (col < r)   // r <= ld_v and ld_v % 4 == 0: the float4 stays in the row
                                *reinterpret_cast<float4 *>(out + col) = acc;
                        } else {
                            const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
                            for (int u = 0; u < 4; ++u)
                                if (col + u < r) out[col + u] = a4[u];
                        }
                    }
                }
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, SK_TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    }
    return fn;
}

// 2-D bf16 tensor [outer x inner] (inner contiguous), box [box_outer x 64], 128-byte swizzle.
bool make_tmap(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [outer x inner] (e4m3 codes), box [box_outer x 128], 128-byte swizzle:
// the same 128-byte rows as the bf16 maps.
bool make_tmap_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {(cuuint32_t)(2 * BK), box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int ST, bool FUSE, bool FP8>
int launch_gemm_variant(const CUtensorMap &tmx, const CUtensorMap &tmw, const LayerTcParams &p, cudaStream_t st) {
    const size_t smem = (size_t)ST * STAGE_BYTES + (FUSE ? 2 * A2_BYTES + B2_BYTES : 0) + sizeof(Ctrl<ST>) + 1024;
    if (smem_optin(reinterpret_cast<const void *>(layer_gemm_tc_kernel<ST, FUSE, FP8>), smem)) return LORA_ERR_CUDA;
    const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
    layer_gemm_tc_kernel<ST, FUSE, FP8><<<grid, kThreadsTC, smem, st>>>(tmx, tmw, p);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace

bool gemm_tc_ok(const lora_pool *pool, int h_in, int h_out, int T, bool fp8) {
    return pool->dtype == LORA_BF16 && h_in % (fp8 ? 2 * BK : BK) == 0 && h_out % 32 == 0 && T > 0 &&
           encode_fn() != nullptr && num_sms() > 0;
}

int launch_gemm_tc(const lora_pool *pool, int h_in, int h_out, const void *x, const void *W, void *y, int T,
                   cudaStream_t st, int matrix, const int *tile_ad, const float *v, int ld_v, const Fp8Base *f8) {
    CUtensorMap tmx, tmw;
    if (f8) {
        if (!make_tmap_u8(&tmx, f8->xq, (uint64_t)h_in, (uint64_t)T, BM) ||
            !make_tmap_u8(&tmw, W, (uint64_t)h_in, (uint64_t)h_out, BN))
            return LORA_ERR_CUDA;
    } else if (!make_tmap(&tmx, x, (uint64_t)h_in, (uint64_t)T, BM) ||
               !make_tmap(&tmw, W, (uint64_t)h_in, (uint64_t)h_out, BN)) {
        return LORA_ERR_CUDA;
    }
    LayerTcParams p;
    p.T = T;
    p.N = h_out;
    p.K = h_in;
    p.num_m = (T + BM - 1) / BM;
    p.num_n = (h_out + BN - 1) / BN;
    p.num_k = h_in / (f8 ? 2 * BK : BK);
    p.num_tiles = p.num_m * p.num_n;
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.status = pool->d_status;
    p.tile_ad = tile_ad;
    p.pv = pool->view();
    p.m = matrix;
    p.v = v;
    p.ld_v = ld_v;
    p.sx = f8 ? f8->sx : nullptr;
    p.w_scale = f8 ? f8->w_scale : 1.f;
    if (f8) {
        if (tile_ad) return launch_gemm_variant<4, true, true>(tmx, tmw, p, st);
        return launch_gemm_variant<4, false, true>(tmx, tmw, p, st);
    }
    if (tile_ad) return launch_gemm_variant<4, true, false>(tmx, tmw, p, st);
    return launch_gemm_variant<4, false, false>(tmx, tmw, p, st);
}

bool shrink_tc_ok(const lora_pool *pool, int h_in, int S) {
    return pool->dtype == LORA_BF16 && h_in % BK == 0 && S <= kShrinkTcMaxS && encode_fn() != nullptr &&
           num_sms() > 0;
}

int launch_shrink_tc(const lora_pool *pool, int matrix, int h_in, const void *x, int T, int *tile_ad,
                     const int *seg_starts, const int *seg_adapter, int S, float *v, int ld_v, cudaStream_t st) {
    CUtensorMap tmx;
    if (!make_tmap(&tmx, x, (uint64_t)h_in, (uint64_t)T, BM)) return LORA_ERR_CUDA;
    ShrinkTcParams p;
    p.T = T;
    p.num_k = h_in / BK;
    // K splits: enough CTAs for two per SM over the expected tiles, at least 4
    // k-blocks per split
    const int est_tiles = std::max(1, tile_ad ? (T + BM - 1) / BM : T / BM);
    p.nsplit = std::max(1, std::min({kShrinkTcSplits, p.num_k / 4, 2 * num_sms() / est_tiles}));
    p.tile_ad = tile_ad;
    p.seg_starts = seg_starts;
    p.seg_adapter = seg_adapter;
    p.S = S;
    p.min_rows = kShrinkTcMinRows;
    p.n_ids = pool->mat_n_ids[matrix];
    p.pv = pool->view();
    p.m = matrix;
    p.v = v;
    p.ld_v = ld_v;
    p.status = pool->d_status;
    // ring: stages of an x tile plus the pool's widest A chunk; two CTAs per SM
    // when the stages and the partials the first CTA of a cluster receives fit
    // in half the shared memory
    const int npad_max = std::min(kFuseMaxRank, (pool->max_rank + 15) / 16 * 16);
    p.stage_bytes = SK_X_BYTES + npad_max * BK * 2;
    const size_t fixed = sizeof(SkCtrl) + 1024;
    const size_t need_recv = (size_t)p.nsplit * BM * ((((npad_max + p.nsplit - 1) / p.nsplit + 3) & ~3) + 4) * 4;
    const size_t need_scan = (size_t)(tile_ad ? 2 * S + 1 : S + 1) * 4;
    p.stages = 0;
    for (size_t budget : {(size_t)113 * 1024, (size_t)227 * 1024}) {
        const int st_n = (int)std::min<size_t>(SK_MAX_STAGES, (budget - fixed) / p.stage_bytes);
        if (st_n >= 4 && (size_t)st_n * p.stage_bytes >= std::max(need_recv, need_scan)) {
            p.stages = st_n;
            break;
        }
    }
    if (p.stages == 0) return LORA_ERR_ARG;       // not reached for ranks <= kFuseMaxRank
    const size_t smem = (size_t)p.stages * p.stage_bytes + fixed;
    if (smem_optin(reinterpret_cast<const void *>(shrink_tc_kernel), smem)) return LORA_ERR_CUDA;
    const int tiles = tile_ad ? (T + BM - 1) / BM : T / kShrinkTcMinRows;
    if (tiles == 0) return LORA_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, p.nsplit);
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = p.nsplit;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, shrink_tc_kernel, tmx, p);
    count_launch();
    return cuda_status(e);
}

}  // namespace lora
