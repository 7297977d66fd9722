// Shared base product of the adapted layer on the 5th-generation tensor cores:
//
//   y[t][n] = sum_k x[t][k] W[n][k]
//
// "The base part is one big shared matmul for the whole batch"
// ("Multi-LoRA Serving", section "The kernel trick: gather, do not merge");
// the per-row low-rank term is added after it by the SGMV expand.
//
// Structure: a persistent kernel, one CTA per SM, 128 x 256 output tiles,
// K in steps of 64.  Warp 0 (one lane) streams x and W tiles into a 4-stage
// shared-memory ring with TMA (128-byte swizzle); warp 1 (one lane) issues
// tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) into one of two TMEM
// accumulators (2 x 256 columns) and commits each ring slot back to the
// producer and each finished accumulator to the epilogue; warps 2-5 read the
// accumulator with tcgen05.ld (each warp its 32-lane TMEM sub-partition, one
// row per thread), round to bf16 and store.  The two accumulators let the epilogue of one tile overlap the
// main loop of the next.
//
// Every mbarrier wait is bounded (by the global timer); a wait that gives up
// sets LORA_DEV_WAIT_TIMEOUT, makes the other roles stop, waits (bounded)
// for its own copies and MMAs in flight, and the CTA frees its TMEM.
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "tc_common.cuh"

namespace lora {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreadsTC = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr unsigned long long kTimeoutNs = 2000000000ull;   // 2 s per wait

struct LayerTcParams {
    int T, N, K;
    int num_m, num_n, num_k, num_tiles;
    __nv_bfloat16 *y;
    int *status;
};

struct Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Bounded wait on one phase; gives up after kTimeoutNs or when *abort is set.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const unsigned long long t0 = now_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u) {
            if (abort && *abort) return false;
            if (now_ns() - t0 > kTimeoutNs) return false;
        }
    }
}

__device__ __forceinline__ void give_up(Ctrl *c, int *status) {
    c->abort = 1;
    __threadfence_block();
    flag(status, LORA_DEV_WAIT_TIMEOUT);
}

__global__ void __launch_bounds__(kThreadsTC, 1)
    layer_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                         LayerTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + STAGES * STAGE_BYTES);
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
        ctrl->abort = 0;
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
                    tma_load_2d(sa, &tmx, kb * BK, mb * BM, &ctrl->full[stage]);
                    tma_load_2d(sa + A_BYTES, &tmw, kb * BK, nb * BN, &ctrl->full[stage]);
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
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16(d, desc_kmajor_sw128(a0 + k * 32), desc_kmajor_sw128(b0 + k * 32), IDESC,
                                 (kb | k) != 0);
                    mma_commit(&ctrl->empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
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

            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = nb * BN + c * 32;
                float f[32];
                __syncwarp();
                tmem_ld32(tmem + (uint32_t)(b * BN + c * 32) + ((uint32_t)(sub * 32) << 16), f);
                if (col0 >= p.N || row >= p.T) continue;
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
        }
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
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

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
    }
    return n;
}

}  // namespace

bool gemm_tc_ok(const lora_pool *pool, int h_in, int h_out, int T) {
    return pool->dtype == LORA_BF16 && h_in % BK == 0 && h_out % 32 == 0 && T > 0 && encode_fn() != nullptr &&
           num_sms() > 0;
}

int launch_gemm_tc(const lora_pool *pool, int h_in, int h_out, const void *x, const void *W, void *y, int T,
                   cudaStream_t st) {
    CUtensorMap tmx, tmw;
    if (!make_tmap(&tmx, x, (uint64_t)h_in, (uint64_t)T, BM) || !make_tmap(&tmw, W, (uint64_t)h_in, (uint64_t)h_out, BN))
        return LORA_ERR_CUDA;
    LayerTcParams p;
    p.T = T;
    p.N = h_out;
    p.K = h_in;
    p.num_m = (T + BM - 1) / BM;
    p.num_n = (h_out + BN - 1) / BN;
    p.num_k = h_in / BK;
    p.num_tiles = p.num_m * p.num_n;
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.status = pool->d_status;
    const size_t smem = (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl) + 1024;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(layer_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return LORA_ERR_CUDA;
        configured = true;
    }
    const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();
    layer_gemm_tc_kernel<<<grid, kThreadsTC, smem, st>>>(tmx, tmw, p);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace lora
