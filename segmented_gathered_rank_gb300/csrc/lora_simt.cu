// CUDA-core kernels for the gathered low-rank update: one thread block per
// token.  BGMV (each decode token gathers its own adapter) fuses shrink and
// expand; SGMV (runs of consecutive tokens share an adapter) runs them as two
// launches with v in between ("Multi-LoRA Serving", section "The kernel trick:
// gather, do not merge").  Ranks are per adapter (S-LoRA slide 10, MBGMM/MBGMV): the
// loops over j run to the adapter's own rank.
#include "internal.cuh"

namespace lora {
namespace {

constexpr int kThreads = 256;

// v[j] = x_t . A_T_a[j] for j < r, one warp per row of A_T, into smem.
template <typename E>
__device__ __forceinline__ void shrink_row(const PoolView &pv, const int *rec, int r, const E *__restrict__ xr,
                                           int h_in, float *vs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int j = warp; j < r; j += nw) {
        const E *ar = page_row<E>(pv, rec[kRecHeader + j]);
        float acc = 0.f;
        for (int k = lane * 8; k < h_in; k += 32 * 8) {
            float xa[8], aa[8];
            load8(xr + k, xa);
            load8(ar + k, aa);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(xa[i], aa[i], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) vs[j] = acc;
    }
}

// y_t[n] += s * sum_j v[j] * B_a[j][n]; 8 consecutive n per thread.
template <typename E>
__device__ __forceinline__ void expand_row(const PoolView &pv, const int *rec, int r, float s, const float *vs,
                                           E *__restrict__ yr, int h_out) {
    for (int n = threadIdx.x * 8; n < h_out; n += blockDim.x * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < r; ++j) {
            float bb[8];
            load8(page_row<E>(pv, rec[kRecHeader + r + j]) + n, bb);
            const float vj = vs[j];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(vj, bb[i], acc[i]);
        }
        float yy[8];
        load8(yr + n, yy);
#pragma unroll
        for (int i = 0; i < 8; ++i) yy[i] = fmaf(s, acc[i], yy[i]);
        store8(yr + n, yy);
    }
}

template <typename E>
__global__ void __launch_bounds__(kThreads) bgmv_token_kernel(PoolView pv, int m, int h_in, int h_out,
                                                              const E *__restrict__ x, E *__restrict__ y,
                                                              const int *__restrict__ token_adapter) {
    extern __shared__ float vs[];
    const int t = blockIdx.x;
    const int a = token_adapter[t];
    if (a < 0) return;
    const int *rec = lookup(pv, a, m);
    if (!rec) return;
    const int r = rec[0];
    const float s = __int_as_float(rec[1]);
    shrink_row<E>(pv, rec, r, x + (long long)t * h_in, h_in, vs);
    __syncthreads();
    expand_row<E>(pv, rec, r, s, vs, y + (long long)t * h_out, h_out);
}

template <typename E>
__global__ void __launch_bounds__(kThreads) shrink_token_kernel(PoolView pv, int m, int h_in,
                                                                const E *__restrict__ x, float *__restrict__ v,
                                                                int ld_v, const int *__restrict__ seg_starts,
                                                                const int *__restrict__ seg_adapter, int S, int T) {
    extern __shared__ float vs[];
    const int t = blockIdx.x;
    if (t == 0) check_segments(seg_starts, S, T, pv.status);
    const int a = seg_adapter[segment_of(seg_starts, S, t)];
    if (a < 0) return;
    const int *rec = lookup(pv, a, m);
    if (!rec) return;
    const int r = rec[0];
    shrink_row<E>(pv, rec, r, x + (long long)t * h_in, h_in, vs);
    __syncthreads();
    for (int j = threadIdx.x; j < r; j += blockDim.x) v[(long long)t * ld_v + j] = vs[j];
}

template <typename E>
__global__ void __launch_bounds__(kThreads) expand_token_kernel(PoolView pv, int m, int h_out,
                                                                const float *__restrict__ v, int ld_v,
                                                                E *__restrict__ y, const int *__restrict__ seg_starts,
                                                                const int *__restrict__ seg_adapter, int S, int T) {
    extern __shared__ float vs[];
    const int t = blockIdx.x;
    if (t == 0) check_segments(seg_starts, S, T, pv.status);
    const int a = seg_adapter[segment_of(seg_starts, S, t)];
    if (a < 0) return;
    const int *rec = lookup(pv, a, m);
    if (!rec) return;
    const int r = rec[0];
    for (int j = threadIdx.x; j < r; j += blockDim.x) vs[j] = v[(long long)t * ld_v + j];
    __syncthreads();
    expand_row<E>(pv, rec, r, __int_as_float(rec[1]), vs, y + (long long)t * h_out, h_out);
}

// Plain tiled base product y = x . W^T on CUDA cores (64 x 64 tile, 4 x 4
// per thread).  Used for fp32 pools and shapes the tensor-core path does
// not take.
template <typename E>
__global__ void __launch_bounds__(256) base_gemm_simt_kernel(const E *__restrict__ x, const E *__restrict__ W,
                                                             E *__restrict__ y, int T, int h_in, int h_out) {
    __shared__ float xs[32][64 + 4];
    __shared__ float ws[32][64 + 4];
    const int tm = blockIdx.y * 64, tn = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < h_in; k0 += 32) {
        // 64 rows x 32 k of x and of W: 2048 elements each, 8 per thread.
        for (int i = threadIdx.x; i < 64 * 4; i += 256) {
            const int row = i >> 2, kk = (i & 3) * 8;
            float tmp[8];
            if (tm + row < T && k0 + kk < h_in) load8(x + (long long)(tm + row) * h_in + k0 + kk, tmp);
            else for (int q = 0; q < 8; ++q) tmp[q] = 0.f;
            for (int q = 0; q < 8; ++q) xs[kk + q][row] = tmp[q];
            if (tn + row < h_out && k0 + kk < h_in) load8(W + (long long)(tn + row) * h_in + k0 + kk, tmp);
            else for (int q = 0; q < 8; ++q) tmp[q] = 0.f;
            for (int q = 0; q < 8; ++q) ws[kk + q][row] = tmp[q];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            float a[4], b[4];
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
            for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
            for (int i = 0; i < 4; ++i)
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    for (int i = 0; i < 4; ++i) {
        const int row = tm + ty * 4 + i;
        if (row >= T) continue;
        for (int j = 0; j < 4; ++j) {
            const int col = tn + tx * 4 + j;
            if (col < h_out) {
                if constexpr (sizeof(E) == 2) y[(long long)row * h_out + col] = __float2bfloat16_rn(acc[i][j]);
                else y[(long long)row * h_out + col] = acc[i][j];
            }
        }
    }
}

}  // namespace

int launch_bgmv(const lora_pool *p, int matrix, int h_in, int h_out, const void *x, void *y,
                const int *token_adapter, int T, cudaStream_t st) {
    const int n_ids = p->mat_n_ids[matrix];
    if (bgmv_cluster_ok(p, h_in, h_out, T, n_ids))
        return launch_bgmv_cluster(p, matrix, h_in, h_out, x, y, token_adapter, T, n_ids, st);
    const size_t smem = (size_t)p->max_rank * sizeof(float);
    if (p->dtype == LORA_BF16)
        bgmv_token_kernel<__nv_bfloat16><<<T, kThreads, smem, st>>>(
            p->view(), matrix, h_in, h_out, (const __nv_bfloat16 *)x, (__nv_bfloat16 *)y, token_adapter);
    else
        bgmv_token_kernel<float><<<T, kThreads, smem, st>>>(p->view(), matrix, h_in, h_out, (const float *)x,
                                                           (float *)y, token_adapter);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int launch_shrink(const lora_pool *p, int matrix, int h_in, const void *x, float *v, int ld_v,
                  const int *seg_starts, const int *seg_adapter, int S, int T, cudaStream_t st) {
    if (sgmv_shrink_ok(p, h_in, S)) {
        // long segments on the tensor cores, the rest with warp MMAs
        int min_rows = 0;
        if (shrink_tc_ok(p, h_in, S) && p->mat_max_rank[matrix] >= kShrinkTcSegMinRank) {
            const int rc = launch_shrink_tc(p, matrix, h_in, x, T, nullptr, seg_starts, seg_adapter, S, v, ld_v, st);
            if (rc) return rc;
            min_rows = kShrinkTcMinRows;
        }
        return launch_sgmv_shrink(p, matrix, h_in, x, v, ld_v, seg_starts, seg_adapter, S, T, nullptr, st, false,
                                  min_rows);
    }
    const size_t smem = (size_t)p->max_rank * sizeof(float);
    if (p->dtype == LORA_BF16)
        shrink_token_kernel<__nv_bfloat16><<<T, kThreads, smem, st>>>(
            p->view(), matrix, h_in, (const __nv_bfloat16 *)x, v, ld_v, seg_starts, seg_adapter, S, T);
    else
        shrink_token_kernel<float><<<T, kThreads, smem, st>>>(p->view(), matrix, h_in, (const float *)x, v, ld_v,
                                                             seg_starts, seg_adapter, S, T);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int launch_expand(const lora_pool *p, int matrix, int h_out, const float *v, int ld_v, void *y,
                  const int *seg_starts, const int *seg_adapter, int S, int T, cudaStream_t st) {
    if (sgmv_expand_ok(p, h_out, S))
        return launch_sgmv_expand(p, matrix, h_out, v, ld_v, y, seg_starts, seg_adapter, S, T, nullptr, st);
    const size_t smem = (size_t)p->max_rank * sizeof(float);
    if (p->dtype == LORA_BF16)
        expand_token_kernel<__nv_bfloat16><<<T, kThreads, smem, st>>>(
            p->view(), matrix, h_out, v, ld_v, (__nv_bfloat16 *)y, seg_starts, seg_adapter, S, T);
    else
        expand_token_kernel<float><<<T, kThreads, smem, st>>>(p->view(), matrix, h_out, v, ld_v, (float *)y,
                                                             seg_starts, seg_adapter, S, T);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int launch_base_gemm(const lora_pool *p, int h_in, int h_out, const void *x, const void *W, void *y, int T,
                     cudaStream_t st) {
    dim3 grid((h_out + 63) / 64, (T + 63) / 64);
    if (p->dtype == LORA_BF16)
        base_gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)W, (__nv_bfloat16 *)y, T, h_in, h_out);
    else
        base_gemm_simt_kernel<float><<<grid, 256, 0, st>>>((const float *)x, (const float *)W, (float *)y, T,
                                                           h_in, h_out);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace lora
