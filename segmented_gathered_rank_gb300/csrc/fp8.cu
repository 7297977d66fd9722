// FP8 base product of the adapted layer: the base weights in e4m3, the
// adapters in bf16 ("Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter
// Hot-Swap & Memory": the base may be served in FP8 while adapters trained
// on a bf16 base keep working).
//
//   lora_quantize_e4m3      x (bf16) -> per-row e4m3 codes and fp32 scales
//   lora_layer_forward_fp8  quantise x, then the layer of lora_layer_forward
//                           with the tensor-core GEMM in FP8 (kind::f8f6f4)
//
// Quantisation of row t, with a = max_k |x[t][k]| (448 is e4m3's largest
// finite value): s_x[t] = a / 448 and r = 448 / a (fp32 divisions, once per
// row), q[t][k] = e4m3(x[t][k] * r) with the product in fp32 and the
// conversion rounding to nearest even and saturating at +-448.  A row with
// a < 2^-120 (zeros included) takes s_x = 1 and all-zero codes.
#include "internal.cuh"

namespace lora {
namespace {

constexpr int kQThreads = 256;
constexpr float kTinyRow = 7.52316384526264e-37f;   // 2^-120

// e4m3 codes of two floats, rounded to nearest even and saturated at +-448
// (cvt.rn.satfinite.e4m3x2.f32: `upper` goes to bits 8-15, `lower` to bits 0-7).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float upper, float lower) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(d) : "f"(upper), "f"(lower));
    return d;
}

// One CTA per row: the row's largest magnitude, then its codes.  Rows of up
// to kQThreads * 8 * kQVec elements are read once, each thread keeping its
// elements in registers between the two steps; longer rows are read twice.
constexpr int kQVec = 4;

__global__ void __launch_bounds__(kQThreads) quantize_e4m3_kernel(const __nv_bfloat16 *__restrict__ x, int h,
                                                                   uint8_t *__restrict__ q, float *__restrict__ sx) {
    __shared__ float wmax[kQThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    const __nv_bfloat16 *xr = x + (long long)t * h;
    uint8_t *qr = q + (long long)t * h;
    const bool held = h <= kQThreads * 8 * kQVec;
    uint4 v[kQVec];
    float m = 0.f;
    if (held) {
#pragma unroll
        for (int u = 0; u < kQVec; ++u) {
            const int i = (tid + u * kQThreads) * 8;
            v[u] = i < h ? *reinterpret_cast<const uint4 *>(xr + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQVec; ++u) {
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    } else {
        for (int i = tid * 8; i < h; i += kQThreads * 8) {
            float f[8];
            load8(xr + i, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) wmax[tid >> 5] = m;
    __syncthreads();
    float amax = 0.f;
#pragma unroll
    for (int w = 0; w < kQThreads / 32; ++w) amax = fmaxf(amax, wmax[w]);
    const bool tiny = !(amax >= kTinyRow);
    const float s = tiny ? 1.f : __fdiv_rn(amax, 448.f);
    const float r = tiny ? 0.f : __fdiv_rn(448.f, amax);
    if (tid == 0) sx[t] = s;
    auto convert = [&](const float *f, int i) {
        uint32_t w[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            // two codes per conversion: the lower byte holds element 2e, the upper 2e + 1
            const uint32_t lo = cvt_e4m3x2(__fmul_rn(f[4 * h2 + 1], r), __fmul_rn(f[4 * h2], r));
            const uint32_t hi = cvt_e4m3x2(__fmul_rn(f[4 * h2 + 3], r), __fmul_rn(f[4 * h2 + 2], r));
            w[h2] = tiny ? 0u : (lo | (hi << 16));      // a negligible row: +0 codes
        }
        *reinterpret_cast<uint2 *>(qr + i) = make_uint2(w[0], w[1]);
    };
    if (held) {
#pragma unroll
        for (int u = 0; u < kQVec; ++u) {
            const int i = (tid + u * kQThreads) * 8;
            if (i >= h) break;
            float f[8];
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 ff = __bfloat1622float2(h2[e]);
                f[2 * e] = ff.x;
                f[2 * e + 1] = ff.y;
            }
            convert(f, i);
        }
    } else {
        for (int i = tid * 8; i < h; i += kQThreads * 8) {
            float f[8];
            load8(xr + i, f);
            convert(f, i);
        }
    }
}

// The FP8 call's extra scratch after the layer's own: codes [T x h_in], scales [T].
size_t q_offset(const lora_pool *p, int matrix, int S, int T) {
    return (lora_layer_forward_workspace_size(p, matrix, S, T) + 255) & ~(size_t)255;
}

}  // namespace

int launch_quantize(const void *x, int T, int h, void *q, float *sx, cudaStream_t st) {
    if (T == 0) return LORA_OK;
    quantize_e4m3_kernel<<<T, kQThreads, 0, st>>>(static_cast<const __nv_bfloat16 *>(x), h,
                                                  static_cast<uint8_t *>(q), sx);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace lora

using namespace lora;

extern "C" {

int lora_quantize_e4m3(const void *x, int T, int h, void *q, float *sx, lora_stream stream) {
    if (T < 0 || h <= 0 || h % 8) return LORA_ERR_ARG;
    if (T == 0) return LORA_OK;
    if (!x || !q || !sx || !aligned16(x) || ((uintptr_t)q & 7u) || ((uintptr_t)sx & 3u)) return LORA_ERR_ARG;
    return launch_quantize(x, T, h, q, sx, (cudaStream_t)stream);
}

size_t lora_layer_forward_fp8_workspace_size(const lora_pool *p, int matrix, int S, int T) {
    int h_in, h_out;
    if (!p || T < 0 || S < 0 || matrix_dims(p, matrix, &h_in, &h_out)) return 0;
    const size_t q_bytes = ((size_t)T * h_in + 255) & ~(size_t)255;
    return q_offset(p, matrix, S, T) + q_bytes + (size_t)T * sizeof(float) + 256;
}

int lora_layer_forward_fp8(lora_pool *p, int matrix, const void *x, const void *W8, float w_scale, void *y,
                           const int *seg_starts, const int *seg_adapter, int S, int T, void *workspace,
                           size_t ws_bytes, lora_stream stream) {
    if (!p || T < 0 || S < 0 || (S == 0 && T > 0)) return LORA_ERR_ARG;
    int h_in, h_out, rc;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (p->dtype != LORA_BF16) return LORA_ERR_ARG;
    if (h_in % 128 || h_out % 32) return LORA_ERR_SHAPE;
    if (!(w_scale > 0.f) || w_scale > 3.0e38f) return LORA_ERR_ARG;
    if (T == 0) return LORA_OK;
    if (!x || !W8 || !y || !seg_starts || !seg_adapter || !workspace || !aligned16(x) || !aligned16(W8) ||
        !aligned16(y) || !aligned16(workspace))
        return LORA_ERR_ARG;
    if (ws_bytes < lora_layer_forward_fp8_workspace_size(p, matrix, S, T)) return LORA_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *xq = ws + q_offset(p, matrix, S, T);
    float *sx = reinterpret_cast<float *>(xq + (((size_t)T * h_in + 255) & ~(size_t)255));
    const Fp8Base f8{xq, sx, w_scale, true};      // the layer call quantises x on a stream of its own
    return layer_forward_impl(p, matrix, h_in, h_out, x, W8, y, seg_starts, seg_adapter, S, T,
                              reinterpret_cast<float *>(ws), st, &f8);
}

}  // extern "C"
