// lora_layer_forward_noalloc: the adapted layer for callers that cannot
// allocate device memory.
//
// lora_layer_forward needs T * max_rank fp32 of scratch for the low-rank
// activations v (shrink output, expand input) and asks the caller for it.
// Some callers cannot provide it: a C serving runtime that carved all device
// memory into a fixed arena at start-up and has no allocator left to call; a
// latency-critical decode loop that must not call cudaMalloc/cudaFree,
// because those synchronise the whole device and stall every stream; a
// plugin inside a host process whose own allocator is not reachable from C.
// This entry point takes the scratch from a fixed array compiled into the
// library instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds LORA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the variable's name as a device address (on the host
// it names a stand-in object), so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current and
// caches it; make that first call before capturing any stream.  All calls
// share the one array and it keeps the last call's contents: calls whose
// work overlaps on the GPU (two streams, two host threads) race on it and
// must be serialised by the caller.  Nothing in it needs to start at zero:
// the shrink writes every v entry the expand later reads.
#include <mutex>

#include "internal.cuh"

namespace lora {
namespace {

constexpr size_t kScratchFloats = LORA_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
int scratch_address(int device, void **out) {
    if (device < 0 || device >= kMaxDevices) return LORA_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return LORA_ERR_CUDA;
        }
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return LORA_OK;
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" int lora_layer_forward_noalloc(lora_pool *p, int matrix, const void *x, const void *W, void *y,
                                          const int *seg_starts, const int *seg_adapter, int S, int T,
                                          lora_stream stream) {
    if (!p || T < 0 || S < 0 || (S == 0 && T > 0)) return LORA_ERR_ARG;
    int h_in, h_out, rc;
    if ((rc = matrix_dims(p, matrix, &h_in, &h_out))) return rc;
    if (T == 0) return LORA_OK;
    if (!x || !W || !y || !seg_starts || !seg_adapter || !aligned16(x) || !aligned16(W) || !aligned16(y))
        return LORA_ERR_ARG;
    if (lora_layer_forward_workspace_size(p, matrix, S, T) > LORA_NOALLOC_SCRATCH_BYTES)
        return LORA_ERR_ARG;   // beyond the fixed scratch
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return LORA_ERR_CUDA;
    }
    if (device != p->device) return LORA_ERR_ARG;
    void *scratch = nullptr;
    if ((rc = scratch_address(device, &scratch))) return rc;
    return layer_forward_impl(p, matrix, h_in, h_out, x, W, y, seg_starts, seg_adapter, S, T,
                              static_cast<float *>(scratch), (cudaStream_t)stream);
}
