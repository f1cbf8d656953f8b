// nvfp4_linear_noalloc: the NVFP4 linear layer for callers that cannot
// allocate device memory.
//
// nvfp4_linear needs scratch space (the quantized activation, its block
// scales and the activation's global scale) that its caller allocates and
// passes in. Some callers cannot do that: a plugin running inside a host
// application that owns the device memory pool and forbids allocations from
// outside it, a serving loop that reserves all of its memory at start-up so
// that no request can fail half-way on an allocation, or a C caller that has
// no device allocator to hand. This entry point takes the same inputs and
// output but keeps its scratch in a fixed-size array that lives in the
// library itself, so it calls no cudaMalloc, cudaFree or allocating library
// routine.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits. Host code
// only sees a host-side stand-in under the array's name, so the device
// address is looked up once per device with cudaGetSymbolAddress (on the
// first call made while that device is current) and then passed to the
// kernels as an ordinary pointer. The kept address belongs to the device's
// primary context: after a cudaDeviceReset it is stale, so the entry point
// is not to be called on that device again in the same process.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "nvfp4.h"

namespace nvfp4 {
namespace {

// 16 MiB: enough for the activation of an LLM prefill projection of
// 4096 tokens x 5120 features (about 11.8 MB of codes and scales).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on
// first use for that device).
cudaError_t scratch_on_current_device(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_linear_noalloc(const void *X, int64_t M, int64_t K, int64_t ldx,
                                  const uint8_t *Wq, const uint8_t *Ws, const float *g_w,
                                  int64_t N, void *Y, int64_t ldy, const float *g_x,
                                  void *stream) {
    if (M < 0 || N < 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
    const size_t need = nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED);
    if (K % 256 == 0 && need > nvfp4::kNoAllocScratchBytes)
        return NVFP4_ERR_WORKSPACE_TOO_SMALL;  // M x K beyond the fixed scratch
    unsigned char *scratch = nullptr;
    if (nvfp4::scratch_on_current_device(&scratch) != cudaSuccess) return NVFP4_ERR_CUDA;
    // Same launch sequence as nvfp4_linear, with the library's own scratch as
    // the workspace. The kernels clear what they accumulate into (the amax
    // cell, the padding rows of the scales) on every call, so the previous
    // call's contents do no harm.
    return nvfp4_linear(X, M, K, ldx, Wq, Ws, g_w, N, Y, ldy, g_x, NVFP4_LINEAR_UNFUSED,
                        scratch, nvfp4::kNoAllocScratchBytes, stream);
}

}  // extern "C"
