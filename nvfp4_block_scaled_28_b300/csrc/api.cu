// C ABI of the NVFP4 library: argument checks, status codes, workspace
// carving and the launch sequences of each entry point (see include/nvfp4.h).
#include <cmath>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "internal.h"
#include "nvfp4.h"
#include "ptx.cuh"

namespace nvfp4 {

// Device-side error word: kernels OR kDevErrTimeout into it when a bounded
// wait runs out. Kernels receive its address as a parameter.
__device__ unsigned int g_device_error = 0;

int device_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kMaxDevices;
    return dev;
}

unsigned int *device_error_word() {
    static DeviceOnce once;
    static unsigned int *addr[kMaxDevices + 1] = {};
    const int dev = device_slot();
    if (dev == kMaxDevices) return nullptr;
    const cudaError_t e = once.run([](int slot) {
        void *p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_device_error);
        if (r == cudaSuccess) addr[slot] = static_cast<unsigned int *>(p);
        return r;
    });
    return e == cudaSuccess ? addr[dev] : nullptr;
}

const LaunchCfg &launch_cfg() {
    static DeviceOnce once;
    static LaunchCfg cfg[kMaxDevices + 1];
    const int dev = device_slot();
    (void)once.run([](int slot) {
        int sms = 0;
        if (slot < kMaxDevices &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, slot) == cudaSuccess &&
            sms > 0)
            cfg[slot].num_sms = sms;
        return cudaSuccess;
    });
    return cfg[dev];
}

DebugState &debug_state() {
    static DebugState s;
    return s;
}

namespace {

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline nvfp4_status from_cuda(cudaError_t e) {
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Limits of the 32-bit index arithmetic inside the kernels: the element,
// 16-element-block and 16-byte-vector indices of a tensor, plus the few
// grid strides a thread adds ahead of its bounds test, stay below 2^32 when
// a tensor has fewer than 2^28 blocks (2^32 elements, 8 GiB of bfloat16).
constexpr int64_t kMaxBlocks = int64_t(1) << 28;
constexpr int64_t kMaxDim = int64_t(1) << 30;
constexpr int64_t kMaxOutputs = int64_t(1) << 42;  // M x N of one GEMM

nvfp4_status check_bf16_matrix(const void *X, int64_t rows, int64_t cols, int64_t ld) {
    if (rows < 0 || cols < 0 || ld < cols) return NVFP4_ERR_INVALID_ARG;
    if (rows > kMaxDim || cols > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows > 0 && cols > 0 && X == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(X, 16) || (ld % 8) != 0) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

nvfp4_status check_quantize(const void *X, int64_t rows, int64_t cols, int64_t ldx,
                            const float *g, const uint8_t *q, const uint8_t *sf, int layout) {
    if (layout != NVFP4_SF_ROW_MAJOR && layout != NVFP4_SF_MMA_128x4) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s = check_bf16_matrix(X, rows, cols, ldx);
    if (s != NVFP4_OK) return s;
    if (cols % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (layout == NVFP4_SF_MMA_128x4 && cols % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows * (cols / 16) >= kMaxBlocks) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (g == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (rows > 0 && cols > 0 && (q == nullptr || sf == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(g, 4) || !aligned(q, 8)) return NVFP4_ERR_MISALIGNED;
    if (layout == NVFP4_SF_MMA_128x4 && !aligned(sf, 4)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

// Shapes, the weight-side operand and the output of a GEMM / linear call.
nvfp4_status check_gemm_b_and_y(const uint8_t *Bq, const uint8_t *Bs, const float *g_b, int64_t M,
                                int64_t N, int64_t K, const void *Y, int64_t ldy) {
    if (M < 0 || N < 0 || K <= 0 || ldy < N) return NVFP4_ERR_INVALID_ARG;
    if (K % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M * N >= kMaxOutputs) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // tile counts stay 32-bit
    if (M == 0 || N == 0) return NVFP4_OK;
    if (!Bq || !Bs || !g_b || !Y) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(Bq, 16) || !aligned(Bs, 16) || !aligned(g_b, 4) || !aligned(Y, 2))
        return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

nvfp4_status check_gemm(const uint8_t *Aq, const uint8_t *As, const float *g_a,
                        const uint8_t *Bq, const uint8_t *Bs, const float *g_b, int64_t M,
                        int64_t N, int64_t K, const void *Y, int64_t ldy) {
    nvfp4_status s = check_gemm_b_and_y(Bq, Bs, g_b, M, N, K, Y, ldy);
    if (s != NVFP4_OK || M == 0 || N == 0) return s;
    if (!Aq || !As || !g_a) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(Aq, 16) || !aligned(As, 16) || !aligned(g_a, 4)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char *nvfp4_status_string(int status) {
    switch (status) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_MISALIGNED: return "NVFP4_ERR_MISALIGNED";
        case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
        case NVFP4_ERR_WORKSPACE_TOO_SMALL: return "NVFP4_ERR_WORKSPACE_TOO_SMALL";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
        case NVFP4_ERR_BOUNDS: return "NVFP4_ERR_BOUNDS";
        default: return "NVFP4_ERR_UNKNOWN";
    }
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t K, int layout) {
    if (rows < 0 || K < 0) return 0;
    if (layout == NVFP4_SF_ROW_MAJOR) {
        if (K % 16) return 0;
        return static_cast<size_t>(rows) * static_cast<size_t>(K / 16);
    }
    if (layout == NVFP4_SF_MMA_128x4) {
        if (K % 64) return 0;
        return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>(K / 16);
    }
    return 0;
}

nvfp4_status nvfp4_global_scale(const void *X, int64_t rows, int64_t cols, int64_t ldx, float *g,
                                void *stream) {
    nvfp4_status s = check_bf16_matrix(X, rows, cols, ldx);
    if (s != NVFP4_OK) return s;
    if (g == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(g, 4)) return NVFP4_ERR_MISALIGNED;
    if (cols % 8 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows * cols >= kMaxBlocks * 16) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return from_cuda(launch_global_scale(static_cast<const uint16_t *>(X), rows, cols, ldx, g,
                                         static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize(const void *X, int64_t rows, int64_t cols, int64_t ldx, const float *g,
                            uint8_t *q, uint8_t *sf, int sf_layout, void *stream) {
    nvfp4_status s = check_quantize(X, rows, cols, ldx, g, q, sf, sf_layout);
    if (s != NVFP4_OK) return s;
    return from_cuda(launch_quantize(static_cast<const uint16_t *>(X), rows, cols, ldx, g, q, sf,
                                     sf_layout, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize_select(const void *X, int64_t rows, int64_t cols, int64_t ldx,
                                   const float *g, int rule, uint8_t *q, uint8_t *sf,
                                   int sf_layout, void *stream) {
    if (rule != NVFP4_SCALE_ABSMAX && rule != NVFP4_SCALE_FOUR_OVER_SIX && rule != NVFP4_SCALE_MSE)
        return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s = check_quantize(X, rows, cols, ldx, g, q, sf, sf_layout);
    if (s != NVFP4_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t *Xh = static_cast<const uint16_t *>(X);
    if (rule == NVFP4_SCALE_ABSMAX)
        return from_cuda(launch_quantize(Xh, rows, cols, ldx, g, q, sf, sf_layout, st));
    return from_cuda(launch_quantize_select(Xh, rows, cols, ldx, g, rule, q, sf, sf_layout, st));
}

nvfp4_status nvfp4_quantize_weight(const void *W, int64_t N, int64_t K, int64_t ldw, uint8_t *Wq,
                                   uint8_t *Ws, float *g_w, int sf_layout, void *stream) {
    nvfp4_status s = check_quantize(W, N, K, ldw, g_w, Wq, Ws, sf_layout);
    if (s != NVFP4_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_global_scale(static_cast<const uint16_t *>(W), N, K, ldw, g_w, st);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    return from_cuda(
        launch_quantize(static_cast<const uint16_t *>(W), N, K, ldw, g_w, Wq, Ws, sf_layout, st));
}

nvfp4_status nvfp4_sf_to_mma_layout(const uint8_t *sf_row_major, int64_t rows, int64_t K,
                                    uint8_t *sf_mma, void *stream) {
    if (rows < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows > kMaxDim || (rows + 127) / 128 * 128 * (K / 64) >= kMaxBlocks)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0 || K == 0) return NVFP4_OK;
    if (!sf_row_major || !sf_mma) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(sf_row_major, 4) || !aligned(sf_mma, 4)) return NVFP4_ERR_MISALIGNED;
    return from_cuda(
        launch_sf_to_mma(sf_row_major, rows, K, sf_mma, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

nvfp4_status nvfp4_gemm(const uint8_t *Aq, const uint8_t *As, const float *g_a, const uint8_t *Bq,
                        const uint8_t *Bs, const float *g_b, int64_t M, int64_t N, int64_t K,
                        void *Y, int64_t ldy, void *workspace, size_t workspace_bytes,
                        void *stream) {
    nvfp4_status s = check_gemm(Aq, As, g_a, Bq, Bs, g_b, M, N, K, Y, ldy);
    if (s != NVFP4_OK) return s;
    if (workspace_bytes < nvfp4_gemm_workspace_bytes(M, N, K))
        return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    (void)workspace;
    if (M == 0 || N == 0) return NVFP4_OK;
    if (M <= kSkinnyMaxM) {
        // few activation rows: weights as the 128-row MMA operand
        SkinnyArgs sa{Bq, Bs, g_b, Aq, As, nullptr, 0, g_a, M, N, K,
                      static_cast<uint16_t *>(Y), ldy, 0};
        return from_cuda(launch_gemm_skinny(sa, static_cast<cudaStream_t>(stream)));
    }
    GemmArgs a{Aq, As, g_a, Bq, Bs, g_b, M, N, K, static_cast<uint16_t *>(Y), ldy};
    return from_cuda(launch_gemm_plain(a, static_cast<cudaStream_t>(stream)));
}

// nvfp4_linear workspace: [g_x, barrier counter | amax partials] header,
// X codes, X scales.
constexpr size_t kLinearHeader = 256 + sizeof(uint32_t) * kMaxAmaxPartials;
static_assert(kLinearHeader == 8448, "offset of X's codes documented in nvfp4.h");

}  // extern "C"

namespace {

// The activation quantization step of the linear layers: X -> codes and
// tile-layout scales in the workspace. With *g_x == nullptr one launch also
// computes g_x into the workspace header (a small X: every CTA reduces the
// amax itself; else amax partials, a grid barrier, quantization) and *g_x is
// pointed at it; the GEMM that follows runs as its programmatic dependent.
cudaError_t quantize_activation(const uint16_t *Xh, int64_t M, int64_t K, int64_t ldx,
                                const float **g_x, uint8_t *ws, cudaStream_t st) {
    float *gx_slot = reinterpret_cast<float *>(ws);
    uint32_t *partials = reinterpret_cast<uint32_t *>(ws + 256);
    uint8_t *xq = ws + kLinearHeader;
    uint8_t *xs = xq + round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    if (*g_x != nullptr) return launch_quantize(Xh, M, K, ldx, *g_x, xq, xs, NVFP4_SF_MMA_128x4, st);
    unsigned int *counter = reinterpret_cast<unsigned int *>(ws + 64);
    *g_x = gx_slot;
    if (M * K <= kQuantizeSmallElems) return launch_quantize_small(Xh, M, K, ldx, gx_slot, xq, xs, st);
    if (M * K <= kQuantizeClusterElems) {
        const cudaError_t e = launch_quantize_cluster(Xh, M, K, ldx, gx_slot, xq, xs, st);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch_quantize_fused(Xh, M, K, ldx, partials, counter, gx_slot, xq, xs, st);
}

}  // namespace

extern "C" {

size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode) {
    if (M < 0 || N < 0 || K < 0 || K % 256 != 0) return 0;
    (void)mode;
    size_t bytes = kLinearHeader;  // g_x and the amax partials
    bytes += round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    bytes += round_up(nvfp4_sf_bytes(M, K, NVFP4_SF_MMA_128x4), 256);
    bytes += nvfp4_gemm_workspace_bytes(M, N, K);
    return bytes;
}

}  // extern "C"

namespace {

// nvfp4_linear and nvfp4_linear_grouped: `wg` describes the weight groups
// (count 0: one group, g_w one float).
nvfp4_status linear_impl(const void *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq,
                         const uint8_t *Ws, const float *g_w, int64_t N, void *Y, int64_t ldy,
                         const float *g_x, int mode, void *workspace, size_t workspace_bytes,
                         void *stream, const WeightGroups &wg) {
    if (mode != NVFP4_LINEAR_UNFUSED && mode != NVFP4_LINEAR_FUSED) return NVFP4_ERR_INVALID_ARG;
    nvfp4_status s = check_bf16_matrix(X, M, K, ldx);
    if (s != NVFP4_OK) return s;
    s = check_gemm_b_and_y(Wq, Ws, g_w, M, N, K, Y, ldy);
    if (s != NVFP4_OK) return s;
    if (M == 0 || N == 0) return NVFP4_OK;
    // per-group scales live in the CTA-pair kernel's extended epilogue
    if (wg.count > 1 && M > kSkinnyMaxM && gemm_kernel_choice() == kGemmSingle)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (g_x != nullptr && !aligned(g_x, 4)) return NVFP4_ERR_MISALIGNED;
    const size_t need = nvfp4_linear_workspace_bytes(M, N, K, mode);
    if (workspace_bytes < need) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;
    if (M * (K / 16) >= kMaxBlocks) return NVFP4_ERR_UNSUPPORTED_SHAPE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *xq = ws + kLinearHeader;
    uint8_t *xs = xq + round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    const uint16_t *Xh = static_cast<const uint16_t *>(X);
    if (mode == NVFP4_LINEAR_FUSED && M <= kSkinnyFusedMaxM && K <= kSkinnyFusedMaxK) {
        // one launch: the GEMM computes g_x (when not given) and quantizes X
        // tiles in shared memory; no codes in HBM
        SkinnyArgs sa{Wq, Ws, g_w, nullptr, nullptr, Xh, ldx, g_x, M, N, K,
                      static_cast<uint16_t *>(Y), ldy, 1, wg};
        if (debug_state().capture_fused_operand) {
            // testing hook: the operand the kernel quantized in shared
            // memory goes where the unfused path leaves it
            sa.dbg_xq = xq;
            sa.dbg_xs = xs;
        }
        return from_cuda(launch_gemm_skinny(sa, st));
    }
    // unfused (and fused beyond 8 rows or K = 6144: the resident operand
    // holds 8 rows of up to 6144 K)
    if (quantize_activation(Xh, M, K, ldx, &g_x, ws, st) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (M <= kSkinnyMaxM) {
        SkinnyArgs sa{Wq, Ws, g_w, xq, xs, nullptr, 0, g_x, M, N, K,
                      static_cast<uint16_t *>(Y), ldy, 0, wg};
        return from_cuda(launch_gemm_skinny(sa, st));
    }
    GemmArgs a{xq, xs, g_x, Wq, Ws, g_w, M, N, K, static_cast<uint16_t *>(Y), ldy};
    a.groups = wg;
    return from_cuda(launch_gemm_plain(a, st));
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_linear(const void *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq,
                          const uint8_t *Ws, const float *g_w, int64_t N, void *Y, int64_t ldy,
                          const float *g_x, int mode, void *workspace, size_t workspace_bytes,
                          void *stream) {
    return linear_impl(X, M, K, ldx, Wq, Ws, g_w, N, Y, ldy, g_x, mode, workspace,
                       workspace_bytes, stream, WeightGroups{});
}

nvfp4_status nvfp4_linear_grouped(const void *X, int64_t M, int64_t K, int64_t ldx,
                                  const uint8_t *Wq, const uint8_t *Ws, const float *g_w,
                                  const int64_t *group_n, int groups, void *Y, int64_t ldy,
                                  const float *g_x, int mode, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    if (group_n == nullptr || groups < 1 || groups > kMaxGroups) return NVFP4_ERR_INVALID_ARG;
    WeightGroups wg;
    wg.count = groups;
    int64_t N = 0;
    for (int g = 0; g < groups; ++g) {
        if (group_n[g] <= 0) return NVFP4_ERR_INVALID_ARG;
        if (group_n[g] % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        N += group_n[g];
        if (N > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        wg.end[g] = static_cast<int>(N);
    }
    return linear_impl(X, M, K, ldx, Wq, Ws, g_w, N, Y, ldy, g_x, mode, workspace,
                       workspace_bytes, stream, wg);
}

size_t nvfp4_linear_lora_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r) {
    if (M < 0 || N < 0 || K < 0 || r < 0 || K % 256 != 0) return 0;
    return nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED) +
           round_up(static_cast<size_t>(M) * static_cast<size_t>(r) * 2, 256) +
           round_up(lora_partial_bytes(M, r), 256);
}

nvfp4_status nvfp4_linear_lora(const void *X, int64_t M, int64_t K, int64_t ldx,
                               const uint8_t *Wq, const uint8_t *Ws, const float *g_w, int64_t N,
                               const void *lora_A, const void *lora_B, int64_t r,
                               float lora_scale, void *Y, int64_t ldy, const float *g_x,
                               void *workspace, size_t workspace_bytes, void *stream) {
    nvfp4_status s = check_bf16_matrix(X, M, K, ldx);
    if (s != NVFP4_OK) return s;
    s = check_gemm_b_and_y(Wq, Ws, g_w, M, N, K, Y, ldy);
    if (s != NVFP4_OK) return s;
    if (r != 16 && r != 32 && r != 48 && r != 64) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!std::isfinite(lora_scale)) return NVFP4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return NVFP4_OK;
    // the up projection rides in the CTA-pair kernel, the one used above 128 rows
    if (M <= kSkinnyMaxM || gemm_kernel_choice() == kGemmSingle)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M * (K / 16) >= kMaxBlocks) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (lora_A == nullptr || lora_B == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(lora_A, 16) || !aligned(lora_B, 16)) return NVFP4_ERR_MISALIGNED;
    if (g_x != nullptr && !aligned(g_x, 4)) return NVFP4_ERR_MISALIGNED;
    const size_t need = nvfp4_linear_lora_workspace_bytes(M, N, K, r);
    if (workspace_bytes < need) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *gx_slot = reinterpret_cast<float *>(ws);
    uint8_t *xq = ws + kLinearHeader;
    uint8_t *xs = xq + round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    uint8_t *lora_ws = ws + nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED);
    uint16_t *Lp = reinterpret_cast<uint16_t *>(lora_ws);
    float *part = reinterpret_cast<float *>(
        lora_ws + round_up(static_cast<size_t>(M) * static_cast<size_t>(r) * 2, 256));
    const uint16_t *Xh = static_cast<const uint16_t *>(X);
    if (g_x == nullptr) {
        if (launch_global_scale(Xh, M, K, ldx, gx_slot, st) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        g_x = gx_slot;
    }
    // one pass over X: codes, scales and the pre-scaled down projection
    if (launch_quantize_lora(Xh, M, K, ldx, g_x, g_w, lora_scale,
                             static_cast<const uint16_t *>(lora_A), r, xq, xs, part, Lp,
                             st) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    GemmArgs a{xq, xs, g_x, Wq, Ws, g_w, M, N, K, static_cast<uint16_t *>(Y), ldy};
    a.lora_Lp = Lp;
    a.lora_B = static_cast<const uint16_t *>(lora_B);
    a.lora_r = r;
    return from_cuda(launch_gemm_pair(a, st));
}

nvfp4_status nvfp4_linear_bias_requant(const void *X, int64_t M, int64_t K, int64_t ldx,
                                       const uint8_t *Wq, const uint8_t *Ws, const float *g_w,
                                       int64_t N, const void *bias, void *Y, int64_t ldy,
                                       const float *g_y, uint8_t *Yq, uint8_t *Ys,
                                       const float *g_x, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    nvfp4_status s = check_bf16_matrix(X, M, K, ldx);
    if (s != NVFP4_OK) return s;
    if (M < 0 || N < 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
    const bool requant = Yq != nullptr || Ys != nullptr || g_y != nullptr;
    if (requant && (Yq == nullptr || Ys == nullptr || g_y == nullptr)) return NVFP4_ERR_INVALID_ARG;
    if (Y == nullptr && !requant) return NVFP4_ERR_INVALID_ARG;
    if (Y != nullptr && ldy < N) return NVFP4_ERR_INVALID_ARG;
    if (K % 256 != 0 || N % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return NVFP4_OK;
    // the epilogue lives in the decode kernel's variants up to 64 rows and
    // in the CTA-pair kernel (beyond 128 rows unless the single-CTA kernel is
    // selected for comparison)
    if (M > kSkinnyMaxM && gemm_kernel_choice() == kGemmSingle) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M * (K / 16) >= kMaxBlocks || M * (N / 16) >= kMaxBlocks)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!Wq || !Ws || !g_w) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(Wq, 16) || !aligned(Ws, 16) || !aligned(g_w, 4)) return NVFP4_ERR_MISALIGNED;
    if (!aligned(bias, 16) || !aligned(Y, 2) || !aligned(Yq, 16) || !aligned(Ys, 16) ||
        !aligned(g_y, 4))
        return NVFP4_ERR_MISALIGNED;
    if (g_x != nullptr && !aligned(g_x, 4)) return NVFP4_ERR_MISALIGNED;
    const size_t need = nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED);
    if (workspace_bytes < need) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *xq = ws + kLinearHeader;
    uint8_t *xs = xq + round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    if (quantize_activation(static_cast<const uint16_t *>(X), M, K, ldx, &g_x, ws, st) !=
        cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (M <= kSkinnyExtMaxM) {
        // the re-quantization in the epilogue for a few rows (or when Y is
        // not stored, or its rows are not 16-byte aligned for the
        // quantizer's vector loads), else a dependent quantize pass over Y
        const bool y_vec = Y != nullptr && aligned(Y, 16) && ldy % 8 == 0;
        const bool in_epi = requant && (M <= kSkinnyEpiRequantMaxM || !y_vec);
        SkinnyArgs sa{Wq, Ws, g_w, xq, xs, nullptr, 0, g_x, M, N, K,
                      static_cast<uint16_t *>(Y), Y ? ldy : N, 0};
        sa.bias = static_cast<const uint16_t *>(bias);
        if (in_epi) {
            sa.g_y = g_y;
            sa.Yq = Yq;
            sa.Ys = Ys;
        }
        if (launch_gemm_skinny(sa, st) != cudaSuccess) return NVFP4_ERR_CUDA;
        if (!requant || in_epi) return NVFP4_OK;
        return from_cuda(launch_quantize(static_cast<const uint16_t *>(Y), M, N, ldy, g_y, Yq, Ys,
                                         NVFP4_SF_MMA_128x4, st));
    }
    GemmArgs a{xq, xs, g_x, Wq, Ws, g_w, M, N, K, static_cast<uint16_t *>(Y), Y ? ldy : N};
    a.bias = static_cast<const uint16_t *>(bias);
    a.g_y = g_y;
    a.Yq = Yq;
    a.Ys = Ys;
    return from_cuda(launch_gemm_pair(a, st));
}

nvfp4_status nvfp4_linear_bias_requant_dynamic(const void *X, int64_t M, int64_t K, int64_t ldx,
                                               const uint8_t *Wq, const uint8_t *Ws,
                                               const float *g_w, int64_t N, const void *bias,
                                               void *Y, int64_t ldy, float *g_y_out, uint8_t *Yq,
                                               uint8_t *Ys, const float *g_x, void *workspace,
                                               size_t workspace_bytes, void *stream) {
    nvfp4_status s = check_bf16_matrix(X, M, K, ldx);
    if (s != NVFP4_OK) return s;
    if (M < 0 || N < 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
    if (g_y_out == nullptr) return NVFP4_ERR_INVALID_ARG;
    // Y is read back by the quantizer: its rows as that quantizer's input
    s = check_bf16_matrix(Y, M, N, ldy);
    if (s != NVFP4_OK) return s;
    if (K % 256 != 0 || N % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(g_y_out, 4)) return NVFP4_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *cell = reinterpret_cast<uint32_t *>(g_y_out);
    if (M == 0 || N == 0) {
        // an empty Y has amax 0, so g_y = 1 (as nvfp4_global_scale gives)
        return (launch_cell_reset(cell, st) == cudaSuccess &&
                launch_amax_cell_to_scale(cell, st) == cudaSuccess)
                   ? NVFP4_OK
                   : NVFP4_ERR_CUDA;
    }
    if (!Y || !Yq || !Ys) return NVFP4_ERR_INVALID_ARG;
    // the epilogue: the decode kernel up to 64 rows, else the CTA-pair kernel
    if (M > kSkinnyMaxM && gemm_kernel_choice() == kGemmSingle) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M * (K / 16) >= kMaxBlocks || M * (N / 16) >= kMaxBlocks)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!Wq || !Ws || !g_w) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(Wq, 16) || !aligned(Ws, 16) || !aligned(g_w, 4)) return NVFP4_ERR_MISALIGNED;
    if (!aligned(bias, 16) || !aligned(Yq, 16) || !aligned(Ys, 16)) return NVFP4_ERR_MISALIGNED;
    if (g_x != nullptr && !aligned(g_x, 4)) return NVFP4_ERR_MISALIGNED;
    const size_t need = nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED);
    if (workspace_bytes < need) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return NVFP4_ERR_MISALIGNED;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *xq = ws + kLinearHeader;
    uint8_t *xs = xq + round_up(static_cast<size_t>(M) * static_cast<size_t>(K / 2), 256);
    // 1. X's operand; 2. the amax cell zeroed (after 1 completes); 3. the
    // GEMM, whose epilogue folds max |y| into the cell; 4. the cell turned
    // into g_y; 5. Y quantized with it (Y comes back from L2 when it fits)
    if (quantize_activation(static_cast<const uint16_t *>(X), M, K, ldx, &g_x, ws, st) !=
            cudaSuccess ||
        launch_cell_reset(cell, st) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    cudaError_t e;
    if (M <= kSkinnyExtMaxM) {
        SkinnyArgs sa{Wq, Ws, g_w, xq, xs, nullptr, 0, g_x, M, N, K,
                      static_cast<uint16_t *>(Y), ldy, 0};
        sa.bias = static_cast<const uint16_t *>(bias);
        sa.y_amax = cell;
        e = launch_gemm_skinny(sa, st);
    } else {
        GemmArgs a{xq, xs, g_x, Wq, Ws, g_w, M, N, K, static_cast<uint16_t *>(Y), ldy};
        a.bias = static_cast<const uint16_t *>(bias);
        a.y_amax = cell;
        e = launch_gemm_pair(a, st);
    }
    if (e != cudaSuccess || launch_amax_cell_to_scale(cell, st) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return from_cuda(launch_quantize(static_cast<const uint16_t *>(Y), M, N, ldy, g_y_out, Yq, Ys,
                                     NVFP4_SF_MMA_128x4, st));
}

nvfp4_status nvfp4_device_error(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(word)) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    }
    if (word & kDevErrBounds) return NVFP4_ERR_BOUNDS;
    return (word & kDevErrTimeout) ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

nvfp4_status nvfp4_debug_select_gemm_kernel(int kernel) {
    if (kernel != kGemmPair && kernel != kGemmSingle) return NVFP4_ERR_INVALID_ARG;
    debug_state().gemm_kernel = kernel;
    return NVFP4_OK;
}

nvfp4_status nvfp4_debug_capture_fused_operand(int on) {
    if (on != 0 && on != 1) return NVFP4_ERR_INVALID_ARG;
    debug_state().capture_fused_operand = on;
    return NVFP4_OK;
}

nvfp4_status nvfp4_debug_set_fault_injection(int mode, uint32_t timeout_us) {
    if (mode != 0 && mode != 1) return NVFP4_ERR_INVALID_ARG;
    debug_state().inject = mode;
    debug_state().timeout_ns =
        timeout_us == 0 ? 2000000000ull : static_cast<uint64_t>(timeout_us) * 1000ull;
    return NVFP4_OK;
}

}  // extern "C"
