// Internal launchers shared by the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "nvfp4.h"

namespace nvfp4 {

// 32-bit division by a runtime constant with a multiply-high and a shift
// (round-up reciprocal method); valid for every 32-bit dividend.
struct FastDiv {
    uint32_t d, mul, shift;
    FastDiv() : d(1), mul(0), shift(0) {}
    explicit FastDiv(uint32_t divisor) : d(divisor), mul(0), shift(0) {
        if (d > 1) {
            uint32_t s = 0;
            while ((1ull << s) < d) ++s;
            shift = s;
            mul = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - d)) / d + 1);
        }
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        if (d == 1) return n;
        return static_cast<uint32_t>(
            (static_cast<uint64_t>(__umulhi(n, mul)) + n) >> shift);
    }
};

// Slot of the current device for per-device one-time set-up (kernel
// attributes, occupancy queries, device symbols): 0 .. kMaxDevices - 1, or
// kMaxDevices when the device cannot be told.
constexpr int kMaxDevices = 64;
int device_slot();

// Per-device one-time set-up (kernel attributes, occupancy queries, device
// symbols) that host threads may reach concurrently: `init(slot)` runs
// under a lock until it first succeeds for the current device, and what it
// wrote is visible to every later caller (release / acquire on the flag).
class DeviceOnce {
  public:
    template <class F>
    cudaError_t run(F &&init) {
        const int slot = device_slot();
        if (ready_[slot].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (ready_[slot].load(std::memory_order_relaxed)) return cudaSuccess;
        const cudaError_t e = init(slot);
        if (e == cudaSuccess) ready_[slot].store(1, std::memory_order_release);
        return e;
    }

  private:
    std::mutex mu_;
    std::atomic<int> ready_[kMaxDevices + 1] = {};
};

struct LaunchCfg {
    int num_sms = 148;
};
// Launch configuration of the current device.
const LaunchCfg &launch_cfg();

// global scale (g_out doubles as the reduction cell)
cudaError_t launch_global_scale(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                float *g_out, cudaStream_t st);

cudaError_t launch_quantize(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                            const float *g, uint8_t *q, uint8_t *sf, int layout,
                            cudaStream_t st);

// Largest grid of the fused dynamic quantizer (one amax partial per CTA).
constexpr int kMaxAmaxPartials = 2048;

// Activation quantization with a dynamic global scale g = amax / (6 * 448)
// in one cooperative launch: amax partials, a grid-wide barrier on
// `counter`, then quantization; the second read of X comes from L2 when X
// fits there. The counter is zeroed by a one-thread kernel launched before
// it as a programmatic dependent of the preceding kernel (no memset, which
// would break the launch chain).
cudaError_t launch_quantize_fused(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                  uint32_t *partials, unsigned int *counter, float *g_out,
                                  uint8_t *q, uint8_t *sf, cudaStream_t st);

// The same for a small X (at most kQuantizeSmallElems elements) in one
// plain launch of a few CTAs that each reduce the amax of all of X.
constexpr int64_t kQuantizeSmallElems = 64 * 1024;
cudaError_t launch_quantize_small(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                  float *g_out, uint8_t *q, uint8_t *sf, cudaStream_t st);

// The same for a medium X (at most kQuantizeClusterElems elements) in one
// cluster of kQuantizeClusterCtas CTAs that exchange their partial amax
// through distributed shared memory. cudaErrorNotSupported (nothing
// launched) where such a cluster does not fit on the device.
constexpr int64_t kQuantizeClusterElems = 512 * 1024;
constexpr int kQuantizeClusterCtas = 16;
cudaError_t launch_quantize_cluster(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                    float *g_out, uint8_t *q, uint8_t *sf, cudaStream_t st);

// A 32-bit cell zeroed once the preceding kernel has completed (a
// programmatic dependent launch: the chain of dependent launches stays
// unbroken, as a memset would break it).
cudaError_t launch_cell_reset(uint32_t *cell, cudaStream_t st);

// The amax cell (bfloat16 magnitude bits) turned in place into the global
// scale g = amax / (6 * 448), or 1 for 0, once the preceding kernel has
// completed (a programmatic dependent launch).
cudaError_t launch_amax_cell_to_scale(uint32_t *cell, cudaStream_t st);

// Launch configuration for kernels that take part in programmatic
// dependent launch chains.
cudaLaunchAttribute pdl_attribute();

cudaError_t launch_sf_to_mma(const uint8_t *sf_rm, int64_t rows, int64_t K, uint8_t *sf_mma,
                             cudaStream_t st);

// Weight groups of a grouped projection: the weight rows (output columns)
// are `count` consecutive groups, group g ending at column end[g] (each a
// multiple of 256) with its own global scale g_b[g]. count <= 1: one group.
constexpr int kMaxGroups = 8;
struct WeightGroups {
    int count = 0;
    int end[kMaxGroups] = {};
};

// Group of output column n (ends ascending; columns past the last end
// belong to the last group).
__host__ __device__ inline int weight_group_of(const WeightGroups &w, int n) {
    int g = 0;
#pragma unroll
    for (int i = 0; i < kMaxGroups - 1; ++i) g += (i < w.count - 1 && n >= w.end[i]) ? 1 : 0;
    return g;
}

// Quantization under the four-over-six or MSE block-scale rule
// (nvfp4_scale_rule), one thread per 16-element block.
cudaError_t launch_quantize_select(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                   const float *g, int rule, uint8_t *q, uint8_t *sf, int layout,
                                   cudaStream_t st);

struct GemmArgs {
    const uint8_t *Aq, *As;
    const float *g_a;
    const uint8_t *Bq, *Bs;
    const float *g_b;
    int64_t M, N, K;
    uint16_t *Y;  // nullptr: the bfloat16 output is not stored
    int64_t ldy;
    // Epilogue extensions (CTA-pair kernel only): a bfloat16 bias of N added
    // to every row before the bfloat16 rounding, and the NVFP4 re-quantization
    // of the bfloat16 output with the decode-direction global scale *g_y into
    // Yq (M x N/2 bytes, dense) and Ys (the 128x4 tile layout, rows padded).
    const uint16_t *bias = nullptr;
    const float *g_y = nullptr;
    uint8_t *Yq = nullptr;
    uint8_t *Ys = nullptr;
    WeightGroups groups;  // g_b then points at groups.count floats
    // LoRA: L' (M x lora_r bfloat16, pre-scaled by lora_scale / (g_a g_b))
    // and the up projection (N x lora_r bfloat16) add L' B^T to the FP4
    // accumulator; lora_r in {16, 32, 48, 64}
    const uint16_t *lora_Lp = nullptr;
    const uint16_t *lora_B = nullptr;
    int64_t lora_r = 0;
    // The largest |y| of the stored bfloat16 output (rows < M), folded into
    // *y_amax (bfloat16 magnitude bits, zeroed beforehand) by atomic maxima
    uint32_t *y_amax = nullptr;
};

// The fused pass for a LoRA linear: NVFP4 codes + tile-layout scales of X
// (given g_x) and the down projection X A^T (A r x K) per K range into
// `part` (lora_partial_bytes), then L' = bf16((lora_scale / (g_x g_w)) *
// the ranges' sum, in range order).
cudaError_t launch_quantize_lora(const uint16_t *X, int64_t rows, int64_t K, int64_t ldx,
                                 const float *g_x, const float *g_w, float lora_scale,
                                 const uint16_t *A, int64_t r, uint8_t *q, uint8_t *sf,
                                 float *part, uint16_t *Lp, cudaStream_t st);
size_t lora_partial_bytes(int64_t rows, int64_t r);

// Single-CTA kernel, 128 x 256 tiles (plain epilogue only).
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t st);
// CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles: every epilogue
// extension (bias, re-quantization, LoRA stage, weight groups).
cudaError_t launch_gemm_pair(const GemmArgs &a, cudaStream_t st);
// Kernel for plain and grouped GEMMs with M > 128 (nvfp4_debug_select_gemm_kernel).
enum GemmKernel { kGemmPair = 0, kGemmSingle = 1 };
int gemm_kernel_choice();
// The plain / grouped GEMM through the selected kernel.
cudaError_t launch_gemm_plain(const GemmArgs &a, cudaStream_t st);

// Skinny-M GEMM (Y^T = W X^T, weights as the 128-row MMA operand).
constexpr int64_t kSkinnyMaxM = 128;       // activation rows it handles
constexpr int64_t kSkinnyFusedMaxM = 8;    // ... with in-kernel quantization of X
constexpr int64_t kSkinnyFusedMaxK = 6144; // ... held resident in shared memory
constexpr int64_t kSkinnyExtMaxM = 64;     // ... with the bias / re-quantization / amax epilogue
// ... re-quantizing Y in that epilogue (with a given g_y): a 16-element
// block spans 16 lanes there and the per-row work sits on few warps, so
// beyond 2 rows a dependent quantize pass over the stored Y is faster
// (27648 x 5120: M = 1 25.3 vs 31.4 us, M = 2 27.6 vs 30.2, M = 4 31.2 vs 30.7)
constexpr int64_t kSkinnyEpiRequantMaxM = 2;
struct SkinnyArgs {
    const uint8_t *Wq, *Ws;  // weights: codes (N x K/2), scales (128x4 tile layout)
    const float *g_w;
    const uint8_t *Xq, *Xs;  // unfused: activation codes (M x K/2), tile-layout scales
    const uint16_t *X;       // fused: bfloat16 activation, leading dimension ldx
    int64_t ldx;
    const float *g_x;
    int64_t M, N, K;
    uint16_t *Y;
    int64_t ldy;
    int fused;
    WeightGroups groups = {};  // g_w then points at groups.count floats
    // fused, testing hook: where CTA 0 writes the operand it quantized
    uint8_t *dbg_xq = nullptr;
    uint8_t *dbg_xs = nullptr;
    // Epilogue extensions, as GemmArgs' (N % 256 == 0 with Yq): a bfloat16
    // bias of N, the NVFP4 re-quantization of the bfloat16 output under *g_y
    // into Yq / Ys (rows padded to 128), the output's amax into *y_amax;
    // Y may then be null (not stored)
    const uint16_t *bias = nullptr;
    const float *g_y = nullptr;
    uint8_t *Yq = nullptr;
    uint8_t *Ys = nullptr;
    uint32_t *y_amax = nullptr;
};
cudaError_t launch_gemm_skinny(const SkinnyArgs &a, cudaStream_t st);

// Device address of the library's error word on the current device.
unsigned int *device_error_word();

// fault-injection state for the bounded-wait tests
struct DebugState {
    int inject = 0;
    uint64_t timeout_ns = 2000000000ull;
    int gemm_kernel = 0;  // GemmKernel for plain and grouped GEMMs with M > 128
    int capture_fused_operand = 0;  // 1: the fused decode kernel writes its operand out
};
DebugState &debug_state();

}  // namespace nvfp4
