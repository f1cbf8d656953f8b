// Dense FP4 tensor-core peak probe (measurement library libnvfp4_probe.so,
// declared in include/nvfp4_probe.h; not part of the linear-layer library):
// every CTA issues back-to-back tcgen05.mma kind::mxf4nvf4 (128 x N x 64,
// E4M3 block scales) on operands that stay in shared memory, so no global
// traffic limits the rate. The measured FLOP/s is the ceiling the GEMM is
// compared against.
//
// The issuing loop is specialised at compile time per variant and unrolled
// by 4 with constant descriptor offsets: with run-time variant tests inside
// the loop the warp's own scalar work, not the tensor core, set the rate.
#include <cuda_runtime.h>

#include <cstdint>

#include "nvfp4_probe.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // bounded waits: 2 s

// The probe's own error word (bounded waits that ran out).
__device__ unsigned int g_probe_error = 0;

int device_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kMaxDevices;
    return dev;
}

unsigned int *device_error_word() {
    static unsigned int *addr[kMaxDevices] = {};
    const int dev = device_slot();
    if (dev == kMaxDevices) return nullptr;
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_probe_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

constexpr int kPeakThreads = 128;
constexpr int kSmem = 16384 + 32768 + 1024 + 1024 + 1024;

enum Variant {
    kFp4N256 = 0,      // 128 x 256 x 64, one accumulator
    kFp4N128 = 1,      // 128 x 128 x 64
    kFp4TwoWarps = 2,  // 128 x 128 x 64 from two warps, one accumulator each
    kFp4Copies = 3,    // + the GEMM's 3 scale copies per MMA, same thread
    kFp4CopyWarp = 4,  // + 3 scale copies per MMA from a second warp
    kFp4Stage = 5,     // + per 4 MMAs: commit, mbarrier poll, fence (a GEMM stage)
    kBf16N256 = 6,     // kind::f16 BF16 128 x 256 x 16 (calibration)
    kFp4Pair = 7,      // CTA pair (cta_group::2): 256 x 256 x 64 per instruction
};

// One FP4 MMA under one elect; with COPIES, the step's three scale copies
// (A tile, two 128-row B tiles) first.
template <bool COPIES>
__device__ __forceinline__ void fp4_step(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc, uint64_t da,
                                         uint64_t db0, uint64_t db1) {
    if (COPIES) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 t;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "add.u32 t, %6, 4;\n\t"
            "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%5], %7;\n\t"
            "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%6], %8;\n\t"
            "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], %9;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
            " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb), "l"(da), "l"(db0),
            "l"(db1)
            : "memory");
    } else {
        mma_mxf4nvf4_elect(d, a, b, idesc, sfa, sfb, acc);
    }
}

// `iters` MMAs (a multiple of 4) from this warp into accumulator `acc_col`.
template <int V>
__device__ __forceinline__ void issue_loop(uint32_t tmem, uint32_t acc_col, int iters,
                                           uint64_t ad, uint64_t bd, uint32_t sf_col,
                                           uint64_t da, uint64_t db0, uint64_t db1,
                                           uint64_t *poll_bar, uint64_t *commit_bar,
                                           unsigned int *err) {
    constexpr uint32_t N = (V == kFp4N128 || V == kFp4TwoWarps) ? 128u : 256u;
    constexpr uint32_t idesc = V == kBf16N256 ? idesc_bf16(128, N) : idesc_mxf4nvf4(128, N);
    const uint32_t sfa = tmem + sf_col, sfb = sfa + 4;
    for (int i = 0; i < iters; i += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (i | k) != 0;
            if (V == kBf16N256)
                mma_bf16_elect(tmem + acc_col, ad + 2 * k, bd + 2 * k, idesc, acc);
            else
                fp4_step<V == kFp4Copies>(tmem + acc_col, ad + 2 * k, bd + 2 * k, idesc, sfa, sfb,
                                          acc, da, db0, db1);
        }
        if (V == kFp4Stage) {
            tc_commit_elect(commit_bar);
            int done = 0;
            if ((threadIdx.x & 31) == 0) done = mbar_try_wait(smem_addr(poll_bar), 1) ? 1 : 0;
            done = __shfl_sync(0xFFFFFFFFu, done, 0);
            if (!done) record_timeout(err);  // the fresh barrier's previous phase is complete
            tc_fence_after();
        }
    }
}

template <int V>
__global__ void __launch_bounds__(kPeakThreads, 1)
    mma_peak_kernel(int iters, uint64_t timeout_ns, unsigned int *err,
                    unsigned long long *cycles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *a = smem;                   // 128 rows x 128 B
    uint8_t *b = smem + 16384;           // 256 rows x 128 B
    uint8_t *sf = smem + 16384 + 32768;  // 3 x 512 B scale tiles, all 1.0
    // bar[0..1]: completion per issuing warp; bar[2]: per-stage commits;
    // bar[3]: a fresh barrier whose previous phase (parity 1) counts as done
    uint64_t *bar = reinterpret_cast<uint64_t *>(sf + 1536);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 4);

    // operands: codes 0x22 (1.0, 1.0), scales 0x38 (1.0)
    for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(smem)[i] = 0x22222222u;
    for (int i = threadIdx.x; i < 1536 / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(sf)[i] = 0x38383838u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(bar + i, 1);
        fence_mbar_init();
    }
    fence_proxy_async_shared();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t ad = sdesc_sw128(smem_addr(a)), bd = sdesc_sw128(smem_addr(b));
    const uint64_t da = sdesc_sf(smem_addr(sf)), db0 = sdesc_sf(smem_addr(sf + 512)),
                   db1 = sdesc_sf(smem_addr(sf + 1024));
    constexpr bool two = V == kFp4TwoWarps;
    if (warp == 0 || (two && warp == 1)) {
        // scales for the MMAs: columns 448 (A) and 452..459 (B)
        if (warp == 0) {
            tmem_cp_32x128b_x4_elect(tmem + 448, da);
            tmem_cp_32x128b_x4_elect(tmem + 452, db0);
            tmem_cp_32x128b_x4_elect(tmem + 456, db1);
        }
        if (two) {
            // both warps' MMAs read the scales warp 0 copied
            if (warp == 0) tc_commit_elect(bar + 2);
            int ok = 1;
            if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar + 2, 0, timeout_ns) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok && (threadIdx.x & 31) == 0) record_timeout(err);
            tc_fence_after();
        }
        const int my_iters = two ? iters / 2 : iters;
        const unsigned long long t0 = clock64();
        issue_loop<V>(tmem, two ? static_cast<uint32_t>(warp) * 128u : 0u, my_iters, ad, bd, 448,
                      da, db0, db1, bar + 3, bar + 2, err);
        tc_commit_elect(bar + warp);
        int ok = 1;
        if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar + warp, 0, timeout_ns) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        const unsigned long long t1 = clock64();
        if ((threadIdx.x & 31) == 0) {
            if (!ok) record_timeout(err);
            if (blockIdx.x == 0 && warp == 0) *cycles = t1 - t0;
        }
        __syncwarp();
    } else if (V == kFp4CopyWarp && warp == 1) {
        // the three scale copies per MMA of warp 0, into columns no MMA reads
        for (int i = 0; i < iters; ++i) {
            const uint32_t slot = tmem + 464 + static_cast<uint32_t>(i & 1) * 12;
            tmem_cp_32x128b_x4_elect(slot, da);
            tmem_cp_32x128b_x4_elect(slot + 4, db0);
            tmem_cp_32x128b_x4_elect(slot + 8, db1);
        }
        tc_commit_elect(bar + 1);
        int ok = 1;
        if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar + 1, 0, timeout_ns) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if ((threadIdx.x & 31) == 0 && !ok) record_timeout(err);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// CTA-pair form: clusters of 2, rank 0 issues 256 x 256 x 64 MMAs whose
// halves run on both SMs (each holds 128 rows of A and of B, same offsets).
__global__ void __launch_bounds__(kPeakThreads, 1)
    mma_peak_pair_kernel(int iters, uint64_t timeout_ns, unsigned int *err,
                         unsigned long long *cycles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *a = smem;                   // 128 rows x 128 B
    uint8_t *b = smem + 16384;           // 128 rows x 128 B (this CTA's half of B)
    uint8_t *sf = smem + 16384 + 32768;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sf + 1536);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 4);
    for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(smem)[i] = 0x22222222u;
    for (int i = threadIdx.x; i < 1536 / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(sf)[i] = 0x38383838u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(bar + i, 1);
        fence_mbar_init();
    }
    fence_proxy_async_shared();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp == 0 && cluster_ctarank() == 0) {
        const uint64_t ad = sdesc_sw128(smem_addr(a)), bd = sdesc_sw128(smem_addr(b));
        const uint64_t da = sdesc_sf(smem_addr(sf)), db0 = sdesc_sf(smem_addr(sf + 512)),
                       db1 = sdesc_sf(smem_addr(sf + 1024));
        sf_copy3_pair_elect(tmem + 448, tmem + 452, da, db0, db1);
        constexpr uint32_t idesc = idesc_mxf4nvf4(256, 256);
        const unsigned long long t0 = clock64();
        for (int i = 0; i < iters; i += 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_mxf4nvf4_pair_elect(tmem, ad + 2 * k, bd + 2 * k, idesc, tmem + 448,
                                        tmem + 452, (i | k) != 0);
        }
        tc_commit_pair_mc_elect(bar + 0, 0x1);
        int ok = 1;
        if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar + 0, 0, timeout_ns) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        const unsigned long long t1 = clock64();
        if ((threadIdx.x & 31) == 0) {
            if (!ok) record_timeout(err);
            if (blockIdx.x == 0) *cycles = t1 - t0;
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the partner's TMEM and shared memory outlive the MMAs
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

cudaError_t launch_pair(int ctas, int iters, unsigned long long *cycles, cudaStream_t st) {
    static bool attr_of[kMaxDevices + 1] = {};
    bool &attr = attr_of[device_slot()];
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(mma_peak_pair_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorInvalidSymbol;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas & ~1, 1, 1);
    cfg.blockDim = dim3(kPeakThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mma_peak_pair_kernel, iters, kTimeoutNs, err,
                              cycles);
}

template <int V>
cudaError_t launch_v(int ctas, int iters, unsigned long long *cycles, cudaStream_t st) {
    static bool attr_of[kMaxDevices + 1] = {};
    bool &attr = attr_of[device_slot()];
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel<V>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorInvalidSymbol;
    mma_peak_kernel<V><<<ctas, kPeakThreads, kSmem, st>>>(iters, kTimeoutNs, err,
                                                          cycles);
    return cudaGetLastError();
}

cudaError_t launch_mma_peak(int ctas, int iters, int variant, unsigned long long *cycles,
                            cudaStream_t st) {
    switch (variant) {
        case kFp4N256: return launch_v<kFp4N256>(ctas, iters, cycles, st);
        case kFp4N128: return launch_v<kFp4N128>(ctas, iters, cycles, st);
        case kFp4TwoWarps: return launch_v<kFp4TwoWarps>(ctas, iters, cycles, st);
        case kFp4Copies: return launch_v<kFp4Copies>(ctas, iters, cycles, st);
        case kFp4CopyWarp: return launch_v<kFp4CopyWarp>(ctas, iters, cycles, st);
        case kFp4Stage: return launch_v<kFp4Stage>(ctas, iters, cycles, st);
        case kBf16N256: return launch_v<kBf16N256>(ctas, iters, cycles, st);
        case kFp4Pair: return launch_pair(ctas, iters, cycles, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace nvfp4

extern "C" {

NVFP4_PROBE_API int nvfp4_mma_peak_probe(int ctas, int iters, int variant, unsigned long long *cycles,
                         void *stream) {
    if (ctas <= 0 || iters <= 0 || cycles == nullptr) return 1;
    if (variant < 0 || variant > 7) return 1;
    if (variant == 7 && ctas < 2) return 1;  // clusters of 2
    // unrolled by 4 MMAs per warp; variant 2 splits them over two warps
    if (iters % (variant == 2 ? 8 : 4) != 0) return 1;
    if ((reinterpret_cast<uintptr_t>(cycles) & 7) != 0) return 2;
    return nvfp4::launch_mma_peak(ctas, iters, variant, cycles, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? 0
               : 5;
}

NVFP4_PROBE_API int nvfp4_probe_error(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return 5;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, nvfp4::g_probe_error, sizeof(word)) != cudaSuccess) return 5;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(nvfp4::g_probe_error, &zero, sizeof(zero)) != cudaSuccess) return 5;
    }
    return word ? 6 : 0;
}

}  // extern "C"
