// Dense FP4 tensor-core peak probe: every CTA issues back-to-back
// tcgen05.mma kind::mxf4nvf4 (128 x N x 64, E4M3 block scales) on
// operands that stay in shared memory, so no global traffic limits the
// rate. The measured FLOP/s is the ceiling the GEMM is compared against.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int kPeakThreads = 128;
constexpr int kSmem = 16384 + 32768 + 1024 + 1024 + 1024;

// variant: bits 0-1 select N (0: 256, 1: 128, 2: 192); bits 2-3 the number
// of accumulators the MMAs rotate through (1, 2 or 4); bit 4 adds the three
// scale copies per MMA that the GEMM issues; bit 5 issues from two warps
// (warp w owns accumulator w, each warp issuing iters / 2); bit 6 issues
// kind::f16 BF16 MMAs of 128 x N x 16 instead (calibration); bit 7 issues
// the three scale copies per MMA from a second warp, concurrently; bits 8-10
// add, after every 4 MMAs, the GEMM's per-stage bookkeeping: a tcgen05.commit
// to an mbarrier (bit 8), a tcgen05.fence::after_thread_sync (bit 9), a
// warp-wide poll of a completed mbarrier by lane 0 and a shuffle (bit 10);
// bit 11 issues, in front of every 4 MMAs, five 128-row x 32-byte scale
// copies (tcgen05.cp 128x256b) from the MMA warp itself; bit 12 polls the
// completed mbarrier with every lane instead of lane 0 + shuffle; bits 13-15
// stall the issuing warp with a dependent chain of (value * 32) integer
// multiply-adds after every 4 MMAs (queue-depth measurement).
__global__ void __launch_bounds__(kPeakThreads, 1)
    mma_peak_kernel(int iters, int variant, uint64_t timeout_ns, unsigned int *err,
                    unsigned long long *cycles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *a = smem;                   // 128 rows x 128 B (values arbitrary)
    uint8_t *b = smem + 16384;           // 256 rows x 128 B
    uint8_t *sf = smem + 16384 + 32768;  // 3 x 512 B scale tiles, all 1.0
    // bar[0..1]: one per issuing warp; bar[2]: per-stage commits; bar[3]: a
    // fresh barrier whose previous phase (parity 1) counts as complete
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
    const bool two_issuers = (variant >> 5) & 1;
    const bool copy_warp = (variant >> 7) & 1;
    if (copy_warp && warp == 1) {
        // scale copies from a second warp, 3 per MMA of warp 0, into columns
        // no MMA reads
        for (int i = 0; i < iters; ++i) {
            const uint32_t slot = 464 + static_cast<uint32_t>(i & 1) * 12;
            tmem_cp_32x128b_x4_elect(tmem + slot, sdesc_sf(smem_addr(sf)));
            tmem_cp_32x128b_x4_elect(tmem + slot + 4, sdesc_sf(smem_addr(sf + 512)));
            tmem_cp_32x128b_x4_elect(tmem + slot + 8, sdesc_sf(smem_addr(sf + 1024)));
        }
        tc_commit_elect(bar + 1);
        int ok = 1;
        if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar + 1, 0, timeout_ns) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if ((threadIdx.x & 31) == 0 && !ok) record_timeout(err);
        __syncwarp();
    }
    if (warp == 0 || (two_issuers && warp == 1)) {
        // the whole warp runs the loop; one elected lane issues
        const uint32_t n_sel = variant & 3;
        const uint32_t N = n_sel == 0 ? 256u : (n_sel == 1 ? 128u : 192u);
        const uint32_t accs = 1u << ((variant >> 2) & 3);
        const bool copies = (variant >> 4) & 1;
        const bool bf16 = (variant >> 6) & 1;
        const uint32_t sfa = tmem + 448, sfb = tmem + 452;
        if (warp == 0) {
            tmem_cp_32x128b_x4_elect(sfa, sdesc_sf(smem_addr(sf)));
            tmem_cp_32x128b_x4_elect(sfb, sdesc_sf(smem_addr(sf + 512)));
            tmem_cp_32x128b_x4_elect(sfb + 4, sdesc_sf(smem_addr(sf + 1024)));
        }
        const uint32_t idesc = bf16 ? idesc_bf16(128, N) : idesc_mxf4nvf4(128, N);
        const uint64_t ad = sdesc_sw128(smem_addr(a)), bd = sdesc_sw128(smem_addr(b));
        const int my_iters = two_issuers ? iters / 2 : iters;
        const uint32_t acc_base = two_issuers ? static_cast<uint32_t>(warp) * N : 0u;
        const uint32_t first = two_issuers ? 1u : accs;
        const unsigned long long t0 = clock64();
        for (int i = 0; i < my_iters; ++i) {
            if (copies) {  // the GEMM's per-MMA scale traffic: 1 + 2 copies
                const uint32_t slot = 464 + static_cast<uint32_t>(i & 1) * 12;
                tmem_cp_32x128b_x4_elect(tmem + slot, sdesc_sf(smem_addr(sf)));
                tmem_cp_32x128b_x4_elect(tmem + slot + 4, sdesc_sf(smem_addr(sf + 512)));
                tmem_cp_32x128b_x4_elect(tmem + slot + 8, sdesc_sf(smem_addr(sf + 1024)));
            }
            const uint32_t acc = two_issuers ? acc_base : (static_cast<uint32_t>(i) % accs) * N;
            const uint64_t koff = static_cast<uint64_t>(i & 3) * 2;
            if (bf16)
                mma_bf16_elect(tmem + acc, ad + koff, bd + koff, idesc,
                               i >= static_cast<int>(first));
            else
                mma_mxf4nvf4_elect(tmem + acc, ad + koff, bd + koff, idesc, sfa, sfb,
                                   i >= static_cast<int>(first));
            if ((i & 3) == 0 && ((variant >> 11) & 1)) {
                // 4 KiB source images (contents irrelevant to the timing)
                for (int c = 0; c < 5; ++c)
                    tmem_cp_128x256b_elect(tmem + 464 + 8 * static_cast<uint32_t>(c),
                                           sdesc_128x32(smem_addr(smem)));
            }
            if ((i & 3) == 3 && ((variant >> 13) & 7)) {
                uint32_t x = static_cast<uint32_t>(i);
                const int n = 32 * ((variant >> 13) & 7);
                for (int k = 0; k < n; ++k) asm volatile("mad.lo.u32 %0, %0, 3, 1;" : "+r"(x));
                if (x == 0xFFFFFFFFu) record_timeout(err);  // keeps the chain live
            }
            if ((i & 3) == 3) {
                if ((variant >> 12) & 1) {
                    if (!mbar_try_wait(smem_addr(bar + 3), 1)) record_timeout(err);
                }
                if ((variant >> 8) & 1) tc_commit_elect(bar + 2);
                if ((variant >> 9) & 1) tc_fence_after();
                if ((variant >> 10) & 1) {
                    int done = 0;
                    if ((threadIdx.x & 31) == 0) done = mbar_try_wait(smem_addr(bar + 3), 1) ? 1 : 0;
                    done = __shfl_sync(0xFFFFFFFFu, done, 0);
                    if (!done) record_timeout(err);
                }
            }
        }
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_mma_peak(int ctas, int iters, int variant, unsigned long long *cycles,
                            cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorInvalidSymbol;
    mma_peak_kernel<<<ctas, kPeakThreads, kSmem, st>>>(iters, variant,
                                                        debug_state().timeout_ns, err, cycles);
    return cudaGetLastError();
}

}  // namespace nvfp4
