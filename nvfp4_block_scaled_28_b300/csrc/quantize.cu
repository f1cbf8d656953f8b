// NVFP4 quantization kernels: per-tensor amax -> global scale, the
// bandwidth-bound bfloat16 -> NVFP4 quantizer, and the scale-layout
// permutation used by the tensor-core GEMM.
//
// Format ("nvfp4-gemma4" page, section 2; "nvfp4-difusion" page, section 2):
// E2M1 codes two per byte, one E4M3 scale per 16 consecutive elements.
// Scale rule (absmax, the same section's table) with the decode-direction
// global scale g of this library:
//   S = E4M3_rne_satfinite((amax_block / 6) / g)
//   r = 1 / (e4m3(S) * g)   (0 when S == 0)
//   code = E2M1_rne_satfinite(x * r), sign bit = sign bit of x.
// Every float step is one IEEE binary32 operation (explicit _rn intrinsics,
// never contracted), so the bytes do not depend on compiler flags.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;


// One warp-uniform round of U blocks per lane: blocks i = base + lane +
// u * stride (stride a multiple of 32, base of the warp's lane 0). All loads
// are issued before the math. The four scale bytes of blocks 4j..4j+3 are
// consecutive in both layouts (K / 16 is a multiple of 4 in the tile
// layout), so lane 4j gathers them by shuffle and stores one 32-bit word
// where it is aligned and whole (kGather; fewer store transactions for
// HBM-bound runs); otherwise each lane stores its byte.
// Blocks in [total, total_pad) are padding rows of the tile layout: scale 0.
template <int kLayout, int U, bool kGather>
__device__ __forceinline__ void quantize_round(const uint16_t *__restrict__ X, uint32_t base,
                                               uint32_t stride, uint32_t total,
                                               uint32_t total_pad, uint32_t kbpr, uint64_t ldx,
                                               FastDiv div_kbpr, float g, const float *rtab,
                                               uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t kb4 = kbpr >> 2;
    uint4 va[U], vb[U];
    uint32_t row[U], kb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = base + lane + u * stride;
        row[u] = div_kbpr.div(i);
        kb[u] = i - row[u] * kbpr;
        va[u] = make_uint4(0, 0, 0, 0);
        vb[u] = va[u];
        if (i < total && NVFP4_CHECK(row[u] < total / kbpr && kb[u] < kbpr)) {
            const uint4 *src = reinterpret_cast<const uint4 *>(X + row[u] * ldx + kb[u] * 16ull);
            va[u] = ld_stream(src);
            vb[u] = ld_stream(src + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = base + lane + u * stride;
        uint32_t S = 0, lo, hi;
        if (i < total) {
            S = quantize16_tab(va[u], vb[u], g, rtab, lo, hi);
            *reinterpret_cast<uint2 *>(q + static_cast<uint64_t>(i) * 8) = make_uint2(lo, hi);
        }
        // the scale buffer holds `total` bytes (row-major) or the tiles of
        // the rows padded to 128 (tile layout)
        [[maybe_unused]] const uint64_t sf_end = kLayout == NVFP4_SF_ROW_MAJOR
                                    ? static_cast<uint64_t>(total)
                                    : static_cast<uint64_t>((total / kbpr + 127) / 128 * 128) * kbpr;
        const uint32_t end = kLayout == NVFP4_SF_ROW_MAJOR ? total : total_pad;
        const uint64_t off = kLayout == NVFP4_SF_ROW_MAJOR
                                 ? static_cast<uint64_t>(i)
                                 : ((static_cast<uint64_t>(row[u] >> 7) * kb4 + (kb[u] >> 2)) << 9) +
                                       ((row[u] & 31u) << 4) + (((row[u] & 127u) >> 5) << 2) +
                                       (kb[u] & 3u);
        if (!kGather) {
            if (i < end && NVFP4_CHECK(off < sf_end)) sf[off] = static_cast<uint8_t>(S);
            continue;
        }
        const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, S, 1);
        const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, S, 2);
        const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, S, 3);
        const bool whole = (i & 3u) == 0 && i + 3 < end &&
                           ((reinterpret_cast<uintptr_t>(sf) + off) & 3u) == 0;
        if (whole) {
            if (NVFP4_CHECK(off + 3 < sf_end))
                *reinterpret_cast<uint32_t *>(sf + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
        } else if (i < end) {
            // the lane leading a whole group stored this byte already
            const uint32_t lead = i & ~3u;
            const uint64_t lead_off = off - (i - lead);
            const bool lead_whole = lead + 3 < end &&
                                    ((reinterpret_cast<uintptr_t>(sf) + lead_off) & 3u) == 0;
            if ((!lead_whole || (i & 3u) == 0) && NVFP4_CHECK(off < sf_end))
                sf[off] = static_cast<uint8_t>(S);
        }
    }
}

// Warp-uniform rounds of 4 blocks per lane over all blocks; in the tile
// layout also the blocks of the padding rows up to the next multiple of 128
// (scale 0). Launched in plain stream order (measured: as a programmatic
// dependent of the GEMM before it, the given-g linear took 3.5 us longer);
// the GEMM after it may start its set-up early.
template <int kLayout>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const uint16_t *__restrict__ X,
                                                            uint32_t rows, uint32_t rows_pad,
                                                            uint32_t kbpr, uint64_t ldx,
                                                            FastDiv div_kbpr,
                                                            const float *__restrict__ g_ptr,
                                                            uint8_t *__restrict__ q,
                                                            uint8_t *__restrict__ sf) {
    pdl_launch_dependents();
    const float g = *g_ptr;
    __shared__ float rtab[128];
    fill_recip_table(rtab, g);
    __syncthreads();
    const uint32_t total = rows * kbpr;
    const uint32_t total_pad = rows_pad * kbpr;
    const uint32_t stride = gridDim.x * blockDim.x;
    constexpr int U = 4;
    for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total_pad;
         base += U * stride)
        quantize_round<kLayout, U, true>(X, base, stride, total, total_pad, kbpr, ldx, div_kbpr,
                                         g, rtab, q, sf);
}

// amax(|X|) over 16-byte vectors as a bfloat16 magnitude bit pattern,
// combined across the grid with atomicMax on `cell` (zeroed by the kernel
// before it, which this one waits for, as it may also have written X).
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t *__restrict__ X,
                                                        uint32_t rows, uint32_t vpr,
                                                        uint64_t ldx, FastDiv div_vpr,
                                                        uint32_t *cell) {
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t total = rows * vpr;
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t acc = 0;
    uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < total; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t j = i + u * stride;
            const uint32_t r = div_vpr.div(j), c = j - r * vpr;
            v[u] = (NVFP4_CHECK(r < rows && c < vpr)
                        ? ld_stream(reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull))
                        : make_uint4(0, 0, 0, 0));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc = max_u16x2(acc, max_u16x2(max_u16x2(v[u].x & m, v[u].y & m),
                                           max_u16x2(v[u].z & m, v[u].w & m)));
        }
    }
    for (; i < total; i += stride) {
        const uint32_t r = div_vpr.div(i), c = i - r * vpr;
        const uint4 v = (NVFP4_CHECK(r < rows && c < vpr)
                        ? ld_stream(reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull))
                        : make_uint4(0, 0, 0, 0));
        acc = max_u16x2(acc, max_u16x2(max_u16x2(v.x & m, v.y & m), max_u16x2(v.z & m, v.w & m)));
    }
    uint32_t a = max(acc & 0xFFFFu, acc >> 16);
    a = __reduce_max_sync(0xFFFFFFFFu, a);
    __shared__ uint32_t warp_max[kThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t b = threadIdx.x < kThreads / 32 ? warp_max[threadIdx.x] : 0u;
        b = __reduce_max_sync(0xFFFFFFFFu, b);
        if (threadIdx.x == 0 && b != 0) atomicMax(cell, b);
    }
}

// Dynamic activation quantization in one launch: every CTA reduces the amax
// of its share of X into partials[blockIdx.x], the grid meets at a barrier
// (all CTAs are co-resident: cooperative launch), then every CTA reduces
// the same partials to the same g (integer max, one IEEE division) and
// quantizes into the tensor-core scale layout. The second read of X hits L2
// when X fits there. `counter` is zero at launch. The barrier wait is
// bounded: on timeout the CTA records it in the error word and goes on.
__global__ void __launch_bounds__(kThreads) quantize_fused_kernel(
    const uint16_t *__restrict__ X, uint32_t rows, uint32_t rows_pad, uint32_t kbpr, uint64_t ldx,
    FastDiv div_kbpr, uint32_t vpr, FastDiv div_vpr, uint32_t *partials, unsigned int *counter,
    float *g_out, uint8_t *__restrict__ q, uint8_t *__restrict__ sf, uint64_t timeout_ns,
    unsigned int *err) {
    pdl_launch_dependents();
    pdl_wait();  // X may come from the previous kernel
    // ---- amax of this CTA's share (16-byte vectors, 4 in flight)
    {
        const uint32_t total = rows * vpr;
        const uint32_t stride = gridDim.x * blockDim.x;
        const uint32_t m = 0x7FFF7FFFu;
        uint32_t acc = 0;
        uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
        for (; i + 7 * stride < total; i += 8 * stride) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t j = i + u * stride;
                const uint32_t r = div_vpr.div(j), c = j - r * vpr;
                v[u] = (NVFP4_CHECK(r < rows && c < vpr)
                        ? ld_stream(reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull))
                        : make_uint4(0, 0, 0, 0));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                acc = max_u16x2(acc, max_u16x2(max_u16x2(v[u].x & m, v[u].y & m),
                                               max_u16x2(v[u].z & m, v[u].w & m)));
        }
        for (; i < total; i += stride) {
            const uint32_t r = div_vpr.div(i), c = i - r * vpr;
            const uint4 v = (NVFP4_CHECK(r < rows && c < vpr)
                        ? ld_stream(reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull))
                        : make_uint4(0, 0, 0, 0));
            acc = max_u16x2(acc,
                            max_u16x2(max_u16x2(v.x & m, v.y & m), max_u16x2(v.z & m, v.w & m)));
        }
        uint32_t a = max(acc & 0xFFFFu, acc >> 16);
        a = __reduce_max_sync(0xFFFFFFFFu, a);
        __shared__ uint32_t warp_max[kThreads / 32];
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t b = threadIdx.x < kThreads / 32 ? warp_max[threadIdx.x] : 0u;
            b = __reduce_max_sync(0xFFFFFFFFu, b);
            if (threadIdx.x == 0) {
                partials[blockIdx.x] = b;
                __threadfence();
                atomicAdd(counter, 1u);
                // wait for every CTA's partial
                const uint64_t t0 = global_timer_ns();
                while (atomicAdd(counter, 0u) < gridDim.x) {
                    if (global_timer_ns() - t0 > timeout_ns) {
                        record_timeout(err);
                        break;
                    }
                }
                __threadfence();
            }
        }
        __syncthreads();
    }
    // ---- g from all partials (the same value in every CTA)
    __shared__ float g_sh;
    if (threadIdx.x < 32) {
        uint32_t b = 0;
        for (uint32_t i = threadIdx.x; i < gridDim.x; i += 32)
            b = max(b, *reinterpret_cast<volatile uint32_t *>(partials + i));
        b = __reduce_max_sync(0xFFFFFFFFu, b);
        if (threadIdx.x == 0) {
            const float amax = __uint_as_float(b << 16);
            g_sh = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
        }
    }
    __syncthreads();
    const float g = g_sh;
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    __shared__ float rtab[128];
    fill_recip_table(rtab, g);
    __syncthreads();
    // ---- quantize (padding rows of the last 128-row group get scale 0)
    const uint32_t total = rows * kbpr;
    const uint32_t total_pad = rows_pad * kbpr;
    const uint32_t stride = gridDim.x * blockDim.x;
    constexpr int U = 4;
    for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total_pad;
         base += U * stride)
        quantize_round<NVFP4_SF_MMA_128x4, U, false>(X, base, stride, total, total_pad, kbpr, ldx,
                                                     div_kbpr, g, rtab, q, sf);
}

// Dynamic quantization of a small activation (decode rows) in one plain
// launch: every CTA reduces the amax of all of X itself (a few hundred KB
// from L2), so all CTAs hold the same g (integer max, one IEEE division)
// without a grid barrier; CTA 0 stores it; each CTA then quantizes its
// share into the tensor-core scale layout.
__global__ void __launch_bounds__(kThreads) quantize_small_kernel(
    const uint16_t *__restrict__ X, uint32_t rows, uint32_t rows_pad, uint32_t kbpr, uint64_t ldx,
    FastDiv div_kbpr, uint32_t vpr, FastDiv div_vpr, float *g_out, uint8_t *__restrict__ q,
    uint8_t *__restrict__ sf) {
    pdl_launch_dependents();
    pdl_wait();  // X may come from the previous kernel
    __shared__ float g_sh;
    {
        const uint32_t total = rows * vpr;
        const uint32_t m = 0x7FFF7FFFu;
        uint32_t acc = 0;
        // eight 16-byte loads in flight per thread
        uint32_t i = threadIdx.x;
        for (; i + 7 * blockDim.x < total; i += 8 * blockDim.x) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t j = i + u * blockDim.x;
                const uint32_t r = div_vpr.div(j), c = j - r * vpr;
                v[u] = NVFP4_CHECK(r < rows && c < vpr)
                         ? *reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull)
                         : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                acc = max_u16x2(acc, max_u16x2(max_u16x2(v[u].x & m, v[u].y & m),
                                               max_u16x2(v[u].z & m, v[u].w & m)));
        }
        for (; i < total; i += blockDim.x) {
            const uint32_t r = div_vpr.div(i), c = i - r * vpr;
            const uint4 v = NVFP4_CHECK(r < rows && c < vpr)
                         ? *reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull)
                         : make_uint4(0, 0, 0, 0);
            acc = max_u16x2(acc,
                            max_u16x2(max_u16x2(v.x & m, v.y & m), max_u16x2(v.z & m, v.w & m)));
        }
        uint32_t a = max(acc & 0xFFFFu, acc >> 16);
        a = __reduce_max_sync(0xFFFFFFFFu, a);
        __shared__ uint32_t warp_max[kThreads / 32];
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t b = threadIdx.x < kThreads / 32 ? warp_max[threadIdx.x] : 0u;
            b = __reduce_max_sync(0xFFFFFFFFu, b);
            if (threadIdx.x == 0) {
                const float amax = __uint_as_float(b << 16);
                g_sh = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
            }
        }
        __syncthreads();
    }
    const float g = g_sh;
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    __shared__ float rtab[128];
    fill_recip_table(rtab, g);
    __syncthreads();
    const uint32_t total = rows * kbpr;
    const uint32_t total_pad = rows_pad * kbpr;
    const uint32_t stride = gridDim.x * blockDim.x;
    constexpr int U = 4;
    for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total_pad;
         base += U * stride)
        quantize_round<NVFP4_SF_MMA_128x4, U, false>(X, base, stride, total, total_pad, kbpr, ldx,
                                                     div_kbpr, g, rtab, q, sf);
}

// Dynamic quantization of a medium activation (decode rows beyond the small
// kernel's reach) by one thread-block cluster: each CTA reduces the amax of
// its share of X, writes it into slot `rank` of every CTA's shared array
// (distributed shared memory), and after one cluster barrier every CTA
// holds all partials, hence the same g (integer max, one IEEE division),
// without a grid barrier or a zeroed counter. CTA 0 stores g; each CTA then
// quantizes its share of the blocks (the second read of X hits L2).
constexpr int kClusterThreads = 1024;  // one round of loads per phase at decode sizes

__global__ void __launch_bounds__(kClusterThreads) quantize_cluster_kernel(
    const uint16_t *__restrict__ X, uint32_t rows, uint32_t rows_pad, uint32_t kbpr, uint64_t ldx,
    FastDiv div_kbpr, uint32_t vpr, FastDiv div_vpr, float *g_out, uint8_t *__restrict__ q,
    uint8_t *__restrict__ sf) {
    __shared__ uint32_t part[kQuantizeClusterCtas];
    __shared__ float g_sh;
    const uint32_t rank = cluster_ctarank();
    const uint32_t csize = gridDim.x;  // one cluster
    pdl_launch_dependents();
    pdl_wait();  // X may come from the previous kernel
    {
        const uint32_t total = rows * vpr;
        const uint32_t per = (total + csize - 1) / csize;
        const uint32_t lo = rank * per;
        const uint32_t hi = lo + per < total ? lo + per : total;
        const uint32_t m = 0x7FFF7FFFu;
        uint32_t acc = 0;
        uint32_t i = lo + threadIdx.x;
        for (; i + 7 * blockDim.x < hi; i += 8 * blockDim.x) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t j = i + u * blockDim.x;
                const uint32_t r = div_vpr.div(j), c = j - r * vpr;
                v[u] = NVFP4_CHECK(r < rows && c < vpr)
                         ? *reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull)
                         : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                acc = max_u16x2(acc, max_u16x2(max_u16x2(v[u].x & m, v[u].y & m),
                                               max_u16x2(v[u].z & m, v[u].w & m)));
        }
        for (; i < hi; i += blockDim.x) {
            const uint32_t r = div_vpr.div(i), c = i - r * vpr;
            const uint4 v = NVFP4_CHECK(r < rows && c < vpr)
                         ? *reinterpret_cast<const uint4 *>(X + r * ldx + c * 8ull)
                         : make_uint4(0, 0, 0, 0);
            acc = max_u16x2(acc,
                            max_u16x2(max_u16x2(v.x & m, v.y & m), max_u16x2(v.z & m, v.w & m)));
        }
        uint32_t a = max(acc & 0xFFFFu, acc >> 16);
        a = __reduce_max_sync(0xFFFFFFFFu, a);
        __shared__ uint32_t warp_max[kClusterThreads / 32];
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t b = threadIdx.x < kClusterThreads / 32 ? warp_max[threadIdx.x] : 0u;
            b = __reduce_max_sync(0xFFFFFFFFu, b);
            // this CTA's partial into slot `rank` of every CTA of the cluster
            if (threadIdx.x < csize && NVFP4_CHECK(rank < kQuantizeClusterCtas))
                st_cluster_u32(mapa_shared(smem_addr(&part[rank]), threadIdx.x), b);
        }
    }
    cluster_sync_all();  // every partial is in every CTA's array
    if (threadIdx.x < 32) {
        uint32_t b = threadIdx.x < csize ? part[threadIdx.x] : 0u;
        b = __reduce_max_sync(0xFFFFFFFFu, b);
        if (threadIdx.x == 0) {
            const float amax = __uint_as_float(b << 16);
            g_sh = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
        }
    }
    __syncthreads();
    const float g = g_sh;
    if (rank == 0 && threadIdx.x == 0) *g_out = g;
    __shared__ float rtab[128];
    fill_recip_table(rtab, g);
    __syncthreads();
    const uint32_t total = rows * kbpr;
    const uint32_t total_pad = rows_pad * kbpr;
    const uint32_t stride = csize * blockDim.x;
    constexpr int U = 4;
    for (uint32_t base = rank * blockDim.x + (threadIdx.x & ~31u); base < total_pad;
         base += U * stride)
        quantize_round<NVFP4_SF_MMA_128x4, U, false>(X, base, stride, total, total_pad, kbpr, ldx,
                                                     div_kbpr, g, rtab, q, sf);
}

// Zeroes a 32-bit cell (the cooperative quantizer's barrier counter, an
// amax cell), as a programmatic dependent of the kernel before it: it may
// be resident early, and it writes only once that kernel has completed. In
// the linear layer's launch sequence that kernel is the one before this
// call's first use of the cell, which itself waited for the previous use.
__global__ void counter_reset_kernel(unsigned int *counter) {
    pdl_launch_dependents();
    pdl_wait();
    *counter = 0u;
}

// An amax cell (bfloat16 magnitude bits) into the global scale, in place,
// once the kernel that accumulated it has completed. The next kernel is let
// in only then: started earlier, its CTAs would sit on the SMs that the
// amax reduction is still using.
__global__ void amax_cell_to_scale_kernel(uint32_t *cell) {
    pdl_wait();
    pdl_launch_dependents();
    const float amax = __uint_as_float(*cell << 16);
    const float g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
    *reinterpret_cast<float *>(cell) = g;
}

// Row-major scales -> 128x4 tile layout; one thread per group of 4 scales.
__global__ void __launch_bounds__(kThreads) sf_to_mma_kernel(const uint8_t *__restrict__ src,
                                                             uint32_t rows, uint32_t rows_pad,
                                                             uint32_t kb4, FastDiv div_kb4,
                                                             uint8_t *__restrict__ dst) {
    const uint32_t total = rows_pad * kb4;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += gridDim.x * blockDim.x) {
        const uint32_t row = div_kb4.div(i), G = i - row * kb4;
        uint32_t v = 0;
        if (row < rows && NVFP4_CHECK(static_cast<uint64_t>(i) * 4 + 4 <= uint64_t(rows) * kb4 * 4))
            v = *reinterpret_cast<const uint32_t *>(src + static_cast<uint64_t>(i) * 4);
        const uint64_t off = sf_mma_offset(row, G * 4, kb4);
        if (NVFP4_CHECK(off + 4 <= static_cast<uint64_t>(total) * 4))
            *reinterpret_cast<uint32_t *>(dst + off) = v;
    }
}

int grid_for(uint64_t work_items, int per_thread) {
    const uint64_t threads = (work_items + per_thread - 1) / per_thread;
    uint64_t blocks = (threads + kThreads - 1) / kThreads;
    const uint64_t cap = static_cast<uint64_t>(launch_cfg().num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_global_scale(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                float *g_out, cudaStream_t st) {
    // three programmatic dependents in a row (no memset, which would break
    // the launch chain): zero the cell, fold the amax into it, turn it into g
    uint32_t *cell = reinterpret_cast<uint32_t *>(g_out);
    cudaError_t e = launch_cell_reset(cell, st);
    if (e != cudaSuccess) return e;
    const uint32_t vpr = static_cast<uint32_t>(cols / 8);
    const uint64_t total = static_cast<uint64_t>(rows) * vpr;
    if (total > 0) {
        cudaLaunchAttribute attr = pdl_attribute();
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.gridDim = dim3(grid_for(total, 4), 1, 1);
        cfg.stream = st;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, amax_kernel, X, static_cast<uint32_t>(rows), vpr,
                               static_cast<uint64_t>(ldx), FastDiv(vpr), cell);
        if (e != cudaSuccess) return e;
    }
    return launch_amax_cell_to_scale(cell, st);
}

cudaError_t launch_quantize(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                            const float *g, uint8_t *q, uint8_t *sf, int layout,
                            cudaStream_t st) {
    const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
    // the tile layout's padding rows (scale 0) are written by the kernel too
    const uint32_t rows_pad = static_cast<uint32_t>(
        layout == NVFP4_SF_MMA_128x4 ? (rows + 127) / 128 * 128 : rows);
    const uint64_t total_pad = static_cast<uint64_t>(rows_pad) * kbpr;
    if (total_pad == 0) return cudaSuccess;
    const int grid = grid_for(total_pad, 4);
    if (layout == NVFP4_SF_ROW_MAJOR)
        quantize_kernel<NVFP4_SF_ROW_MAJOR><<<grid, kThreads, 0, st>>>(
            X, static_cast<uint32_t>(rows), rows_pad, kbpr, static_cast<uint64_t>(ldx),
            FastDiv(kbpr), g, q, sf);
    else
        quantize_kernel<NVFP4_SF_MMA_128x4><<<grid, kThreads, 0, st>>>(
            X, static_cast<uint32_t>(rows), rows_pad, kbpr, static_cast<uint64_t>(ldx),
            FastDiv(kbpr), g, q, sf);
    return cudaGetLastError();
}

cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

cudaError_t launch_quantize_small(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                  float *g_out, uint8_t *q, uint8_t *sf, cudaStream_t st) {
    const uint32_t vpr = static_cast<uint32_t>(cols / 8);
    const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    int grid = grid_for(static_cast<uint64_t>(rows_pad) * kbpr, 4);
    if (grid > 32) grid = 32;  // each CTA reads all of X for the amax
    cudaLaunchAttribute attr = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_small_kernel, X, static_cast<uint32_t>(rows),
                              rows_pad, kbpr, static_cast<uint64_t>(ldx), FastDiv(kbpr), vpr,
                              FastDiv(vpr), g_out, q, sf);
}

cudaError_t launch_cell_reset(uint32_t *cell, cudaStream_t st) {
    cudaLaunchAttribute attr = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(1, 1, 1);
    cfg.gridDim = dim3(1, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, counter_reset_kernel, reinterpret_cast<unsigned int *>(cell));
}

cudaError_t launch_amax_cell_to_scale(uint32_t *cell, cudaStream_t st) {
    cudaLaunchAttribute attr = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(1, 1, 1);
    cfg.gridDim = dim3(1, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, amax_cell_to_scale_kernel, cell);
}

cudaError_t launch_quantize_cluster(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                    float *g_out, uint8_t *q, uint8_t *sf, cudaStream_t st) {
    const uint32_t vpr = static_cast<uint32_t>(cols / 8);
    const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kQuantizeClusterCtas;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kClusterThreads, 1, 1);
    cfg.gridDim = dim3(kQuantizeClusterCtas, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // per device: does a cluster of 16 fit (else the cooperative quantizer
    // is used instead)
    static DeviceOnce once;
    static bool fits_of[kMaxDevices + 1] = {};
    (void)once.run([&](int slot) {
        // 16 CTAs per cluster is beyond the portable 8
        cudaError_t e = cudaFuncSetAttribute(quantize_cluster_kernel,
                                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        cudaLaunchConfig_t occ = cfg;  // the cluster shape alone
        occ.attrs = &attr[1];
        occ.numAttrs = 1;
        int n = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, quantize_cluster_kernel, &occ);
        if (e != cudaSuccess) (void)cudaGetLastError();
        fits_of[slot] = e == cudaSuccess && n >= 1;
        return cudaSuccess;
    });
    if (!fits_of[device_slot()]) return cudaErrorNotSupported;
    return cudaLaunchKernelEx(&cfg, quantize_cluster_kernel, X, static_cast<uint32_t>(rows),
                              rows_pad, kbpr, static_cast<uint64_t>(ldx), FastDiv(kbpr), vpr,
                              FastDiv(vpr), g_out, q, sf);
}

cudaError_t launch_quantize_fused(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                  uint32_t *partials, unsigned int *counter, float *g_out,
                                  uint8_t *q, uint8_t *sf, cudaStream_t st) {
    static DeviceOnce once;
    static int per_sm_of[kMaxDevices + 1] = {};
    const cudaError_t e_setup = once.run([](int slot) {
        int n = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_fused_kernel, kThreads, 0);
        if (e == cudaSuccess) per_sm_of[slot] = n < 1 ? 1 : (n > 8 ? 8 : n);
        return e;
    });
    if (e_setup != cudaSuccess) return e_setup;
    const int per_sm = per_sm_of[device_slot()];
    const uint32_t vpr = static_cast<uint32_t>(cols / 8);
    const uint32_t kbpr = static_cast<uint32_t>(cols / 16);
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    int grid = launch_cfg().num_sms * per_sm;
    const int need = grid_for(static_cast<uint64_t>(rows_pad) * kbpr, 4);
    if (need < grid) grid = need;
    if (grid > kMaxAmaxPartials) grid = kMaxAmaxPartials;
    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorInvalidSymbol;
    cudaError_t e = launch_cell_reset(counter, st);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, quantize_fused_kernel, X, static_cast<uint32_t>(rows),
                              rows_pad, kbpr, static_cast<uint64_t>(ldx), FastDiv(kbpr), vpr,
                              FastDiv(vpr), partials, counter, g_out, q, sf,
                              debug_state().timeout_ns, err);
}

cudaError_t launch_sf_to_mma(const uint8_t *sf_rm, int64_t rows, int64_t K, uint8_t *sf_mma,
                             cudaStream_t st) {
    const uint32_t kb4 = static_cast<uint32_t>(K / 64);
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    const uint64_t total = static_cast<uint64_t>(rows_pad) * kb4;
    if (total == 0) return cudaSuccess;
    sf_to_mma_kernel<<<grid_for(total, 1), kThreads, 0, st>>>(
        sf_rm, static_cast<uint32_t>(rows), rows_pad, kb4, FastDiv(kb4), sf_mma);
    return cudaGetLastError();
}

}  // namespace nvfp4
