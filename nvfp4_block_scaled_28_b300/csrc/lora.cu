// One pass over the activation for a linear layer with a run-time low-rank
// (LoRA) correction: the NVFP4 quantization of X (absmax rule, given g_x)
// and the LoRA down projection L = X A^T, from the same loads.
//
// The "nvfp4-difusion" page, section 3: a LoRA cannot be merged into NVFP4
// codes, so it is computed at run time, fused with the activation
// quantization in one CUDA pass. Here the down projection is written
// pre-scaled for the GEMM that follows,
//   L' = bf16( (lora_scale / (g_x * g_w)) * X A^T )     (M x r),
// so that the GEMM can add L' B^T into the same FP32 accumulator as the
// FP4 products (extra bfloat16 tensor-core steps) before its epilogue
// multiplies everything by g_x * g_w.
//
// Work split: a CTA owns 128 rows and one K range; the K ranges' partial
// down projections go to FP32 workspace and a small kernel sums them in
// range order (deterministic) and applies the scale. X and A chunks of 64
// columns stream into a shared-memory ring (cp.async, 16-byte pieces, rows
// XOR-swizzled in the tensor core's 128-byte pattern). Each chunk feeds two
// consumers: one elected thread issues the chunk's four
// tcgen05.mma kind::f16 (M = 128 rows of X, N = r rows of A, K = 16 each)
// into an FP32 accumulator in tensor memory, and meanwhile every thread
// quantizes 16-element blocks of the chunk (the standalone quantizer's
// arithmetic), so X is read from HBM once for both and the product costs
// the quantizing warps nothing. A ring slot is refilled once the MMAs that
// read it have completed (tcgen05.commit on the slot's mbarrier).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int kWarps = 8;
constexpr int kRows = 128;          // rows per CTA: one M = 128 tensor-core tile
constexpr int kStages = 3;          // shared-memory ring depth (64-column chunks)
constexpr int kMaxSplit = 8;        // K ranges per row tile
constexpr int kCtasPerSm = 3;       // what the shared-memory budget allows

// 16-byte global -> shared copy; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte piece `p` of row `r` in a ring tile of 128-byte rows.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t p) {
    return r * 128u + ((p ^ (r & 7u)) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

template <int R>
struct LoraCfg {
    static constexpr int X_TILE = kRows * 128;  // 64 bfloat16 per row (16 KiB)
    static constexpr int A_TILE = R * 128;
    static constexpr int TMEM_COLS = R <= 32 ? 32 : 64;  // FP32 accumulator, 128 lanes x R
    static constexpr int BAR_OFF = kStages * (X_TILE + A_TILE);
    // + 1024 to align the ring to the swizzle pattern; barriers, TMEM slot
    static constexpr int SMEM = 1024 + BAR_OFF + 64;
    static_assert(A_TILE % 1024 == 0 && X_TILE % 1024 == 0, "tiles keep the 1024-byte pattern");
    static_assert(R % 16 == 0 && R >= 16 && R <= 64, "N of the M = 128 MMA");
};

// Grid: (row tiles of 128, K ranges). part: FP32 [range][rows_pad][R].
template <int R>
__global__ void __launch_bounds__(32 * kWarps)
    quantize_lora_kernel(const uint16_t *__restrict__ X, uint32_t rows, uint32_t K, uint64_t ldx,
                         const float *__restrict__ g_x, const uint16_t *__restrict__ A,
                         uint32_t chunks_per_range, uint32_t rows_pad, uint8_t *__restrict__ q,
                         uint8_t *__restrict__ sf, float *__restrict__ part, uint64_t timeout_ns,
                         unsigned int *err) {
    using C = LoraCfg<R>;
    extern __shared__ uint8_t lsmem_raw[];
    uint8_t *lsmem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(lsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t xs0 = smem_addr(lsmem);
    const uint32_t as0 = xs0 + kStages * C::X_TILE;
    uint64_t *mma_done = reinterpret_cast<uint64_t *>(lsmem + C::BAR_OFF);  // one per slot
    uint64_t *acc_full = mma_done + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t row0 = blockIdx.x * kRows;
    const uint32_t kb4 = K / 64;
    const uint32_t c_begin = blockIdx.y * chunks_per_range;
    const uint32_t c_end = min(kb4, c_begin + chunks_per_range);
    const int nch = static_cast<int>(c_end - c_begin);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&mma_done[s], 1);
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait();
    const float g = *g_x;
    __shared__ float rtab[128];
    fill_recip_table(rtab, g);  // ordered before its first use by the loop's barrier

    // one chunk of X (128 rows x 128 B) and of A (R rows x 128 B) into slot s
    auto load = [&](int s, uint32_t ch) {
#pragma unroll
        for (int i = 0; i < kRows * 8 / (32 * kWarps); ++i) {
            const uint32_t p = tid + i * 32 * kWarps;
            const uint32_t r = p >> 3, piece = p & 7u;
            const bool ok = row0 + r < rows;
            const uint16_t *src = X + (ok ? (row0 + r) * ldx : 0) + ch * 64u + piece * 8u;
            if (NVFP4_CHECK(swz(r, piece) + 16u <= C::X_TILE && ch * 64u + piece * 8u + 8u <= K))
                cp_async16(xs0 + s * C::X_TILE + swz(r, piece), src, ok ? 16u : 0u);
        }
        for (uint32_t p = tid; p < R * 8u; p += 32 * kWarps) {
            const uint32_t j = p >> 3, piece = p & 7u;
            if (NVFP4_CHECK(swz(j, piece) + 16u <= C::A_TILE && ch * 64u + piece * 8u + 8u <= K))
                cp_async16(as0 + s * C::A_TILE + swz(j, piece),
                           A + static_cast<uint64_t>(j) * K + ch * 64u + piece * 8u, 16u);
        }
    };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nch) load(s, c_begin + s);
        cp_async_commit();
    }

    constexpr uint32_t idesc = idesc_bf16(kRows, R);
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
        cp_async_wait<kStages - 2>();
        fence_proxy_async_shared();  // this thread's copies of chunk i, to the tensor core
        // the slot refilled below held chunk i - 1: its MMAs must have read it
        const bool refill = i + kStages - 1 < nch;
        int timed_out = 0;
        if (tid == 0 && refill && i >= 1)
            timed_out = !mbar_wait(&mma_done[(i - 1) % kStages], ((i - 1) / kStages) & 1,
                                   timeout_ns);
        // chunk i is complete in shared memory and every thread is done
        // with chunk i - 1
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) record_timeout(err);
            ok = false;
            break;
        }
        const int s = i % kStages;
        const uint32_t xs = xs0 + s * C::X_TILE, as = as0 + s * C::A_TILE;
        if (warp == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_elect(tmem, sdesc_sw128(xs + ks * 32), sdesc_sw128(as + ks * 32), idesc,
                               (i | ks) != 0);
            tc_commit_elect(&mma_done[s]);
        }
        if (refill) load((i + kStages - 1) % kStages, c_begin + i + kStages - 1);
        cp_async_commit();
        const uint32_t ch = c_begin + i;
        // quantization: one thread per 16-element block (4 per row of the
        // chunk), the standalone quantizer's arithmetic; the four lanes of a
        // row gather its scale bytes into one aligned word of the tile layout
#pragma unroll
        for (int u = 0; u < kRows * 4 / (32 * kWarps); ++u) {
            const uint32_t id = tid + u * 32 * kWarps;
            const uint32_t r = id >> 2, blk = id & 3u;
            const uint4 a = lds128(xs + swz(r, 2u * blk)), b = lds128(xs + swz(r, 2u * blk + 1u));
            uint32_t lo, hi;
            const uint32_t S = quantize16_tab(a, b, g, rtab, lo, hi);
            const uint32_t row = row0 + r;
            if (row < rows && NVFP4_CHECK(ch * 32u + blk * 8u + 8u <= K / 2))
                *reinterpret_cast<uint2 *>(q + static_cast<uint64_t>(row) * (K / 2) + ch * 32u +
                                           blk * 8u) = make_uint2(lo, hi);
            uint32_t w = S << (8u * blk);
            w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
            w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
            const uint64_t soff = sf_mma_offset(row, ch * 4u, kb4);
            if (blk == 0 && NVFP4_CHECK(soff + 4 <= static_cast<uint64_t>(rows_pad) * (K / 16)))
                *reinterpret_cast<uint32_t *>(sf + soff) = w;
        }
    }
    cp_async_wait<0>();
    // every MMA issued has completed (also after an abort: TMEM is released
    // only once nothing writes it)
    if (warp == 0) tc_commit_elect(acc_full);
    int done = 1;
    if (tid == 0) done = mbar_wait(acc_full, 0, timeout_ns);
    if (!__syncthreads_and(done)) {
        if (tid == 0) record_timeout(err);
        ok = false;
    }
    tc_fence_after();
    if (ok && warp < 4) {
        // this K range's partial down projection: warp w reads TMEM lanes
        // (rows) 32w .. 32w + 31, one row per thread (an empty range, which
        // the split never makes, would contribute zeros)
        const uint32_t row = row0 + warp * 32 + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float *dst = part + (static_cast<uint64_t>(blockIdx.y) * rows_pad + row) * R;
        constexpr int NCOL = R <= 32 ? 32 : 64;
        uint32_t v[NCOL];
        if (nch > 0) {
            if constexpr (NCOL == 32)
                tmem_ld_32x32b_x32(taddr, v);
            else
                tmem_ld_32x32b_x64(taddr, v);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int j = 0; j < NCOL; ++j) v[j] = 0u;
        }
        if (NVFP4_CHECK(row < rows_pad)) {
#pragma unroll
            for (int j = 0; j < R; j += 4)
                *reinterpret_cast<float4 *>(dst + j) =
                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// L'[m, j] = bf16( lora_scale / (g_x g_w) * sum over K ranges, in order ).
// Four consecutive entries per thread; all ranges' partials are loaded
// before the ordered sum, so their latencies overlap.
template <int R>
__global__ void __launch_bounds__(256)
    lora_finalize_kernel(const float *__restrict__ part, uint32_t rows, uint32_t rows_pad,
                         uint32_t ranges, const float *__restrict__ g_x,
                         const float *__restrict__ g_w, float lora_scale,
                         uint16_t *__restrict__ Lp) {
    pdl_launch_dependents();
    pdl_wait();
    const float factor = __fdiv_rn(lora_scale, __fmul_rn(*g_x, *g_w));
    const uint64_t total4 = static_cast<uint64_t>(rows) * R / 4;  // R % 16 == 0
    const uint64_t range4 = static_cast<uint64_t>(rows_pad) * R / 4;
    const float4 *p4 = reinterpret_cast<const float4 *>(part);
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total4;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        float4 v[kMaxSplit];
#pragma unroll
        for (int r = 0; r < kMaxSplit; ++r)
            if (r < static_cast<int>(ranges)) v[r] = p4[r * range4 + i];
        float4 sum = v[0];
#pragma unroll
        for (int r = 1; r < kMaxSplit; ++r) {
            if (r < static_cast<int>(ranges)) {
                sum.x = __fadd_rn(sum.x, v[r].x);
                sum.y = __fadd_rn(sum.y, v[r].y);
                sum.z = __fadd_rn(sum.z, v[r].z);
                sum.w = __fadd_rn(sum.w, v[r].w);
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(__fmul_rn(sum.x, factor),
                                                        __fmul_rn(sum.y, factor));
        const __nv_bfloat162 hi = __floats2bfloat162_rn(__fmul_rn(sum.z, factor),
                                                        __fmul_rn(sum.w, factor));
        reinterpret_cast<uint2 *>(Lp)[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                                                      *reinterpret_cast<const uint32_t *>(&hi));
    }
}

struct Split {
    uint32_t ranges, chunks_per_range;
};

// K ranges per 128-row tile: about kCtasPerSm CTAs per SM in all, at most
// kMaxSplit, every range non-empty.
Split lora_split(int64_t rows_pad, int64_t K) {
    const uint32_t kb4 = static_cast<uint32_t>(K / 64);
    const uint32_t tiles = static_cast<uint32_t>(rows_pad / kRows);
    uint32_t want =
        (kCtasPerSm * static_cast<uint32_t>(launch_cfg().num_sms) + tiles - 1) / tiles;
    want = want < 1 ? 1 : (want > kMaxSplit ? kMaxSplit : want);
    if (want > kb4) want = kb4;
    const uint32_t cpr = (kb4 + want - 1) / want;
    return {(kb4 + cpr - 1) / cpr, cpr};
}

template <int R>
cudaError_t launch_r(const uint16_t *X, int64_t rows, int64_t K, int64_t ldx, const float *g_x,
                     const float *g_w, float lora_scale, const uint16_t *A, uint8_t *q, uint8_t *sf,
                     float *part, uint16_t *Lp, cudaStream_t st) {
    using C = LoraCfg<R>;
    static DeviceOnce once;
    const cudaError_t e_setup = once.run([](int) {
        return cudaFuncSetAttribute(quantize_lora_kernel<R>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (e_setup != cudaSuccess) return e_setup;
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    const Split sp = lora_split(rows_pad, K);
    unsigned int *err = device_error_word();
    if (err == nullptr) return cudaErrorInvalidSymbol;
    cudaLaunchAttribute attr = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(32 * kWarps, 1, 1);
    cfg.gridDim = dim3(rows_pad / kRows, sp.ranges, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_lora_kernel<R>, X,
                                       static_cast<uint32_t>(rows), static_cast<uint32_t>(K),
                                       static_cast<uint64_t>(ldx), g_x, A, sp.chunks_per_range,
                                       rows_pad, q, sf, part, debug_state().timeout_ns, err);
    if (e != cudaSuccess) return e;
    const uint64_t total = static_cast<uint64_t>(rows) * R / 4;  // four entries a thread
    uint64_t blocks = (total + 255) / 256;
    const uint64_t cap = static_cast<uint64_t>(launch_cfg().num_sms) * 4;
    if (blocks > cap) blocks = cap;
    cfg.blockDim = dim3(256, 1, 1);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, lora_finalize_kernel<R>, part, static_cast<uint32_t>(rows),
                              rows_pad, sp.ranges, g_x, g_w, lora_scale, Lp);
}

}  // namespace

cudaError_t launch_quantize_lora(const uint16_t *X, int64_t rows, int64_t K, int64_t ldx,
                                 const float *g_x, const float *g_w, float lora_scale,
                                 const uint16_t *A, int64_t r, uint8_t *q, uint8_t *sf,
                                 float *part, uint16_t *Lp, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    switch (r) {
        case 16: return launch_r<16>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, part, Lp, st);
        case 32: return launch_r<32>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, part, Lp, st);
        case 48: return launch_r<48>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, part, Lp, st);
        case 64: return launch_r<64>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, part, Lp, st);
        default: return cudaErrorInvalidValue;
    }
}

size_t lora_partial_bytes(int64_t rows, int64_t r) {
    return static_cast<size_t>(kMaxSplit) * static_cast<size_t>((rows + 127) / 128 * 128) *
           static_cast<size_t>(r) * sizeof(float);
}

}  // namespace nvfp4
