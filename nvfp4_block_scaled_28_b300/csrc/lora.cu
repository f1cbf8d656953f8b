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
// Work split: a CTA owns 64 rows (16 per warp) and one K range; the K
// ranges' partial down projections go to FP32 workspace and a small kernel
// sums them in range order (deterministic) and applies the scale. X and A
// chunks of 64 columns stream into a 4-deep shared-memory ring (cp.async,
// 16-byte pieces, XOR-swizzled rows). From each chunk in shared memory the
// threads quantize one 16-element block each (the standalone quantizer's
// arithmetic) and the warps take their 16 x 16 pieces with ldmatrix for the
// tensor-core product with A (mma.sync m16n8k16), so X is read from HBM once
// for both.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int kWarps = 4;
constexpr int kRows = 16 * kWarps;  // rows per CTA
constexpr int kStages = 4;          // shared-memory ring depth (64-column chunks)
constexpr int kMaxSplit = 8;        // K ranges per row tile

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

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
    static constexpr int X_TILE = kRows * 128;  // 64 bfloat16 per row (8 KiB)
    static constexpr int A_TILE = R * 128;
    static constexpr int SMEM = kStages * (X_TILE + A_TILE);
};

// Grid: (row tiles of 128, K ranges). part: FP32 [range][rows_pad][R].
template <int R>
__global__ void __launch_bounds__(32 * kWarps)
    quantize_lora_kernel(const uint16_t *__restrict__ X, uint32_t rows, uint32_t K, uint64_t ldx,
                         const float *__restrict__ g_x, const uint16_t *__restrict__ A,
                         uint32_t chunks_per_range, uint32_t rows_pad, uint8_t *__restrict__ q,
                         uint8_t *__restrict__ sf, float *__restrict__ part) {
    using C = LoraCfg<R>;
    extern __shared__ __align__(128) uint8_t lsmem[];
    const uint32_t xs0 = smem_addr(lsmem);
    const uint32_t as0 = xs0 + kStages * C::X_TILE;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, c = lane & 3;
    const uint32_t row0 = blockIdx.x * kRows;
    const uint32_t kb4 = K / 64;
    const uint32_t c_begin = blockIdx.y * chunks_per_range;
    const uint32_t c_end = min(kb4, c_begin + chunks_per_range);
    const int nch = static_cast<int>(c_end - c_begin);
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

    float acc[R / 8][4];
#pragma unroll
    for (int n = 0; n < R / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
    const uint32_t ra = row0 + warp * 16 + gq;
    // ldmatrix lane roles: matrix m = lane / 8, row lane % 8
    const uint32_t lm = lane >> 3, lr = lane & 7;
    const uint32_t a_row = warp * 16 + (lm & 1u) * 8 + lr;  // X piece rows of this lane
    for (int i = 0; i < nch; ++i) {
        cp_async_wait<kStages - 2>();
        __syncthreads();  // chunk i landed; every warp is done with chunk i - 1
        if (i + kStages - 1 < nch) load((i + kStages - 1) % kStages, c_begin + i + kStages - 1);
        cp_async_commit();
        const int s = i % kStages;
        const uint32_t xs = xs0 + s * C::X_TILE, as = as0 + s * C::A_TILE;
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
        // down projection: this warp's 16 rows times the chunk of A
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(xs + swz(a_row, 2u * ks + (lm >> 1)), a0, a1, a2, a3);
#pragma unroll
            for (int pr = 0; pr < R / 16; ++pr) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(as + swz(pr * 16u + (lm >> 1) * 8u + lr, 2u * ks + (lm & 1u)), b0, b1,
                            b2, b3);
                mma_bf16_16816(acc[2 * pr], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(acc[2 * pr + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    cp_async_wait<0>();
    // this K range's partial down projection, rows ra and rb
    float *pa = part + (static_cast<uint64_t>(blockIdx.y) * rows_pad + ra) * R;
    float *pb = pa + 8 * R;
    if (NVFP4_CHECK(ra + 8 < rows_pad)) {  // rows ra and ra + 8 of this range's partials
#pragma unroll
        for (int n = 0; n < R / 8; ++n) {
            *reinterpret_cast<float2 *>(pa + n * 8 + 2 * c) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(pb + n * 8 + 2 * c) = make_float2(acc[n][2], acc[n][3]);
        }
    }
}

// L'[m, j] = bf16( lora_scale / (g_x g_w) * sum over K ranges, in order ).
template <int R>
__global__ void __launch_bounds__(256)
    lora_finalize_kernel(const float *__restrict__ part, uint32_t rows, uint32_t rows_pad,
                         uint32_t ranges, const float *__restrict__ g_x,
                         const float *__restrict__ g_w, float lora_scale,
                         uint16_t *__restrict__ Lp) {
    pdl_launch_dependents();
    pdl_wait();
    const float factor = __fdiv_rn(lora_scale, __fmul_rn(*g_x, *g_w));
    const uint64_t total = static_cast<uint64_t>(rows) * R;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        float sum = part[i];
        for (uint32_t sidx = 1; sidx < ranges; ++sidx)
            sum = __fadd_rn(sum, part[static_cast<uint64_t>(sidx) * rows_pad * R + i]);
        const __nv_bfloat16 v = __float2bfloat16_rn(__fmul_rn(sum, factor));
        Lp[i] = *reinterpret_cast<const uint16_t *>(&v);
    }
}

struct Split {
    uint32_t ranges, chunks_per_range;
};

// K ranges per 64-row tile: about four CTAs per SM in all, at most
// kMaxSplit, every range non-empty.
Split lora_split(int64_t rows_pad, int64_t K) {
    const uint32_t kb4 = static_cast<uint32_t>(K / 64);
    const uint32_t tiles = static_cast<uint32_t>(rows_pad / kRows);
    uint32_t want = (4u * static_cast<uint32_t>(launch_cfg().num_sms) + tiles - 1) / tiles;
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
                                       rows_pad, q, sf, part);
    if (e != cudaSuccess) return e;
    const uint64_t total = static_cast<uint64_t>(rows) * R;
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
