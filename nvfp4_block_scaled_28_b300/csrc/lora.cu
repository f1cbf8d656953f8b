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
// Work split: a CTA owns 16 rows; its 8 warps take 64-column chunks of K
// round robin. Per 16 x 16 piece a warp holds the bfloat16 values in the
// register layout of mma.sync m16n8k16 (lane = 4 g + c: rows g and g + 8,
// columns 2c, 2c + 1, 8 + 2c, 9 + 2c), so one load feeds both the quantizer
// (a 16-element block is one row of the piece, spread over a lane quad) and
// the tensor-core product with A. The warps' partial products are summed in
// warp order (deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// Scale byte and the two code words of one 16-element block held by a lane
// quad: this lane has elements (2c, 2c+1) in w_lo and (8+2c, 9+2c) in w_hi.
// Returns S; `lo` / `hi` get the block's code bytes 0..3 / 4..7 (every lane
// of the quad ends with the same words).
__device__ __forceinline__ uint32_t quantize_quad(uint32_t w_lo, uint32_t w_hi, int c, float g,
                                                  uint32_t &lo, uint32_t &hi) {
    uint32_t m = max_u16x2(w_lo & 0x7FFF7FFFu, w_hi & 0x7FFF7FFFu);
    m = max(m & 0xFFFFu, m >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    const float amax = __uint_as_float(m << 16);
    const float v = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
    const uint32_t S = cvt_e4m3_satfinite(v);
    const float s = e4m3_to_f32(S);
    const float denom = __fmul_rn(s, g);
    const float r = denom > 0.0f ? __frcp_rn(denom) : 0.0f;
    const uint64_t rr = (static_cast<uint64_t>(__float_as_uint(r)) << 32) | __float_as_uint(r);
    lo = codes2(w_lo, rr) << (8 * c);
    hi = codes2(w_hi, rr) << (8 * c);
    lo |= __shfl_xor_sync(0xFFFFFFFFu, lo, 1);
    hi |= __shfl_xor_sync(0xFFFFFFFFu, hi, 1);
    lo |= __shfl_xor_sync(0xFFFFFFFFu, lo, 2);
    hi |= __shfl_xor_sync(0xFFFFFFFFu, hi, 2);
    return S;
}

template <int R>
__global__ void __launch_bounds__(32 * kWarps)
    quantize_lora_kernel(const uint16_t *__restrict__ X, uint32_t rows, uint32_t K, uint64_t ldx,
                         const float *__restrict__ g_x, const float *__restrict__ g_w,
                         float lora_scale, const uint16_t *__restrict__ A, uint8_t *__restrict__ q,
                         uint8_t *__restrict__ sf, uint16_t *__restrict__ Lp) {
    __shared__ float red[kWarps][16][R];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, c = lane & 3;
    const uint32_t row0 = blockIdx.x * 16u;
    const uint32_t ra = row0 + gq, rb = ra + 8;
    const uint32_t kb4 = K / 64;
    pdl_launch_dependents();
    pdl_wait();
    if (row0 >= rows) {
        // padding rows of the 128-row scale tiles: scale 0
        for (uint32_t i = threadIdx.x; i < 16u * kb4; i += blockDim.x)
            *reinterpret_cast<uint32_t *>(sf + sf_mma_offset(row0 + i / kb4, (i % kb4) * 4, kb4)) =
                0u;
        return;
    }
    const bool va = ra < rows, vb = rb < rows;
    const float g = *g_x;
    const uint16_t *xa = X + static_cast<uint64_t>(va ? ra : 0) * ldx;
    const uint16_t *xb = X + static_cast<uint64_t>(vb ? rb : 0) * ldx;
    float acc[R / 8][4];
#pragma unroll
    for (int n = 0; n < R / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

    for (uint32_t ch = warp; ch < kb4; ch += kWarps) {
        uint32_t qa0 = 0, qa1 = 0, qb0 = 0, qb1 = 0, sa = 0, sb = 0;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t k0 = ch * 64u + ks * 16u + 2u * c;
            const uint32_t a0 = va ? ld_u32(xa + k0) : 0u, a2 = va ? ld_u32(xa + k0 + 8) : 0u;
            const uint32_t a1 = vb ? ld_u32(xb + k0) : 0u, a3 = vb ? ld_u32(xb + k0 + 8) : 0u;
            uint32_t lo, hi;
            sa |= quantize_quad(a0, a2, c, g, lo, hi) << (8 * ks);
            if (c == ks) {
                qa0 = lo;
                qa1 = hi;
            }
            sb |= quantize_quad(a1, a3, c, g, lo, hi) << (8 * ks);
            if (c == ks) {
                qb0 = lo;
                qb1 = hi;
            }
#pragma unroll
            for (int n = 0; n < R / 8; ++n) {
                const uint16_t *arow = A + static_cast<uint64_t>(n * 8 + gq) * K + k0;
                mma_bf16_16816(acc[n], a0, a1, a2, a3, ld_u32(arow), ld_u32(arow + 8));
            }
        }
        // lane c stores block c of the chunk for both rows; lanes 0 / 1 the
        // rows' four scale bytes (one aligned word of the tile layout)
        if (va)
            *reinterpret_cast<uint2 *>(q + static_cast<uint64_t>(ra) * (K / 2) + ch * 32u + c * 8u) =
                make_uint2(qa0, qa1);
        if (vb)
            *reinterpret_cast<uint2 *>(q + static_cast<uint64_t>(rb) * (K / 2) + ch * 32u + c * 8u) =
                make_uint2(qb0, qb1);
        if (c == 0)
            *reinterpret_cast<uint32_t *>(sf + sf_mma_offset(ra, ch * 4u, kb4)) = va ? sa : 0u;
        if (c == 1)
            *reinterpret_cast<uint32_t *>(sf + sf_mma_offset(rb, ch * 4u, kb4)) = vb ? sb : 0u;
    }
#pragma unroll
    for (int n = 0; n < R / 8; ++n) {
        red[warp][gq][n * 8 + 2 * c] = acc[n][0];
        red[warp][gq][n * 8 + 2 * c + 1] = acc[n][1];
        red[warp][gq + 8][n * 8 + 2 * c] = acc[n][2];
        red[warp][gq + 8][n * 8 + 2 * c + 1] = acc[n][3];
    }
    __syncthreads();
    const float factor = __fdiv_rn(lora_scale, __fmul_rn(g, *g_w));
    for (int i = threadIdx.x; i < 16 * R; i += blockDim.x) {
        const int rr = i / R, col = i % R;
        float sum = red[0][rr][col];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) sum = __fadd_rn(sum, red[w][rr][col]);
        if (row0 + rr < rows) {
            const __nv_bfloat16 v = __float2bfloat16_rn(__fmul_rn(sum, factor));
            Lp[static_cast<uint64_t>(row0 + rr) * R + col] = *reinterpret_cast<const uint16_t *>(&v);
        }
    }
}

template <int R>
cudaError_t launch_r(const uint16_t *X, int64_t rows, int64_t K, int64_t ldx, const float *g_x,
                     const float *g_w, float lora_scale, const uint16_t *A, uint8_t *q, uint8_t *sf,
                     uint16_t *Lp, cudaStream_t st) {
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    cudaLaunchAttribute attr = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(32 * kWarps, 1, 1);
    cfg.gridDim = dim3(rows_pad / 16, 1, 1);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_lora_kernel<R>, X, static_cast<uint32_t>(rows),
                              static_cast<uint32_t>(K), static_cast<uint64_t>(ldx), g_x, g_w,
                              lora_scale, A, q, sf, Lp);
}

}  // namespace

cudaError_t launch_quantize_lora(const uint16_t *X, int64_t rows, int64_t K, int64_t ldx,
                                 const float *g_x, const float *g_w, float lora_scale,
                                 const uint16_t *A, int64_t r, uint8_t *q, uint8_t *sf,
                                 uint16_t *Lp, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    switch (r) {
        case 16: return launch_r<16>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, Lp, st);
        case 32: return launch_r<32>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, Lp, st);
        case 48: return launch_r<48>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, Lp, st);
        case 64: return launch_r<64>(X, rows, K, ldx, g_x, g_w, lora_scale, A, q, sf, Lp, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nvfp4
