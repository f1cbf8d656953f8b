// NVFP4 quantization with a searched block scale: the four-over-six and MSE
// rules of the scale-selection table on the "nvfp4-gemma4" page, section 2
// (absmax is the rule of quantize.cu).
//
//   four-over-six: each block maps its maximum to 6 (S6, the absmax scale)
//                  or to 4 (S4 = E4M3_rne((amax / 4) / g)), whichever gives
//                  the smaller block reconstruction error;
//   MSE:           the smallest block error over S6, S4 and every E4M3
//                  scale from e4m3(S6) / 2 to 2 * e4m3(S6).
// The page gives neither a candidate grid nor a tie rule; the ones used
// here: equal errors keep S6, else the smallest scale (candidates are tried
// in ascending order and only a strictly smaller error replaces the best).
// The block error is the sum over the 16 values, in element order, of
// (x - x_hat)^2 in binary64 with one rounding per subtraction, product and
// addition; x_hat = e2m1(code) * e4m3(S) * g is exact in binary64. Codes
// under a candidate scale are computed exactly as the absmax quantizer does
// (r = 1 / (e4m3(S) * g) in binary32, code = E2M1_rne_satfinite(x * r)), so
// the rule changes only which scale is kept.
//
// One thread per 16-element block; offline-weight work (binary64 is slow on
// this part, but a 5120 x 5120 weight takes milliseconds).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// E2M1 magnitude of a 3-bit code: 0, 0.5 for exponent 0; (1 + m/2) * 2^(e-1).
__device__ __forceinline__ float e2m1_mag(uint32_t m) {
    const uint32_t e = m >> 1, man = m & 1u;
    return e == 0 ? 0.5f * static_cast<float>(man)
                  : __uint_as_float(((e - 1u + 127u) << 23) | (man << 22));
}

// Codes of the block (a: elements 0..7, b: 8..15, bfloat16 pairs; xd: the
// same 16 values in binary64) under the scale byte S, and their
// reconstruction error.
__device__ __forceinline__ double codes_and_error(uint4 a, uint4 b, const double (&xd)[16],
                                                  float g, uint32_t S, uint32_t &lo,
                                                  uint32_t &hi) {
    const float s = e4m3_to_f32(S);
    const float denom = __fmul_rn(s, g);
    const float r = denom > 0.0f ? __frcp_rn(denom) : 0.0f;
    const uint64_t rr = (static_cast<uint64_t>(__float_as_uint(r)) << 32) | __float_as_uint(r);
    lo = codes4(a.x, a.y, rr) | (codes4(a.z, a.w, rr) << 16);
    hi = codes4(b.x, b.y, rr) | (codes4(b.z, b.w, rr) << 16);
    const double sg = __dmul_rn(static_cast<double>(s), static_cast<double>(g));  // exact
    double err = 0.0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t code = ((i < 8 ? lo : hi) >> (4 * (i & 7))) & 15u;
        const double mag = __dmul_rn(static_cast<double>(e2m1_mag(code & 7u)), sg);  // exact
        const double xhat = (code & 8u) ? -mag : mag;
        const double d = __dsub_rn(xd[i], xhat);
        err = __dadd_rn(err, __dmul_rn(d, d));
    }
    return err;
}

template <int kRule>
__device__ uint32_t quantize16_select(uint4 a, uint4 b, float g, uint32_t &lo, uint32_t &hi) {
    const float amax = __uint_as_float(amax_bits16(a, b) << 16);
    const uint32_t S6 = cvt_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 6.0f), g));
    const uint32_t S4 = cvt_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 4.0f), g));
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    double xd[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        xd[i] = static_cast<double>((i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]));
    double best = codes_and_error(a, b, xd, g, S6, lo, hi);
    uint32_t S = S6;
    if (kRule == NVFP4_SCALE_FOUR_OVER_SIX) {
        if (S4 != S6) {
            uint32_t l4, h4;
            const double e = codes_and_error(a, b, xd, g, S4, l4, h4);
            if (e < best) {
                S = S4;
                lo = l4;
                hi = h4;
            }
        }
        return S;
    }
    // MSE: ascending E4M3 bytes (ascending values) in the window, plus S4.
    // Eight codes per binade above the subnormals, so the window and S4
    // (about 1.5 e4m3(S6)) lie within 16 codes of S6; iterating by offset
    // keeps the threads of a warp on the same candidates.
    const float v6 = e4m3_to_f32(S6);
    const float wlo = 0.5f * v6, whi = 2.0f * v6;  // exact
    for (int j = -16; j <= 16; ++j) {
        const int ci = static_cast<int>(S6) + j;
        if (j == 0 || ci < 1 || ci > 0x7E) continue;
        const uint32_t c = static_cast<uint32_t>(ci);
        const float v = e4m3_to_f32(c);
        if (c != S4 && (v < wlo || v > whi)) continue;
        uint32_t lc, hc;
        const double e = codes_and_error(a, b, xd, g, c, lc, hc);
        if (e < best) {
            best = e;
            S = c;
            lo = lc;
            hi = hc;
        }
    }
    return S;
}

template <int kRule, int kLayout>
__global__ void __launch_bounds__(kThreads)
    quantize_select_kernel(const uint16_t *__restrict__ X, uint32_t rows, uint32_t rows_pad,
                           uint32_t kbpr, uint64_t ldx, const float *__restrict__ g_ptr,
                           uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
    const float g = *g_ptr;
    const uint64_t total = static_cast<uint64_t>(kLayout == NVFP4_SF_ROW_MAJOR ? rows : rows_pad) *
                           kbpr;
    const uint32_t kb4 = kbpr >> 2;
    const uint64_t sf_end = static_cast<uint64_t>(kLayout == NVFP4_SF_ROW_MAJOR ? rows : rows_pad) *
                            kbpr;  // bytes of the scale buffer
    (void)sf_end;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint32_t row = static_cast<uint32_t>(i / kbpr);
        const uint32_t kb = static_cast<uint32_t>(i - static_cast<uint64_t>(row) * kbpr);
        if (row >= rows) {  // padding rows of the tile layout
            const uint64_t off = sf_mma_offset(row, kb, kb4);
            if (NVFP4_CHECK(off < sf_end)) sf[off] = 0;
            continue;
        }
        if (!NVFP4_CHECK(kb < kbpr)) continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(X + row * ldx + kb * 16u);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        uint32_t lo, hi;
        const uint32_t S = quantize16_select<kRule>(a, b, g, lo, hi);
        *reinterpret_cast<uint2 *>(q + static_cast<uint64_t>(row) * (kbpr * 8u) + kb * 8u) =
            make_uint2(lo, hi);
        const uint64_t off = kLayout == NVFP4_SF_ROW_MAJOR ? i : sf_mma_offset(row, kb, kb4);
        if (NVFP4_CHECK(off < sf_end)) sf[off] = static_cast<uint8_t>(S);
    }
}

template <int kRule, int kLayout>
cudaError_t launch_rule(const uint16_t *X, uint32_t rows, uint32_t rows_pad, uint32_t kbpr,
                        uint64_t ldx, const float *g, uint8_t *q, uint8_t *sf, cudaStream_t st) {
    const uint64_t total =
        static_cast<uint64_t>(kLayout == NVFP4_SF_ROW_MAJOR ? rows : rows_pad) * kbpr;
    uint64_t blocks = (total + kThreads - 1) / kThreads;
    const uint64_t cap = static_cast<uint64_t>(launch_cfg().num_sms) * 8;
    if (blocks > cap) blocks = cap;
    quantize_select_kernel<kRule, kLayout><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(
        X, rows, rows_pad, kbpr, ldx, g, q, sf);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_select(const uint16_t *X, int64_t rows, int64_t cols, int64_t ldx,
                                   const float *g, int rule, uint8_t *q, uint8_t *sf, int layout,
                                   cudaStream_t st) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const uint32_t r = static_cast<uint32_t>(rows), kbpr = static_cast<uint32_t>(cols / 16);
    const uint32_t rows_pad = static_cast<uint32_t>((rows + 127) / 128 * 128);
    const uint64_t ld = static_cast<uint64_t>(ldx);
    const bool mma = layout == NVFP4_SF_MMA_128x4;
    if (rule == NVFP4_SCALE_FOUR_OVER_SIX)
        return mma ? launch_rule<NVFP4_SCALE_FOUR_OVER_SIX, NVFP4_SF_MMA_128x4>(X, r, rows_pad, kbpr,
                                                                              ld, g, q, sf, st)
                   : launch_rule<NVFP4_SCALE_FOUR_OVER_SIX, NVFP4_SF_ROW_MAJOR>(X, r, rows_pad, kbpr,
                                                                              ld, g, q, sf, st);
    if (rule == NVFP4_SCALE_MSE)
        return mma ? launch_rule<NVFP4_SCALE_MSE, NVFP4_SF_MMA_128x4>(X, r, rows_pad, kbpr, ld, g,
                                                                    q, sf, st)
                   : launch_rule<NVFP4_SCALE_MSE, NVFP4_SF_ROW_MAJOR>(X, r, rows_pad, kbpr, ld, g,
                                                                    q, sf, st);
    return cudaErrorInvalidValue;
}

}  // namespace nvfp4
