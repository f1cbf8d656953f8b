// The NVFP4 block quantizer's arithmetic, shared by the standalone
// quantizer and the GEMM that quantizes activations in its producer, so both
// produce the same bytes.
//
// Format ("nvfp4-gemma4" page, section 2; "nvfp4-difusion" page, section 2):
// E2M1 codes two per byte (even element in the low nibble), one E4M3 scale
// per 16 consecutive elements. Scale rule (absmax) with the decode-direction
// global scale g:
//   S = E4M3_rne_satfinite((amax_block / 6) / g)
//   r = 1 / (e4m3(S) * g)   (0 when S == 0)
//   code = E2M1_rne_satfinite(x * r), sign bit = sign bit of x.
// Every float step is one IEEE binary32 operation (explicit _rn intrinsics
// or .rn instructions, never contracted).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

// Byte offset of scale (row, kb) in the 128x4 tensor-core tile layout.
__device__ __forceinline__ uint64_t sf_mma_offset(uint32_t row, uint32_t kb, uint32_t kb4) {
    const uint32_t R = row >> 7, r = row & 127u;
    return ((static_cast<uint64_t>(R) * kb4 + (kb >> 2)) << 9) + ((r & 31u) << 4) +
           ((r >> 5) << 2) + (kb & 3u);
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest |x| of the 8 bfloat16 pairs as a bfloat16 magnitude bit pattern.
// Non-negative floats order like their bit patterns, so this is exact.
__device__ __forceinline__ uint32_t amax_bits16(uint4 a, uint4 b) {
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t t0 = max_u16x2(a.x & m, a.y & m);
    uint32_t t1 = max_u16x2(a.z & m, a.w & m);
    uint32_t t2 = max_u16x2(b.x & m, b.y & m);
    uint32_t t3 = max_u16x2(b.z & m, b.w & m);
    uint32_t t = max_u16x2(max_u16x2(t0, t1), max_u16x2(t2, t3));
    return max(t & 0xFFFFu, t >> 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two E2M1 codes (one byte, low element in the low nibble) of the bfloat16
// pair w scaled by r: both products in one packed IEEE binary32 multiply
// (mul.rn.f32x2: two round-to-nearest products, no flush), then one
// round-to-nearest-even saturating conversion.
__device__ __forceinline__ uint32_t codes2(uint32_t w, uint64_t rr) {
    uint32_t out;
    asm("{\n\t.reg .b32 l, h;\n\t.reg .b64 p, q;\n\t.reg .f32 x, y;\n\t.reg .b8 b;\n\t"
        "shl.b32 l, %1, 16;\n\t"
        "and.b32 h, %1, 0xFFFF0000;\n\t"
        "mov.b64 p, {l, h};\n\t"
        "mul.rn.f32x2 q, p, %2;\n\t"
        "mov.b64 {x, y}, q;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b, y, x;\n\t"
        "cvt.u32.u8 %0, b;\n\t}"
        : "=r"(out)
        : "r"(w), "l"(rr));
    return out;
}

// Four E2M1 codes of the two bfloat16 pairs w0 (elements 0,1) and w1
// (elements 2,3), packed little-end first.
__device__ __forceinline__ uint32_t codes4(uint32_t w0, uint32_t w1, uint64_t rr) {
    return codes2(w0, rr) | (codes2(w1, rr) << 8);
}

// The per-block multiplier r = 1 / (e4m3(S) * g), 0 when the product is 0
// (or not a number: byte 0x7F, which the saturating conversion never
// produces).
__device__ __forceinline__ float scale_recip(uint32_t S, float g) {
    const float denom = __fmul_rn(e4m3_to_f32(S), g);
    return denom > 0.0f ? __frcp_rn(denom) : 0.0f;
}

// scale_recip for all 128 scale bytes, by the threads of the block (the
// caller synchronizes before use).
__device__ __forceinline__ void fill_recip_table(float *rtab, float g) {
    for (uint32_t i = threadIdx.x; i < 128u; i += blockDim.x) rtab[i] = scale_recip(i, g);
}

// The block's scale byte S = E4M3_rne_satfinite((amax / 6) / g).
__device__ __forceinline__ uint32_t block_scale(uint4 a, uint4 b, float g) {
    const float amax = __uint_as_float(amax_bits16(a, b) << 16);
    return cvt_e4m3_satfinite(__fdiv_rn(__fdiv_rn(amax, 6.0f), g));
}

// The block's 16 codes under the multiplier r, into (lo, hi).
__device__ __forceinline__ void block_codes16(uint4 a, uint4 b, float r, uint32_t &lo,
                                              uint32_t &hi) {
    const uint64_t rr = (static_cast<uint64_t>(__float_as_uint(r)) << 32) | __float_as_uint(r);
    lo = codes4(a.x, a.y, rr) | (codes4(a.z, a.w, rr) << 16);
    hi = codes4(b.x, b.y, rr) | (codes4(b.z, b.w, rr) << 16);
}

// Quantize one 16-element block held in (a, b). Returns the scale byte and
// writes the 8 code bytes into (lo, hi).
__device__ __forceinline__ uint32_t quantize16(uint4 a, uint4 b, float g, uint32_t &lo,
                                               uint32_t &hi) {
    const uint32_t S = block_scale(a, b, g);
    block_codes16(a, b, scale_recip(S, g), lo, hi);
    return S;
}

// quantize16 with r read from a table that fill_recip_table filled for the
// same g (the table holds exactly what scale_recip computes).
__device__ __forceinline__ uint32_t quantize16_tab(uint4 a, uint4 b, float g,
                                                   const float *rtab, uint32_t &lo,
                                                   uint32_t &hi) {
    const uint32_t S = block_scale(a, b, g);
    block_codes16(a, b, NVFP4_CHECK(S < 128u) ? rtab[S] : 0.0f, lo, hi);
    return S;
}

}  // namespace nvfp4
