/*
 * nvfp4_probe.h -- C ABI of the measurement library libnvfp4_probe.so.
 *
 * Not part of the NVFP4 linear-layer library (include/nvfp4.h): this
 * library exists only to measure the dense FP4 tensor-core rate that the
 * GEMM's roofline is compared against. It shares the inline-PTX helpers of
 * the kernels but none of their code paths.
 *
 * Status values are those of nvfp4_status (0 OK, 1 INVALID_ARG,
 * 2 MISALIGNED, 5 CUDA, 6 TIMEOUT).
 */
#ifndef NVFP4_B300_PROBE_H
#define NVFP4_B300_PROBE_H

#if defined(__GNUC__)
#define NVFP4_PROBE_API __attribute__((visibility("default")))
#else
#define NVFP4_PROBE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Dense FP4 tensor-core peak probe: `ctas` CTAs each issue `iters`
 * back-to-back tcgen05.mma kind::mxf4nvf4 instructions on
 * shared-memory-resident operands, from a loop specialised per variant (so
 * the issuing warp's own work does not set the rate):
 *   0  128 x 256 x 64 into one TMEM accumulator
 *   1  128 x 128 x 64
 *   2  128 x 128 x 64 from two warps, one accumulator each (iters / 2 each)
 *   3  variant 0 with the GEMM's three shared->TMEM scale copies
 *      (tcgen05.cp 32x128b.warpx4) in front of every MMA, same thread
 *   4  variant 0 with those copies issued by a second warp concurrently
 *   5  variant 0 with a GEMM stage's bookkeeping after every 4 MMAs:
 *      tcgen05.commit, an mbarrier poll (lane 0 + shuffle), a fence
 *   6  kind::f16 BF16 128 x 256 x 16 (calibration against the BF16 rate)
 *   7  CTA pairs (clusters of 2, tcgen05 cta_group::2): rank 0 issues
 *      256 x 256 x 64 MMAs computed half on each SM (ctas rounded down
 *      to even, at least 2)
 * iters must be a multiple of 4 (of 8 for variant 2).
 * FLOPs = ctas * iters * 2 * 128 * N * K (N = 128 for variants 1 and 2,
 * else 256; K = 16 for variant 6, else 64; for variant 7 per CTA of the
 * even count); time it with events on `stream` (a cudaStream_t as void*).
 * CTA 0 writes its SM clock cycles to *cycles (device pointer, 8-byte
 * aligned). Every wait inside is bounded (2 s); nvfp4_probe_error reports
 * one that ran out.
 * Returns 0, or 1 (invalid argument), 2 (misaligned), 5 (launch failed).
 */
NVFP4_PROBE_API int nvfp4_mma_peak_probe(int ctas, int iters, int variant,
                                         unsigned long long *cycles, void *stream);

/*
 * Synchronize the current device; 6 if a probe kernel recorded a
 * bounded-wait timeout since the last clear, 5 if synchronization failed,
 * else 0. clear != 0 resets the probe's device-side word.
 */
NVFP4_PROBE_API int nvfp4_probe_error(int clear);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_B300_PROBE_H */
