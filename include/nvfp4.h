/*
 * nvfp4.h -- C ABI of the B300 (sm_103a) NVFP4 linear-layer library.
 *
 * The operation (pages "nvfp4-gemma4", section 2, and "nvfp4-difusion",
 * section 2): an NVFP4 tensor stores each element as a 4-bit E2M1 code
 * (1 sign, 2 exponent, 1 mantissa bit), two codes per byte, and one FP8 E4M3
 * scale for every 16 consecutive elements along the reduction axis K.
 * Weights are stored (N, K/2) uint8 with scales (N, K/16) E4M3; activations
 * are quantized at run time; the linear layer is a block-scaled FP4 x FP4
 * matrix product Y = X W^T written out in bfloat16.
 *
 * Readings this library takes where the pages are silent:
 *  - a per-tensor FP32 global scale g in the decode direction,
 *    x_hat = e2m1(code) * e4m3(S) * g, with g = amax(|T|) / (6 * 448)
 *    (g = 1 for an all-zero tensor);
 *  - block scale S = RNE_E4M3_satfinite((amax_block / 6) / g), codes =
 *    RNE_E2M1_satfinite(x * (1 / (e4m3(S) * g))) with ties to the even code,
 *    each step one IEEE binary32 operation; 1/(e4m3(S) * g) is taken as 0
 *    when S = 0;
 *  - the even-k element sits in the low nibble of its byte, and a code's
 *    sign bit is the sign bit of x (a negative value that rounds to zero is
 *    code 0x8).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers of the current CUDA device. The
 *    caller allocates and owns every buffer; the library never allocates,
 *    frees or synchronizes, except nvfp4_device_error(), which synchronizes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Work is enqueued asynchronously on it.
 *  - bfloat16 tensors are passed as void* (2 bytes per element), row-major
 *    with the given leading dimension (elements between consecutive rows).
 *  - Packed codes are row-major (rows, K/2) bytes, contiguous.
 *  - Host threads may call entry points concurrently: the one-time set-up
 *    of each kernel on a device is serialized inside the library. Calls whose
 *    work overlaps on the GPU must not share a workspace or an output.
 *  - Errors are returned as nvfp4_status; nothing aborts the process. Checks
 *    on arguments happen before anything is enqueued: on an error return,
 *    no work was launched. A launch failure returns NVFP4_ERR_CUDA.
 *    A kernel whose internal bounded wait runs out records
 *    NVFP4_ERR_TIMEOUT in a device-side word that nvfp4_device_error()
 *    reports.
 */
#ifndef NVFP4_B300_H
#define NVFP4_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, size < 0, bad enum value */
    NVFP4_ERR_MISALIGNED = 2,        /* a pointer or leading dimension breaks its alignment rule */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 3, /* K (or cols) is not a multiple the entry point needs */
    NVFP4_ERR_WORKSPACE_TOO_SMALL = 4,
    NVFP4_ERR_CUDA = 5,              /* a CUDA runtime or driver call failed */
    NVFP4_ERR_TIMEOUT = 6,           /* a bounded wait inside a kernel ran out */
    NVFP4_ERR_BOUNDS = 7             /* debug build only: a kernel's bounds check failed */
} nvfp4_status;

/* Layout of an E4M3 scale tensor of `rows` rows and K/16 scales per row. */
typedef enum nvfp4_sf_layout {
    /* (rows, K/16) row-major bytes: the layout the "nvfp4-difusion" page
     * declares for weight_scale (section 2). */
    NVFP4_SF_ROW_MAJOR = 0,
    /* Tensor-core tile layout read directly by the GEMM: rows padded up to a
     * multiple of 128, K/16 a multiple of 4. Scale (r, j) lives in the
     * 512-byte tile t = (r / 128) * (K / 64) + j / 4, at byte
     * (r % 32) * 16 + ((r % 128) / 32) * 4 + j % 4 of that tile. Padding
     * rows hold 0. Same values as ROW_MAJOR, permuted. */
    NVFP4_SF_MMA_128x4 = 1
} nvfp4_sf_layout;

/* Human-readable name of a status code (static string, never NULL). */
NVFP4_API const char *nvfp4_status_string(int status);

/* Bytes a scale tensor of `rows` x (K/16) needs in `layout`; 0 if K is not
 * a multiple of 16 (ROW_MAJOR) or 64 (MMA_128x4), or on a bad argument. */
NVFP4_API size_t nvfp4_sf_bytes(int64_t rows, int64_t K, int layout);

/*
 * Per-tensor global scale (decode direction) of a bfloat16 tensor:
 *   *g = amax(|X|) / 2688.0f, or 1.0f if every element is +-0.
 * X: rows x cols bfloat16, leading dimension ldx (>= cols) elements,
 * 16-byte aligned, cols % 8 == 0 and ldx % 8 == 0.
 * g: one float in device memory (4-byte aligned); it is also used as the
 * reduction cell while the call runs, so it must not alias X.
 * rows == 0 or cols == 0 writes 1.0f.
 * Errors: INVALID_ARG (null, negative sizes), MISALIGNED, UNSUPPORTED_SHAPE
 * (cols % 8 != 0), CUDA.
 */
NVFP4_API nvfp4_status nvfp4_global_scale(const void *X, int64_t rows, int64_t cols,
                                int64_t ldx, float *g, void *stream);

/*
 * Dynamic NVFP4 quantization of a bfloat16 tensor ("nvfp4-difusion" page,
 * section 2: the activation is quantized to FP4 at run time), with the
 * global scale read from device memory.
 * X: rows x cols bfloat16 (ldx >= cols, ldx % 8 == 0, 16-byte aligned),
 * cols % 16 == 0 (cols % 64 == 0 for NVFP4_SF_MMA_128x4).
 * g: device pointer to the decode-direction global scale (finite, > 0).
 * q: rows x cols/2 bytes, contiguous, 8-byte aligned.
 * sf: nvfp4_sf_bytes(rows, cols, sf_layout) bytes.
 * Inputs must be finite. Errors: INVALID_ARG, MISALIGNED,
 * UNSUPPORTED_SHAPE, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_quantize(const void *X, int64_t rows, int64_t cols,
                            int64_t ldx, const float *g, uint8_t *q,
                            uint8_t *sf, int sf_layout, void *stream);

/* Block-scale rules of the "nvfp4-gemma4" page's scale-selection table
 * (section 2). */
typedef enum nvfp4_scale_rule {
    /* The block maximum maps to 6: S6 = E4M3_rne((amax / 6) / g). */
    NVFP4_SCALE_ABSMAX = 0,
    /* Each block keeps S6 or S4 = E4M3_rne((amax / 4) / g) (its maximum
     * mapped to 4), whichever gives the smaller block error. */
    NVFP4_SCALE_FOUR_OVER_SIX = 1,
    /* The smallest block error over S6, S4 and every E4M3 scale from
     * e4m3(S6) / 2 to 2 * e4m3(S6) (the page gives no candidate grid; this
     * window is this library's reading). */
    NVFP4_SCALE_MSE = 2
} nvfp4_scale_rule;

/*
 * nvfp4_quantize with a block-scale rule (nvfp4_scale_rule). The block error
 * of a candidate scale S is the sum over the block's 16 values, in element
 * order, of (x - e2m1(code) * e4m3(S) * g)^2 in binary64; codes under S are
 * those the absmax quantizer would write with scale S. Equal errors keep
 * S6, else the smallest scale. NVFP4_SCALE_ABSMAX is nvfp4_quantize itself.
 * Meant for offline weight quantization (nvfp4_global_scale(W) into g
 * first): the search runs in binary64, a few milliseconds for a 5120 x 5120
 * weight with NVFP4_SCALE_MSE.
 * Arguments, layout and errors as nvfp4_quantize; an unknown rule is
 * INVALID_ARG.
 */
NVFP4_API nvfp4_status nvfp4_quantize_select(const void *X, int64_t rows, int64_t cols,
                                            int64_t ldx, const float *g, int rule, uint8_t *q,
                                            uint8_t *sf, int sf_layout, void *stream);

/*
 * Offline weight quantization ("nvfp4-difusion" page, section 2: qweight
 * (out, in/2) uint8 and weight_scale (out, in/16) float8_e4m3fn):
 * nvfp4_global_scale(W) into *g_w, then nvfp4_quantize(W, g_w).
 * W: N x K bfloat16 with leading dimension ldw; Wq: N x K/2 bytes;
 * Ws: nvfp4_sf_bytes(N, K, sf_layout) bytes; g_w: one device float.
 * Same requirements and errors as the two calls it makes.
 */
NVFP4_API nvfp4_status nvfp4_quantize_weight(const void *W, int64_t N, int64_t K,
                                   int64_t ldw, uint8_t *Wq, uint8_t *Ws,
                                   float *g_w, int sf_layout, void *stream);

/*
 * Permute a row-major scale tensor (rows x K/16) into NVFP4_SF_MMA_128x4
 * (padding rows set to 0). K % 64 == 0. sf_mma must not alias sf_row_major.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_sf_to_mma_layout(const uint8_t *sf_row_major, int64_t rows,
                                    int64_t K, uint8_t *sf_mma, void *stream);

/*
 * Block-scaled FP4 GEMM ("nvfp4-difusion" page, section 2: the _scaled_mm
 * call on two float4_e2m1fn_x2 operands with their block scales, bfloat16
 * out), as a tcgen05 kind::mxf4nvf4 tensor-core kernel:
 *   Y[m, n] = bf16( g_a * g_b * sum_k e2m1(Aq[m,k]) e4m3(As[m,k/16])
 *                                    e2m1(Bq[n,k]) e4m3(Bs[n,k/16]) )
 * with FP32 accumulation.
 * Aq: M x K/2, Bq: N x K/2 packed codes, 16-byte aligned.
 * As, Bs: scales in NVFP4_SF_MMA_128x4 layout, 16-byte aligned.
 * g_a, g_b: device pointers to the two global scales.
 * Y: M x N bfloat16, leading dimension ldy >= N (rows that start 16-byte
 * aligned, i.e. 16-byte aligned Y and ldy % 8 == 0, get 16-byte stores).
 * K % 256 == 0; M, N >= 0 (0 is a no-op).
 * M <= 128 (decode) runs a weight-streaming kernel that computes Y^T = W X^T
 * with the weights as the 128-row MMA operand; larger M runs the CTA-pair
 * kernel on 256 x 256 tiles (its partial last wave as 256 x 128 column
 * halves; the same bits either way), or, once
 * nvfp4_debug_select_gemm_kernel(1) was called, the single-CTA kernel on
 * 128 x 256 tiles.
 * workspace / workspace_bytes: scratch; query nvfp4_gemm_workspace_bytes()
 * (0 for every shape in this version). May be NULL when that returns 0.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_gemm(const uint8_t *Aq, const uint8_t *As, const float *g_a,
                        const uint8_t *Bq, const uint8_t *Bs, const float *g_b,
                        int64_t M, int64_t N, int64_t K, void *Y, int64_t ldy,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Scratch bytes nvfp4_gemm needs for this shape (0 for most shapes). */
NVFP4_API size_t nvfp4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* How nvfp4_linear produces the activation's FP4 operand. */
typedef enum nvfp4_linear_mode {
    /* nvfp4_quantize into the workspace, then nvfp4_gemm. */
    NVFP4_LINEAR_UNFUSED = 0,
    /* For M <= 8 and K <= 6144 one kernel does it all: every CTA reads the
     * bfloat16 X, computes g_x when it is not given, and quantizes X once
     * into shared memory (same arithmetic, bit-identical output), so X's
     * codes never travel through HBM and no separate quantize launch is
     * needed. Beyond that (the resident operand holds 8 rows of up to 6144
     * K) this mode runs the unfused sequence. */
    NVFP4_LINEAR_FUSED = 1
} nvfp4_linear_mode;

/*
 * NVFP4 linear layer (the "nvfp4-difusion" page's BlackwellLinear.forward,
 * section 2): quantize the bfloat16 activation dynamically, then the
 * block-scaled FP4 GEMM against pre-quantized weights, bfloat16 out.
 *   Y = bf16( dequant(quantize(X, g_x)) * dequant(Wq, Ws, g_w)^T )
 * X: M x K bfloat16 (ldx >= K, ldx % 8 == 0, 16-byte aligned), K % 256 == 0.
 * Wq: N x K/2; Ws: NVFP4_SF_MMA_128x4 scales; g_w: device float.
 * Y: M x N bfloat16, ldy >= N, 2-byte aligned.
 * g_x: device pointer to the activation's global scale, or NULL to compute
 * it from X on the device first (one extra read of X).
 * mode: nvfp4_linear_mode.
 * workspace: nvfp4_linear_workspace_bytes(M, N, K, mode) bytes, 256-byte
 * aligned. After the call it holds X's quantized form, which a caller may
 * read (to reuse it, or to check it): the global scale used (fp32 at byte
 * 0; written when g_x is NULL), X's codes (M x K/2 bytes at byte 8448) and
 * their NVFP4_SF_MMA_128x4 scales (at byte 8448 + M*K/2 rounded up to a
 * multiple of 256). The fused mode for M <= 8 leaves nothing there (its
 * operand stays in shared memory).
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_linear(const void *X, int64_t M, int64_t K, int64_t ldx,
                          const uint8_t *Wq, const uint8_t *Ws,
                          const float *g_w, int64_t N, void *Y, int64_t ldy,
                          const float *g_x, int mode, void *workspace,
                          size_t workspace_bytes, void *stream);

NVFP4_API size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int mode);

/*
 * Grouped projection: several linear layers that read the same activation
 * (the attention's to_q / to_k / to_v, which the "nvfp4-difusion" page's
 * checkpoint stores as one fused qkv matrix sliced in thirds, section 2;
 * those projections are most of the DiT's compute, section 1) in one call:
 * X is quantized once and one GEMM launch computes every group, each with
 * its own weight global scale (or all equal, for slices of one matrix).
 *   Y[:, cols of group g] = bf16( dequant(quantize(X, g_x)) *
 *                                 dequant(Wq_g, Ws_g, g_w[g])^T )
 * Bitwise equal to `groups` separate nvfp4_linear calls on the groups.
 * Wq: the groups' codes stacked by rows (sum(group_n) x K/2); Ws: their
 * NVFP4_SF_MMA_128x4 scales stacked the same way (each group's tile-layout
 * scales are whole 128-row tiles, so stacking the byte arrays is the
 * layout of the stacked weight).
 * g_w: device array of `groups` floats, one per group.
 * group_n: host array of `groups` output-column counts, each > 0 and a
 * multiple of 256; 1 <= groups <= 8.
 * Y: M x sum(group_n) bfloat16 (ldy >= sum(group_n)); group g's output
 * starts at column sum(group_n[0..g-1]).
 * X, g_x, mode, workspace (nvfp4_linear_workspace_bytes(M, sum(group_n),
 * K, mode)): as nvfp4_linear.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_linear_grouped(const void *X, int64_t M, int64_t K, int64_t ldx,
                                           const uint8_t *Wq, const uint8_t *Ws,
                                           const float *g_w, const int64_t *group_n,
                                           int groups, void *Y, int64_t ldy, const float *g_x,
                                           int mode, void *workspace, size_t workspace_bytes,
                                           void *stream);

/*
 * nvfp4_linear for callers that cannot allocate device memory. The pages
 * have no counterpart: this is a deployment variant of nvfp4_linear.
 *
 * nvfp4_linear needs a caller-allocated workspace. Some callers have no way
 * to provide one: a plugin inside a host application that owns the device
 * memory pool and forbids outside allocations, a serving loop that reserves
 * all of its memory up front so no request can fail on an allocation, or a
 * C caller with no device allocator. This variant keeps the workspace in a
 * fixed 16 MiB array inside the library (held on every GPU that loads the
 * library until the process exits) and calls no cudaMalloc, cudaFree or
 * allocating library routine. The caller still passes X, the weights and Y.
 *
 * Same arguments, layout rules and result as nvfp4_linear with
 * mode = NVFP4_LINEAR_UNFUSED, minus the workspace. Limit:
 * nvfp4_linear_workspace_bytes(M, N, K, NVFP4_LINEAR_UNFUSED) must not
 * exceed 16 MiB (about M * K / 2 * 1.125 bytes; 4096 x 5120 fits), else
 * NVFP4_ERR_WORKSPACE_TOO_SMALL and nothing is launched.
 * The first call on each device looks the array's device address up
 * (cudaGetSymbolAddress) while that device is current and keeps it for the
 * life of the process; make that first call before any stream capture
 * begins. A cudaDeviceReset (or anything else that destroys the device's
 * primary context) invalidates the kept address: do not call this entry
 * point on that device again in the same process. Every call shares the one array and it
 * keeps the previous call's contents: calls whose work overlaps on the GPU
 * (different streams, or different host threads without ordering) race on
 * it, so serialize them.
 */
NVFP4_API nvfp4_status nvfp4_linear_noalloc(const void *X, int64_t M, int64_t K, int64_t ldx,
                                           const uint8_t *Wq, const uint8_t *Ws,
                                           const float *g_w, int64_t N, void *Y, int64_t ldy,
                                           const float *g_x, void *stream);

/*
 * nvfp4_linear with two epilogue steps fused into the GEMM (the pages' DiT
 * and LLM blocks chain these linears: "nvfp4-difusion" page, section 2,
 * BlackwellLinear.forward; the FFN's up projection feeds the down
 * projection, whose first step would quantize this output again):
 *   Y  = bf16( acc * g_x * g_w + bias[n] )     (bias added in fp32 before
 *                                              the single bfloat16 rounding)
 *   Yq, Ys = nvfp4_quantize(Y, g_y, NVFP4_SF_MMA_128x4)   (bit-identical)
 * so the next linear can take (Yq, Ys, g_y) as its activation operand
 * (nvfp4_gemm's A) without reading Y back from HBM.
 * X, Wq, Ws, g_w, g_x, workspace: as nvfp4_linear (mode UNFUSED; the
 * workspace size is nvfp4_linear_workspace_bytes(M, N, K, 0)).
 * bias: N bfloat16 values, 16-byte aligned, or NULL for none.
 * Y: M x N bfloat16 (ldy >= N), or NULL to skip the bfloat16 store.
 * g_y: device float, the decode-direction global scale of Y. It is an
 * input: the amax of Y is not known until every tile is done, so g_y comes
 * from calibration (or from a previous step), as a static activation scale.
 * Yq: M x N/2 bytes (row pitch N/2), 16-byte aligned.
 * Ys: nvfp4_sf_bytes(M, N, NVFP4_SF_MMA_128x4) bytes, 16-byte aligned; the
 * padding rows of the last 128-row group get scale 0.
 * g_y, Yq and Ys are all given or all NULL; Y and Yq are not both NULL.
 * Shapes: K % 256 == 0, N % 256 == 0 (one pair tile of columns, and the
 * next layer's K rule); any M >= 1: up to 64 rows the decode kernel
 * carries this epilogue (a 16-element block of Y spans 16 lanes there),
 * beyond it the CTA-pair kernel (above 128 rows: UNSUPPORTED_SHAPE while
 * the single-CTA kernel is selected for comparison).
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_linear_bias_requant(const void *X, int64_t M, int64_t K, int64_t ldx,
                                                const uint8_t *Wq, const uint8_t *Ws,
                                                const float *g_w, int64_t N, const void *bias,
                                                void *Y, int64_t ldy, const float *g_y,
                                                uint8_t *Yq, uint8_t *Ys, const float *g_x,
                                                void *workspace, size_t workspace_bytes,
                                                void *stream);

/*
 * nvfp4_linear_bias_requant with the output's global scale computed from
 * the output itself, as the next linear would compute it for its own
 * activation (the pages' dynamic activation quantization, "nvfp4-difusion"
 * page, section 2, carried across the chained linears):
 *   Y   = bf16( acc * g_x * g_w + bias[n] )
 *   g_y = amax(|Y|) / (6 * 448), or 1 for an all-zero Y     -> *g_y_out
 *   Yq, Ys = nvfp4_quantize(Y, g_y, NVFP4_SF_MMA_128x4)
 * All bytes equal nvfp4_linear_bias_requant (Y only, same bias) followed by
 * nvfp4_global_scale(Y) and nvfp4_quantize(Y, ...). The GEMM epilogue folds
 * each tile's largest |y| into *g_y_out (used as the amax cell) with atomic
 * maxima, so no pass over Y computes the amax; a small kernel turns it into
 * g_y and the quantizer then reads Y back (from L2 when Y fits there).
 * X, Wq, Ws, g_w, g_x, bias, workspace: as nvfp4_linear_bias_requant.
 * Y: required, M x N bfloat16 (ldy >= N, ldy % 8 == 0, 16-byte aligned).
 * g_y_out: device float (4-byte aligned) that receives g_y; its previous
 * value does not matter.
 * Yq, Ys: as nvfp4_linear_bias_requant.
 * Shapes: as nvfp4_linear_bias_requant. With M = 0 or N = 0 the call only
 * writes *g_y_out = 1 (the global scale of an empty tensor, as
 * nvfp4_global_scale gives it); Y, Yq, Ys and the workspace may then be
 * NULL.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_linear_bias_requant_dynamic(const void *X, int64_t M, int64_t K,
                                                        int64_t ldx, const uint8_t *Wq,
                                                        const uint8_t *Ws, const float *g_w,
                                                        int64_t N, const void *bias, void *Y,
                                                        int64_t ldy, float *g_y_out, uint8_t *Yq,
                                                        uint8_t *Ys, const float *g_x,
                                                        void *workspace, size_t workspace_bytes,
                                                        void *stream);

/*
 * NVFP4 linear layer with a run-time low-rank (LoRA) correction, the LoRA
 * kept beside the quantized weight ("nvfp4-difusion" page, section 3: a LoRA
 * cannot be merged into NVFP4 codes; its computation is fused with the
 * activation quantization in one CUDA pass instead):
 *   Y = bf16( dequant(quantize(X, g_x)) * dequant(Wq, Ws, g_w)^T
 *             + lora_scale * (X A^T) B^T )
 * with the LoRA branch on the unquantized bfloat16 X. Launches: (g_x NULL:
 * the global scale of X), one pass over X writing its NVFP4 codes and
 * scales and the down projection L' = bf16(lora_scale / (g_x g_w) * X A^T)
 * (tensor-core warp MMAs on the same loads), then the CTA-pair GEMM, which
 * adds L' B^T into its FP32 accumulator with r / 16 bfloat16 tensor-core
 * K-steps per tile before the epilogue scales by g_x g_w.
 * lora_A: r x K bfloat16 (the down projection), lora_B: N x r bfloat16 (the
 * up projection), both contiguous and 16-byte aligned; r in {16, 32, 48,
 * 64}; lora_scale finite (alpha / r in the usual LoRA notation).
 * Rounding of L' to bfloat16 puts a relative error of about 2^-9 on the
 * correction term.
 * M > 128 (the CTA-pair kernel; fewer rows return UNSUPPORTED_SHAPE).
 * X, Wq, Ws, g_w, Y, g_x: as nvfp4_linear; workspace:
 * nvfp4_linear_lora_workspace_bytes(M, N, K, r) bytes, 256-byte aligned.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
NVFP4_API nvfp4_status nvfp4_linear_lora(const void *X, int64_t M, int64_t K, int64_t ldx,
                                        const uint8_t *Wq, const uint8_t *Ws, const float *g_w,
                                        int64_t N, const void *lora_A, const void *lora_B,
                                        int64_t r, float lora_scale, void *Y, int64_t ldy,
                                        const float *g_x, void *workspace,
                                        size_t workspace_bytes, void *stream);

NVFP4_API size_t nvfp4_linear_lora_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);

/*
 * Synchronize the current device, then return NVFP4_ERR_BOUNDS if a kernel
 * of the debug build (libnvfp4_b300_debug.so, compiled with
 * NVFP4_DEBUG_CHECKS: every index a kernel forms for a global or shared
 * access is checked against its buffer, and an access that fails is
 * recorded and skipped) found an index out of bounds, NVFP4_ERR_TIMEOUT if
 * a kernel recorded a bounded-wait timeout, in both cases since the last
 * clear, NVFP4_ERR_CUDA if the synchronization failed, else NVFP4_OK.
 * clear != 0 resets the device-side word.
 */
NVFP4_API nvfp4_status nvfp4_device_error(int clear);

/*
 * Testing hook for the bounded waits (no fault is involved): with
 * mode = 1 the next GEMM launches' TMA producer issues no loads, so the
 * consumers' waits run out after timeout_us microseconds and the kernel
 * records NVFP4_ERR_TIMEOUT and returns. mode = 0 restores normal
 * operation; timeout_us = 0 restores the default limit (2 s).
 */
NVFP4_API nvfp4_status nvfp4_debug_set_fault_injection(int mode, uint32_t timeout_us);

/*
 * Testing and comparison hook: the GEMM kernel used for M > 128 by
 * nvfp4_gemm, nvfp4_linear and nvfp4_linear_grouped from the next call on
 * (process-wide, all devices). kernel = 0: CTA pairs on 256 x 256 tiles
 * (default); kernel = 1: the single-CTA kernel (128 x 256 tiles, one SM per
 * tile). Both issue the same K = 64 MMAs in K order, so they give the same
 * bits. While kernel = 1, the entry points whose epilogues live in the
 * CTA-pair kernel (bias / re-quantization, LoRA, grouped projections above
 * 128 rows) return UNSUPPORTED_SHAPE. Errors: INVALID_ARG (kernel not 0 or
 * 1).
 */
NVFP4_API nvfp4_status nvfp4_debug_select_gemm_kernel(int kernel);

/*
 * Testing hook for the fused decode mode (NVFP4_LINEAR_FUSED with M <= 8,
 * K <= 6144), whose quantized activation otherwise never leaves shared
 * memory: with on = 1, CTA 0 of the fused kernel also writes the codes and
 * tile-layout scales it produced into the workspace, at the offsets where
 * the unfused path leaves them (see nvfp4_linear), so that they can be
 * compared byte for byte. Process-wide; on = 0 (default) turns it off.
 * Errors: INVALID_ARG (on not 0 or 1).
 */
NVFP4_API nvfp4_status nvfp4_debug_capture_fused_operand(int on);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_B300_H */
