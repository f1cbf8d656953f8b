/*
 * NVFP4 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and the cpu_baseline leg of bench.py may
 * load, call or execute anything under oracle/. The product library never
 * links, imports or falls back to this file, and this file shares no code,
 * header, table or constant generator with the CUDA path.
 *
 * What it computes, and where the definitions come from:
 *
 *  - "nvfp4-gemma4" page, section 2 ("Que es realmente NVFP4"): an NVFP4 value
 *    is an E2M1 element (1 sign, 2 exponent, 1 mantissa bit); elements are
 *    grouped 16 at a time along the reduction axis, and each group shares one
 *    FP8 E4M3 scale (4 exponent, 3 mantissa bits).  The same section's table
 *    names the absmax rule: the largest magnitude of the block defines the
 *    scale.
 *  - "nvfp4-difusion" page, section 2 ("NVFP4 sin vLLM"): weights are stored
 *    (out, in/2) as uint8 with two FP4 values per byte, scales (out, in/16) as
 *    float8_e4m3fn; activations are quantized dynamically in forward(), then
 *    a block-scaled FP4 x FP4 matmul writes bfloat16.
 *  - The same section's table names two more block-scale rules: "MSE" tries
 *    several scales and keeps the one with the smallest block reconstruction
 *    error; "four-over-six" lets each block map its maximum to 4 or to 6,
 *    whichever errs less (quantize_block_rule states the candidates and the
 *    tie rule taken where the page gives none).
 *  - Where the pages are silent, these readings are taken: a per-tensor
 *    FP32 global scale g in the decode
 *    direction (x_hat = e2m1 * e4m3 * g) with g = amax_tensor / (6 * 448);
 *    block scale S = RNE_E4M3_satfinite((amax_block / 6) / g); codes by RNE
 *    onto the E2M1 grid with saturation at 6, ties to the even code; even-k
 *    element in the low nibble; sign bit = sign bit of x (so -0 and negative
 *    values that round to zero give code 0x8); an all-zero block gets S = 0.
 *
 * Every floating-point step of the quantizer is one IEEE-754 binary32
 * operation rounded to nearest even, in the order written (the file is built
 * with -ffp-contract=off and without -ffast-math, on x86-64 SSE arithmetic).
 * The roundings onto E2M1 and E4M3 are written as what they are: the nearest
 * representable value, found by comparing against every value of the format,
 * with ties going to the value whose code is even.
 *
 * The GEMM reference is the dense contraction of the dequantized operands,
 * summed in FP64 (every product of two dequantized values is exact in FP64),
 * multiplied by g_x * g_w in FP64 and rounded once to bfloat16.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- formats */

/* Value of a 4-bit E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1),
 * bit 0 mantissa; exponent 0 is subnormal (0 or 0.5). */
double oracle_e2m1_value(int code)
{
    int sign = (code >> 3) & 1;
    int exp = (code >> 1) & 3;
    int man = code & 1;
    double mag;
    if (exp == 0)
        mag = 0.5 * man;                      /* 0.M x 2^(1-bias) */
    else
        mag = (1.0 + 0.5 * man) * ldexp(1.0, exp - 1);
    return sign ? -mag : mag;
}

/* Value of an E4M3 (float8_e4m3fn) byte: bit 7 sign, bits 6..3 exponent
 * (bias 7), bits 2..0 mantissa; exponent 0 is subnormal; S.1111.111 is NaN
 * and there is no infinity. */
double oracle_e4m3_value(int byte)
{
    int sign = (byte >> 7) & 1;
    int exp = (byte >> 3) & 15;
    int man = byte & 7;
    double mag;
    if (exp == 15 && man == 7)
        return NAN;
    if (exp == 0)
        mag = (man / 8.0) * ldexp(1.0, -6);
    else
        mag = (1.0 + man / 8.0) * ldexp(1.0, exp - 7);
    return sign ? -mag : mag;
}

/* Nearest finite non-negative E4M3 value to v >= 0, ties to the even code;
 * values beyond the largest finite value (448) saturate to it. Returns the
 * byte (sign bit clear). */
uint8_t oracle_e4m3_rne_satfinite(float v)
{
    if (!(v <= 448.0f))            /* above the top value, or +inf */
        return 0x7E;
    int best = 0;
    double best_err = INFINITY;
    for (int b = 0; b <= 0x7E; ++b) {
        double err = fabs((double)v - oracle_e4m3_value(b));
        if (err < best_err || (err == best_err && (b & 1) == 0)) {
            best = b;
            best_err = err;
        }
    }
    return (uint8_t)best;
}

/* Nearest E2M1 magnitude code (0..7) to y >= 0, ties to the even code;
 * y above 6 (including +inf) saturates to code 7 (value 6). */
int oracle_e2m1_rne_satfinite(float y)
{
    if (!(y <= 6.0f))
        return 7;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 7; ++c) {
        double err = fabs((double)y - oracle_e2m1_value(c));
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return best;
}

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double once to the nearest bfloat16 (8-bit significand, float32
 * exponent range), ties to even; overflow goes to infinity. */
uint16_t oracle_bf16_from_double(double y)
{
    if (isnan(y))
        return 0x7FC0;
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    double a = fabs(y);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    frexp(a, &e);                      /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;                     /* a = 1.f * 2^E */
    if (E < -126)
        E = -126;                      /* subnormal range keeps the quantum */
    int qexp = E - 7;                  /* 7 stored fraction bits */
    double n = nearbyint(ldexp(a, -qexp)); /* default mode: nearest, ties even */
    double r = ldexp(n, qexp);
    if (r > 3.3895313892515355e38)     /* (2 - 2^-7) * 2^127 */
        return sign | 0x7F80;
    float f = (float)r;                /* exact: r is a bfloat16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* --------------------------------------------------------- global scale */

/* g = amax(|X|) / (6 * 448) as one fp32 division; g = 1 for an all-zero
 * tensor. X is bfloat16 bits, rows x cols with row stride ld (elements). */
float oracle_global_scale(const uint16_t *X, int64_t rows, int64_t cols, int64_t ld)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(bf16_to_float(X[r * ld + c]));
            if (a > amax)
                amax = a;
        }
    if (amax == 0.0f)
        return 1.0f;
    return amax / 2688.0f;
}

/* ------------------------------------------------------------ quantizer */

/* The E2M1 codes of the 16 values under block scale byte S: each |x| times
 * r = 1 / (e4m3(S) * g) (fp32), rounded onto the grid; sign bit from x. */
static void block_codes(const float *vals, float g, uint8_t S, int *codes)
{
    float s = (float)oracle_e4m3_value(S);        /* exact */
    float denom = s * g;
    float r = (denom > 0.0f) ? 1.0f / denom : 0.0f;
    for (int i = 0; i < 16; ++i) {
        float y = fabsf(vals[i]) * r;
        int m = oracle_e2m1_rne_satfinite(y);
        codes[i] = (signbit(vals[i]) ? 8 : 0) | m;
    }
}

/* Block reconstruction error of the codes under S: the sum over the 16
 * values, in element order, of (x - x_hat)^2 in FP64 (one rounding per
 * subtraction, product and addition), x_hat = e2m1(code) * e4m3(S) * g
 * (exact in FP64). */
static double block_error(const float *vals, float g, uint8_t S, const int *codes)
{
    double err = 0.0;
    for (int i = 0; i < 16; ++i) {
        double xhat = oracle_e2m1_value(codes[i]) * oracle_e4m3_value(S) * (double)g;
        double d = (double)vals[i] - xhat;
        double sq = d * d;
        err = err + sq;
    }
    return err;
}

/* Quantize one row segment of 16 values under a block-scale rule ("nvfp4-gemma4"
 * page, section 2, the scale-selection table):
 *   0 absmax: S6 = RNE_E4M3((amax / 6) / g), the block maximum maps to 6;
 *   1 four-over-six: S6, or S4 = RNE_E4M3((amax / 4) / g) (the maximum maps to
 *     4), whichever has the smaller block error; equal errors keep S6;
 *   2 MSE: the smallest block error over S6, S4 and every E4M3 scale from
 *     e4m3(S6) / 2 to 2 * e4m3(S6); equal errors keep S6, else the smallest
 *     scale (the pages give no candidate grid: this window is the reading).
 * Writes 8 packed bytes and returns the E4M3 scale byte. */
static uint8_t quantize_block_rule(const uint16_t *x, float g, int rule, uint8_t *packed)
{
    float vals[16];
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        vals[i] = bf16_to_float(x[i]);
        float a = fabsf(vals[i]);
        if (a > amax)
            amax = a;
    }
    float v = (amax / 6.0f) / g;                 /* two fp32 divisions */
    uint8_t S = oracle_e4m3_rne_satfinite(v);
    int codes[16];
    block_codes(vals, g, S, codes);
    if (rule != 0) {
        double best = block_error(vals, g, S, codes);
        uint8_t S6 = S;
        uint8_t S4 = oracle_e4m3_rne_satfinite((amax / 4.0f) / g);
        double lo = oracle_e4m3_value(S6) / 2.0, hi = oracle_e4m3_value(S6) * 2.0;
        for (int b = 1; b <= 0x7E; ++b) {
            if (b == S6)
                continue;
            int in = (b == S4) || (rule == 2 && oracle_e4m3_value(b) >= lo &&
                                   oracle_e4m3_value(b) <= hi);
            if (!in)
                continue;
            int c[16];
            block_codes(vals, g, (uint8_t)b, c);
            double e = block_error(vals, g, (uint8_t)b, c);
            if (e < best) {
                best = e;
                S = (uint8_t)b;
                memcpy(codes, c, sizeof c);
            }
        }
    }
    for (int j = 0; j < 8; ++j)
        packed[j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
    return S;
}

/* X: bf16 bits, rows x cols (cols % 16 == 0), row stride ld elements.
 * q: rows x cols/2 bytes (row-major, contiguous).
 * sf: rows x cols/16 E4M3 bytes (row-major, contiguous).
 * rule: 0 absmax, 1 four-over-six, 2 MSE (quantize_block_rule). */
void oracle_quantize_rule(const uint16_t *X, int64_t rows, int64_t cols, int64_t ld,
                          float g, int rule, uint8_t *q, uint8_t *sf)
{
    int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            sf[r * nb + b] = quantize_block_rule(X + r * ld + b * 16, g, rule,
                                                 q + r * (cols / 2) + b * 8);
}

/* The absmax rule (the one the activations use). */
void oracle_quantize(const uint16_t *X, int64_t rows, int64_t cols, int64_t ld,
                     float g, uint8_t *q, uint8_t *sf)
{
    oracle_quantize_rule(X, rows, cols, ld, g, 0, q, sf);
}

/* x_hat = e2m1(code) * e4m3(S) * g, in FP64; out is rows x cols. */
void oracle_dequantize(const uint8_t *q, const uint8_t *sf, float g,
                       int64_t rows, int64_t cols, double *out)
{
    int64_t nb = cols / 16;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < cols; ++k) {
            uint8_t byte = q[r * (cols / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[r * cols + k] = oracle_e2m1_value(code)
                              * oracle_e4m3_value(sf[r * nb + k / 16]) * (double)g;
        }
}

/* ----------------------------------------------------------------- GEMM */

/* Y[m, n] = bf16( (sum_k e2m1(Xq[m,k]) s_x[m,k/16] e2m1(Wq[n,k]) s_w[n,k/16])
 *                 * g_x * g_w + bias[n] ), the sum in FP64 in increasing k; bias
 * is an optional bfloat16 vector of N (NULL: no bias) added exactly in FP64
 * before the one rounding to bfloat16 (the linear layer's bias, applied where
 * the pages' forward() applies it: to the matmul output).
 * Row-major operands: Xq M x K/2, Xs M x K/16, Wq N x K/2, Ws N x K/16.
 * Only the n_rows rows listed in row_ids (or all M rows if row_ids is NULL,
 * then n_rows must be M) are computed; output row i of Y (and of Yd, if not
 * NULL) holds row row_ids[i]. */
void oracle_gemm_rows(const uint8_t *Xq, const uint8_t *Xs, float g_x,
                      const uint8_t *Wq, const uint8_t *Ws, float g_w,
                      int64_t M, int64_t N, int64_t K,
                      const int64_t *row_ids, int64_t n_rows,
                      const uint16_t *bias, uint16_t *Y, double *Yd)
{
    (void)M;
    int64_t kh = K / 2, nb = K / 16;
    /* Per-code and per-scale value tables, read from the decoders above. */
    double e2m1[16], e4m3[256];
    for (int c = 0; c < 16; ++c)
        e2m1[c] = oracle_e2m1_value(c);
    for (int b = 0; b < 256; ++b)
        e4m3[b] = oracle_e4m3_value(b);
    double alpha = (double)g_x * (double)g_w;
#pragma omp parallel
    {
        /* One dequantized X row at a time (per thread). */
        double *xrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            int64_t m = row_ids ? row_ids[i] : i;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = Xq[m * kh + k / 2];
                int code = (k & 1) ? (byte >> 4) : (byte & 15);
                xrow[k] = e2m1[code] * e4m3[Xs[m * nb + k / 16]];
            }
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                const uint8_t *wq = Wq + n * kh;
                const uint8_t *ws = Ws + n * nb;
                for (int64_t k = 0; k < K; ++k) {
                    uint8_t byte = wq[k / 2];
                    int code = (k & 1) ? (byte >> 4) : (byte & 15);
                    acc += xrow[k] * (e2m1[code] * e4m3[ws[k / 16]]);
                }
                double y = acc * alpha;
                if (bias)
                    y += (double)bf16_to_float(bias[n]);
                if (Yd)
                    Yd[i * N + n] = y;
                if (Y)
                    Y[i * N + n] = oracle_bf16_from_double(y);
            }
        }
        free(xrow);
    }
}

/* Low-rank (LoRA) correction kept beside the NVFP4 weight ("nvfp4-difusion"
 * page, section 3: a LoRA cannot be merged into NVFP4 codes, so its product
 * is computed at run time next to the quantized matmul):
 *   out[i, n] = scale * sum_j ( sum_k X[m,k] * A[j,k] ) * B[n,j],  m = row i
 * in FP64 on the unquantized bfloat16 activation, sums in increasing k and j.
 * X: bfloat16 bits M x K (row stride ldx); A: bfloat16 r x K (the down
 * projection); B: bfloat16 N x r (the up projection); out: n_rows x N.
 * Rows as oracle_gemm_rows. */
void oracle_lora_rows(const uint16_t *X, int64_t ldx, int64_t K, const uint16_t *A, int64_t r,
                      const uint16_t *B, int64_t N, double scale, const int64_t *row_ids,
                      int64_t n_rows, double *out)
{
#pragma omp parallel
    {
        double *l = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            int64_t m = row_ids ? row_ids[i] : i;
            for (int64_t j = 0; j < r; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (double)bf16_to_float(X[m * ldx + k]) *
                           (double)bf16_to_float(A[j * K + k]);
                l[j] = acc;
            }
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < r; ++j)
                    acc += l[j] * (double)bf16_to_float(B[n * r + j]);
                out[i * N + n] = scale * acc;
            }
        }
        free(l);
    }
}

/* Round FP64 values once to bfloat16 (n values). */
void oracle_round_bf16(const double *y, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_double(y[i]);
}

void oracle_gemm(const uint8_t *Xq, const uint8_t *Xs, float g_x,
                 const uint8_t *Wq, const uint8_t *Ws, float g_w,
                 int64_t M, int64_t N, int64_t K, uint16_t *Y, double *Yd)
{
    oracle_gemm_rows(Xq, Xs, g_x, Wq, Ws, g_w, M, N, K, NULL, M, NULL, Y, Yd);
}

/* ------------------------------------------- generic symmetric integer map */

/* The symmetric integer quantizer of the "cuantizacion e inferencia local"
 * page: s = max|x| / (2^(b-1) - 1), q = clamp(round(x / s)), x_hat = s q,
 * in FP64, round half to even. Returns s. Used only to pin the oracle's
 * conventions against the page's worked INT8 example. */
double oracle_symmetric_quantize(const double *x, int64_t n, int bits,
                                 int32_t *q, double *x_hat)
{
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i)
        if (fabs(x[i]) > amax)
            amax = fabs(x[i]);
    double qmax = (double)((1 << (bits - 1)) - 1);
    double s = amax / qmax;
    for (int64_t i = 0; i < n; ++i) {
        double t = (s > 0.0) ? nearbyint(x[i] / s) : 0.0;
        if (t > qmax)
            t = qmax;
        if (t < -qmax)
            t = -qmax;
        q[i] = (int32_t)t;
        x_hat[i] = s * t;
    }
    return s;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
