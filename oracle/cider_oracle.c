/*
 * CPU oracle for the fused per-token INT8 quantize -> INT8 GEMM -> dequant
 * linear layer (W8A8 per-channel, W8A8 per-group, W4A8), in plain C.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it. It shares no code, header, table or
 * helper with the CUDA library; the two meet only at the seeded input
 * generators.
 *
 * What it computes, and where it comes from (pages on the Cider project):
 *  - Cider README (repo mirror), section "Quantization", table rows
 *    "Activations: Symmetric INT8, Per-token", "W8A8 weights: Symmetric INT8,
 *    Per-channel or per-group (gs=64/128)", "W4A8 weights: Symmetric INT4
 *    (zp=8)", "Accumulation: INT32" and "Output dequant:
 *    C_fp16 = C_int32 * s_act * s_weight".
 *  - Same README, section "W8A8 Quantization Granularity" (one scale per
 *    output channel, or one per 64/128 elements) and "Low-Level API"
 *    (quantize_weight_int8, pack_weight_int4 produce codes plus scales).
 *  - Same README, section "Metal Kernel Pipeline": prefill quantizes the
 *    fp16 activations to INT8 plus per-token scales, then INT8 x INT8 ->
 *    INT32 -> fp16 with the scales applied in the store phase; W4A8 unpacks
 *    INT4 to INT8 before the matrix product.
 *  - "min-max" scale (absmax), README section "LLM Quantization" note.
 *
 * Readings taken where the pages are silent:
 *  - scale = absmax / qmax in fp32 (qmax = 127 for INT8, 7 for INT4), one
 *    IEEE division, round to nearest even;
 *  - code = clamp(rint(x / scale), -qmax, qmax): IEEE fp32 division, then
 *    round half to even; -128 is never produced;
 *  - an all-zero row or group has scale 0 and all codes 0 (no division);
 *  - INT4 code q is stored as the nibble q + 8; byte j of a packed row holds
 *    element 2j in its low nibble and element 2j+1 in its high nibble;
 *  - per-channel output: y = fp16_rn(((float)acc * s_act) * s_w[n]);
 *  - per-group output: f = 0; for g ascending: f = f + (float)P_g * s_w[n,g]
 *    (a rounded product, then a rounded sum); y = fp16_rn(f * s_act);
 *  - fp16 rounding is round-to-nearest-even, overflow gives +-inf.
 *  - bf16 activations / outputs (the README roadmap's "automatic dtype
 *    handling (float16/bfloat16)"): a bf16 value is the binary32 value with
 *    the same upper 16 bits; quantization reads it exactly as fp32 and
 *    applies the same formulas; a bf16 output is the fp32 result rounded to
 *    nearest even at 8 significant bits, overflow gives +-inf.
 *
 * Build: plain C11, -O2 -ffp-contract=off -fno-fast-math (every float
 * operation is a single IEEE binary32 operation, as written). OpenMP only
 * spreads independent output rows over threads; it changes no arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, from the format definition.                   */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.        */
/* ------------------------------------------------------------------------ */

float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)frac, -24); /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(frac | 0x400), expo - 25); /* 1.frac * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

/* Round a binary32 value to the nearest binary16, ties to even. */
uint16_t oracle_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)f);
    /* 65504 is the largest finite binary16; the midpoint to the next step
       (65536, not representable) is 65520 and rounds to even, i.e. to inf. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);         /* a = m * 2^e2, m in [0.5, 1) */
    int unbiased = e2 - 1;       /* a in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -14)
        unbiased = -14;          /* subnormal binade shares the 2^-24 step */
    double quantum = ldexp(1.0, unbiased - 10);
    double n = rint(a / quantum); /* exact quotient; rint rounds ties to even */
    uint32_t out;
    if (unbiased == -14 && n < 1024.0) {
        out = (uint32_t)n;       /* subnormal (or exactly the smallest normal) */
    } else {
        int expo = unbiased + 15;
        if (n >= 2048.0) {       /* rounding carried into the next binade */
            n = 1024.0;
            expo += 1;
        }
        if (expo >= 31)
            return (uint16_t)(sign | 0x7C00u);
        out = ((uint32_t)expo << 10) | ((uint32_t)n - 1024u);
    }
    return (uint16_t)(sign | out);
}

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32, from the format definition.                        */
/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits: the    */
/* upper half of a binary32 encoding.                                        */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_float(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bfloat16, ties to even. */
uint16_t oracle_float_to_bf16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    if (isinf(f))
        return (uint16_t)(sign | 0x7F80u);
    int e2;
    (void)frexp(a, &e2);         /* a = m * 2^e2, m in [0.5, 1) */
    int unbiased = e2 - 1;       /* a in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -126)
        unbiased = -126;         /* subnormal binade shares the 2^-133 step */
    double quantum = ldexp(1.0, unbiased - 7);
    double n = rint(a / quantum); /* exact quotient; rint rounds ties to even */
    uint32_t out;
    if (unbiased == -126 && n < 128.0) {
        out = (uint32_t)n;       /* subnormal (or exactly the smallest normal) */
    } else {
        int expo = unbiased + 127;
        if (n >= 256.0) {        /* rounding carried into the next binade */
            n = 128.0;
            expo += 1;
        }
        if (expo >= 255)
            return (uint16_t)(sign | 0x7F80u);
        out = ((uint32_t)expo << 7) | ((uint32_t)n - 128u);
    }
    return (uint16_t)(sign | out);
}

/* Element types of activations and outputs. */
enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

static float elem_to_float(uint16_t v, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_float(v) : oracle_half_to_float(v);
}

static uint16_t float_to_elem(float f, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_float_to_bf16(f) : oracle_float_to_half(f);
}

void oracle_bf16_to_float_array(const uint16_t* b, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_float(b[i]);
}

void oracle_float_to_bf16_array(const float* f, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_float_to_bf16(f[i]);
}

void oracle_half_to_float_array(const uint16_t* h, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_half_to_float(h[i]);
}

void oracle_float_to_half_array(const float* f, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_float_to_half(f[i]);
}

/* ------------------------------------------------------------------------ */
/* Symmetric min-max quantization of one block of fp16 values.               */
/* ------------------------------------------------------------------------ */

/* Quantizes the n contiguous values v[0..n) (fp16 or bf16 bit patterns)
   with the given qmax. Writes the codes to out[0..n) and returns the fp32
   scale. */
static float quantize_block_t(const uint16_t* v, int64_t n, float qmax, int8_t* out, int dtype)
{
    float absmax = 0.0f;
    for (int64_t k = 0; k < n; ++k) {
        float a = fabsf(elem_to_float(v[k], dtype));
        if (a > absmax)
            absmax = a;
    }
    if (absmax == 0.0f) {
        for (int64_t k = 0; k < n; ++k)
            out[k] = 0;
        return 0.0f;
    }
    float scale = absmax / qmax; /* never 0 here: absmax >= 2^-133 (bf16), 2^-24 (fp16) */
    for (int64_t k = 0; k < n; ++k) {
        float x = elem_to_float(v[k], dtype);
        float r = rintf(x / scale);
        if (r > qmax)
            r = qmax;
        if (r < -qmax)
            r = -qmax;
        out[k] = (int8_t)r;
    }
    return scale;
}

static float quantize_block(const uint16_t* v, int64_t n, float qmax, int8_t* out)
{
    return quantize_block_t(v, n, qmax, out, ORACLE_F16);
}

/* ------------------------------------------------------------------------ */
/* Percentile-clipped weight scales (README "LLM Quantization" note: besides */
/* min-max, "the 99th percentile method (clip_percentile=99.9)").           */
/* Reading: the clip value c of a block is the p-th percentile of its |w|,  */
/* by linear interpolation between order statistics (sorted |w| q[0..n),     */
/* position h = (n - 1) * p / 100, c = q[i] + (h - i) * (q[i+1] - q[i]),     */
/* i = floor(h), evaluated in binary64 and rounded to binary32); then        */
/* scale = c / qmax and code = clamp(rint(w / scale)) as for min-max, values */
/* beyond c saturating at +-qmax. p = 100 gives c = absmax (min-max).        */
/* ------------------------------------------------------------------------ */

static int cmp_float(const void* a, const void* b)
{
    float x = *(const float*)a, y = *(const float*)b;
    return (x > y) - (x < y);
}

static float quantize_block_pct(const uint16_t* v, int64_t n, float qmax, double pct,
                                int8_t* out, int dtype)
{
    float* q = (float*)malloc((size_t)n * sizeof(float));
    if (!q)
        return -1.0f;
    for (int64_t k = 0; k < n; ++k)
        q[k] = fabsf(elem_to_float(v[k], dtype));
    qsort(q, (size_t)n, sizeof(float), cmp_float);
    double h = (double)(n - 1) * pct / 100.0;
    int64_t i = (int64_t)floor(h);
    double c = (i + 1 < n) ? (double)q[i] + (h - (double)i) * ((double)q[i + 1] - (double)q[i])
                           : (double)q[n - 1];
    free(q);
    float clip = (float)c;
    if (clip == 0.0f) {
        for (int64_t k = 0; k < n; ++k)
            out[k] = 0;
        return 0.0f;
    }
    float scale = clip / qmax;
    for (int64_t k = 0; k < n; ++k) {
        float r = rintf(elem_to_float(v[k], dtype) / scale);
        if (r > qmax)
            r = qmax;
        if (r < -qmax)
            r = -qmax;
        out[k] = (int8_t)r;
    }
    return scale;
}

/* Codes [N,K] (int8, in [-qmax, qmax]) and scales [N, K/gs] of weights w
   (fp16, or bf16 with w_dtype 1) with percentile-clipped scales; qmax 127
   (INT8) or 7 (INT4, packed by the caller). */
int oracle_quantize_weight_pct(const uint16_t* w, int32_t w_dtype, int64_t N, int64_t K,
                               int32_t group_size, double pct, float qmax, int8_t* codes,
                               float* s_w)
{
    if (group_size < 0 || (group_size > 0 && K % group_size != 0) || !(pct > 0.0) ||
        pct > 100.0)
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
    int rc = 0;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            float sc = quantize_block_pct(w + n * K + g * gs, gs, qmax, pct,
                                          codes + n * K + g * gs, w_dtype);
            if (sc < 0.0f)
                rc = 2;
            s_w[n * G + g] = sc;
        }
    return rc;
}

/* Per-token activation quantization: x [M,K] (fp16, or bf16 with x_dtype 1)
   -> q int8 [M,K], s [M]. */
void oracle_quantize_act_ex(const uint16_t* x, int32_t x_dtype, int64_t M, int64_t K, int8_t* q,
                            float* s)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        s[m] = quantize_block_t(x + m * K, K, 127.0f, q + m * K, x_dtype);
}

void oracle_quantize_act(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* s)
{
    oracle_quantize_act_ex(x, ORACLE_F16, M, K, q, s);
}

/* INT8 weight quantization: w fp16 [N,K] -> wq int8 [N,K].
   group_size 0: one scale per output channel, s_w [N].
   group_size gs > 0: one scale per (n, g), g = k / gs, s_w [N, K/gs]. */
int oracle_quantize_weight_int8(const uint16_t* w, int64_t N, int64_t K, int32_t group_size,
                                int8_t* wq, float* s_w)
{
    if (group_size < 0 || (group_size > 0 && K % group_size != 0))
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g)
            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 127.0f, wq + n * K + g * gs);
    return 0;
}

/* INT4 weight quantization and packing: codes in [-7, 7] with scale
   absmax/7 per output channel (group_size 0) or per (n, g) group; the
   nibble stored is code + 8; byte j of row n = nib[2j] | nib[2j+1] << 4. */
int oracle_pack_weight_int4(const uint16_t* w, int64_t N, int64_t K, int32_t group_size,
                            uint8_t* wp, float* s_w)
{
    if (K % 2 != 0 || group_size < 0 || (group_size > 0 && K % group_size != 0))
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
    int rc = 0;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        int8_t* codes = (int8_t*)malloc((size_t)K);
        if (!codes) {
            rc = 2;
            continue;
        }
        for (int64_t g = 0; g < G; ++g)
            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 7.0f, codes + g * gs);
        for (int64_t j = 0; j < K / 2; ++j) {
            uint8_t lo = (uint8_t)(codes[2 * j] + 8);
            uint8_t hi = (uint8_t)(codes[2 * j + 1] + 8);
            wp[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
        free(codes);
    }
    return rc;
}

/* Inverse of the packing: nibble b -> code b - 8 (a nibble of 0 decodes to
   -8 even though the quantizer never writes it). */
void oracle_unpack_int4(const uint8_t* wp, int64_t N, int64_t K, int8_t* wq)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            uint8_t b = wp[n * (K / 2) + j];
            wq[n * K + 2 * j] = (int8_t)((int)(b & 0x0F) - 8);
            wq[n * K + 2 * j + 1] = (int8_t)((int)(b >> 4) - 8);
        }
}

/* ------------------------------------------------------------------------ */
/* INT8 x INT8 -> INT32 products.                                            */
/* ------------------------------------------------------------------------ */

/* acc[m,n] = sum_k q[m,k] * wq[n,k] in int32 (group_size 0, out [M,N]), or
   the per-group partials P[m,n,g] = sum_{k in group g} q[m,k] * wq[n,k]
   (group_size gs, out [M,N,K/gs]). Both operands are K-contiguous, so this
   is y = x W^T with W stored [out_features, in_features]. */
int oracle_gemm_s32(const int8_t* q, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                    int32_t group_size, int32_t* out)
{
    if (group_size < 0 || (group_size > 0 && K % group_size != 0))
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t g = 0; g < G; ++g) {
                int32_t acc = 0;
                for (int64_t k = g * gs; k < (g + 1) * gs; ++k)
                    acc += (int32_t)q[m * K + k] * (int32_t)wq[n * K + k];
                if (group_size == 0)
                    out[m * N + n] = acc;
                else
                    out[(m * N + n) * G + g] = acc;
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequant epilogues.                                                        */
/* ------------------------------------------------------------------------ */

/* Per-channel: C_fp16 = C_int32 * s_act * s_weight, left to right (the
   output rounded to fp16, or to bf16 with y_dtype 1). */
uint16_t oracle_epilogue_pc_ex(int32_t acc, float s_act, float s_weight, int32_t y_dtype)
{
    float t = (float)acc * s_act;
    t = t * s_weight;
    return float_to_elem(t, y_dtype);
}

uint16_t oracle_epilogue_pc(int32_t acc, float s_act, float s_weight)
{
    return oracle_epilogue_pc_ex(acc, s_act, s_weight, ORACLE_F16);
}

/* Per-group: each group's int32 partial is rescaled by its weight scale and
   summed in ascending group order; the token scale is applied last. */
uint16_t oracle_epilogue_pg_ex(const int32_t* partials, const float* s_weight_row, int64_t G,
                               float s_act, int32_t y_dtype)
{
    float f = 0.0f;
    for (int64_t g = 0; g < G; ++g)
        f = f + (float)partials[g] * s_weight_row[g];
    return float_to_elem(f * s_act, y_dtype);
}

uint16_t oracle_epilogue_pg(const int32_t* partials, const float* s_weight_row, int64_t G,
                            float s_act)
{
    return oracle_epilogue_pg_ex(partials, s_weight_row, G, s_act, ORACLE_F16);
}

/* ------------------------------------------------------------------------ */
/* Whole linear layers: per-token quantize -> INT32 product -> dequant.      */
/* ------------------------------------------------------------------------ */

/* y [M,N] from x [M,K] and INT8 weights wq [N,K] with scales s_w ([N] for
   group_size 0, [N, K/gs] otherwise); x and y are fp16 (dtype 0) or bf16
   (dtype 1). Returns 0 on success. */
int oracle_w8a8_linear_ex(const uint16_t* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                          const int8_t* wq, const float* s_w, int32_t group_size, uint16_t* y,
                          int32_t y_dtype)
{
    if (group_size < 0 || (group_size > 0 && K % group_size != 0))
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        int8_t* q = (int8_t*)malloc((size_t)K);
        int32_t* part = (int32_t*)malloc((size_t)G * sizeof(int32_t));
        if (!q || !part) {
            free(q);
            free(part);
            rc = 2;
            continue;
        }
        float s_act = quantize_block_t(x + m * K, K, 127.0f, q, x_dtype);
        for (int64_t n = 0; n < N; ++n) {
            const int8_t* wrow = wq + n * K;
            for (int64_t g = 0; g < G; ++g) {
                int32_t acc = 0;
                for (int64_t k = g * gs; k < (g + 1) * gs; ++k)
                    acc += (int32_t)q[k] * (int32_t)wrow[k];
                part[g] = acc;
            }
            if (group_size == 0)
                y[m * N + n] = oracle_epilogue_pc_ex(part[0], s_act, s_w[n], y_dtype);
            else
                y[m * N + n] = oracle_epilogue_pg_ex(part, s_w + n * G, G, s_act, y_dtype);
        }
        free(q);
        free(part);
    }
    return rc;
}

int oracle_w8a8_linear(const uint16_t* x, int64_t M, int64_t N, int64_t K, const int8_t* wq,
                       const float* s_w, int32_t group_size, uint16_t* y)
{
    return oracle_w8a8_linear_ex(x, ORACLE_F16, M, N, K, wq, s_w, group_size, y, ORACLE_F16);
}

/* W4A8: unpack the INT4 nibbles to INT8 codes, then the same layer as W8A8
   (per-output-channel scales for group_size 0, per-group otherwise). */
int oracle_w4a8_linear_ex(const uint16_t* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                          const uint8_t* wp, const float* s_w, int32_t group_size, uint16_t* y,
                          int32_t y_dtype)
{
    if (K % 2 != 0)
        return 1;
    int8_t* wq = (int8_t*)malloc((size_t)(N * K));
    if (!wq)
        return 2;
    oracle_unpack_int4(wp, N, K, wq);
    int rc = oracle_w8a8_linear_ex(x, x_dtype, M, N, K, wq, s_w, group_size, y, y_dtype);
    free(wq);
    return rc;
}

int oracle_w4a8_linear(const uint16_t* x, int64_t M, int64_t N, int64_t K, const uint8_t* wp,
                       const float* s_w, int32_t group_size, uint16_t* y)
{
    return oracle_w4a8_linear_ex(x, ORACLE_F16, M, N, K, wp, s_w, group_size, y, ORACLE_F16);
}

/* ------------------------------------------------------------------------ */
/* A16 decode matrix-vector product (weight-only dequantization).           */
/* README "Metal Kernel Pipeline", decode: a matrix-vector kernel "with      */
/* on-the-fly weight dequantization (no activation quantization needed)".    */
/* The activations are used as they are; each weight is dequantized as code  */
/* times its scale. The oracle returns the value of                          */
/*   y[n] = sum_g s_w[n,g] * sum_{k in g} x[k] * wq[n,k]                      */
/* accumulated in binary64 (each x*wq product is exact in binary64; the sums */
/* are far more precise than any binary32 evaluation), unrounded: a GPU      */
/* evaluation in binary32 is compared with it under an error bound.          */
/* w: INT8 codes [N,K] (bits 8) or packed INT4 [N,K/2] (bits 4); s_w [N] for */
/* group_size 0 or [N, K/gs]; x fp16 (dtype 0) or bf16 (dtype 1).            */
/* ------------------------------------------------------------------------ */
int oracle_a16_gemv(const uint16_t* x, int32_t x_dtype, int64_t K, int64_t N, const void* w,
                    int32_t bits, const float* s_w, int32_t group_size, double* y)
{
    if ((bits != 8 && bits != 4) || group_size < 0 || (group_size > 0 && K % group_size != 0) ||
        (bits == 4 && K % 2 != 0))
        return 1;
    int64_t gs = group_size ? group_size : K;
    int64_t G = K / gs;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double total = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            double part = 0.0;
            for (int64_t k = g * gs; k < (g + 1) * gs; ++k) {
                int code;
                if (bits == 8) {
                    code = ((const int8_t*)w)[n * K + k];
                } else {
                    uint8_t b = ((const uint8_t*)w)[n * (K / 2) + k / 2];
                    code = (int)((k % 2) ? (b >> 4) : (b & 0x0F)) - 8;
                }
                part += (double)elem_to_float(x[k], x_dtype) * (double)code;
            }
            total += (double)s_w[n * G + g] * part;
        }
        y[n] = total;
    }
    return 0;
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
