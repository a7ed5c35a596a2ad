/*
 * mxfp8_oracle.c -- plain, slow, single-threaded CPU oracle for the MXFP8
 * block-scaled linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library in mxfp8_block_scaled_x4_gb300/) never calls it and shares
 * no code, header, table or helper with it.
 *
 * What it computes (sources):
 *  - vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear backend",
 *    Purpose section and review thread: BF16 activations are quantized per
 *    call with the 8x4 scale layout; weights are prepared once after load
 *    (K a multiple of 256, scales sliced to [N, K/32], N padded to a multiple
 *    of 128); the block-scaled GEMM output is sliced back to the logical N
 *    and the bias is added.  Only N is padded, never the input.
 *  - prhub summary of vLLM PR #52204, "key source snippets": the size of the
 *    8x4 scale buffer is ceil(m/8)*8 * ceil((k/32)/4)*4 bytes, and the
 *    weight scales are viewed as [N, K/32] (one byte per 32 K elements).
 *  - FlashInfer PR #1214, review of fp4Quantize.cpp: UE8M0 scales go with
 *    32-element blocks.
 *  - The MXFP8 element and scale encodings themselves (E4M3 "fn" elements,
 *    E8M0 power-of-two scale per 32-block, scale exponent =
 *    floor(log2(amax)) - emax(E4M3)=8) follow the public OCP Microscaling
 *    Formats (MX) v1.0 specification, which the pages name by format only.
 *
 * Readings where the pages are silent (labels S1-S12 of the readings):
 *  S1 scale rule (A) = OCP floor rule; rule (B) = smallest power of two that
 *     avoids saturation, kept behind a flag and not used by the layer.
 *  S2 an all-zero block gets scale byte 0x00; its elements keep their sign.
 *  S3 a block holding NaN or Inf gets scale 0xFF and every element 0x7F.
 *  S4 the scale byte is clamped to [0, 254].
 *  S5 E4M3 rounding is round-to-nearest-even with saturation to +-448; the
 *     sign of values that round to zero is kept.
 *  S6 8x4 byte order: offset(m,b) = ((m/8)*(KB/4) + b/4)*32 + (m%8)*4 + b%4,
 *     rows in [M, ceil8(M)) hold 0x00.
 *  S7 prepared weight: data [N_pad][K] row-major (rows >= N are 0x00), scales
 *     in 128-row x 4-block tiles of 512 bytes, tile (t, q) at
 *     ((t*(KB/4)) + q)*512, inner offset (r%32)*16 + (r/32)*4 + (b%4).
 *  S9 bias is added to the exact sum; y_ref is left in double.
 *
 * Everything is computed in double.  Every product of two E4M3 values times
 * two powers of two is exact in double, so the only rounding in y_ref is the
 * order of the cross-block additions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* Value of one E4M3 ("fn" variant: no infinities, S.1111.111 is NaN) byte.
 * Exponent bias 7, 3 mantissa bits, subnormal step 2^-9. */
double oracle_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7) return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);
    else
        mag = ldexp(1.0 + mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* Value of one E8M0 scale byte: 2^(byte-127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Round a finite double to E4M3, nearest with ties to even, saturating
 * magnitudes above the largest finite value (448) to 448.  Keeps the sign of
 * results that are zero. */
uint8_t oracle_e4m3_round(double t) {
    uint8_t sign = signbit(t) ? 0x80 : 0x00;
    double a = fabs(t);
    if (isnan(t)) return 0x7F;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: integer multiples of 2^-9 (code == multiple,
         * and 8 * 2^-9 == 2^-6 is exactly code 0x08, the smallest normal) */
        double u = a * 512.0; /* exact */
        double f = floor(u);
        double rem = u - f;
        if (rem > 0.5 || (rem == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
        return (uint8_t)(sign | (uint8_t)f);
    }
    if (isinf(a)) return (uint8_t)(sign | 0x7E);
    {
        int e = ilogb(a);                 /* floor(log2(a)), exact */
        double frac = (ldexp(a, -e) - 1.0) * 8.0; /* mantissa in units of 1/8, exact */
        double f = floor(frac);
        double rem = frac - f;
        if (rem > 0.5 || (rem == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
        if (f == 8.0) { f = 0.0; e += 1; }
        if (e > 8 || (e == 8 && f > 6.0)) return (uint8_t)(sign | 0x7E); /* 448 */
        return (uint8_t)(sign | ((e + 7) << 3) | (uint8_t)f);
    }
}

/* Array form of oracle_e4m3_round. */
void oracle_e4m3_round_n(const double* t, int64_t n, uint8_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = oracle_e4m3_round(t[i]);
}

/* ---------------------------------------------------------- quantization */

/* Scale byte for one block given amax (> 0, finite).
 * rule 0 (A, the contract): e = floor(log2(amax)) - 8.
 * rule 1 (B): smallest integer e with 448 * 2^e >= amax.
 * Both clamp e + 127 into [0, 254]. */
static int scale_byte_for(double amax, int rule) {
    int e;
    if (rule == 0) {
        e = ilogb(amax) - 8;
    } else {
        e = ilogb(amax) - 9;
        while (ldexp(448.0, e) < amax) e += 1; /* exact comparisons */
    }
    e += 127;
    if (e < 0) e = 0;
    if (e > 254) e = 254;
    return e;
}

/* Quantize one block of 32 values (already widened to double; each value is
 * exactly a float).  Writes 32 element bytes and returns the scale byte. */
uint8_t oracle_quantize_block(const double* v, int rule, uint8_t* elems) {
    double amax = 0.0;
    int nonfinite = 0;
    int i;
    for (i = 0; i < 32; ++i) {
        if (!isfinite(v[i])) nonfinite = 1;
        else if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    if (nonfinite) {                      /* S3 */
        for (i = 0; i < 32; ++i) elems[i] = 0x7F;
        return 0xFF;
    }
    if (amax == 0.0) {                    /* S2 */
        for (i = 0; i < 32; ++i) elems[i] = signbit(v[i]) ? 0x80 : 0x00;
        return 0x00;
    }
    {
        int sb = scale_byte_for(amax, rule);
        for (i = 0; i < 32; ++i) {
            double t = ldexp(v[i], 127 - sb); /* v / 2^(sb-127), exact */
            elems[i] = oracle_e4m3_round(t);
        }
        return (uint8_t)sb;
    }
}

/* Quantize a row-major float matrix [rows, k] (k a multiple of 32) block by
 * block along k.  q: [rows, k] element bytes; sf: [rows, k/32] scale bytes in
 * the plain row-major ("linear") layout. */
void oracle_quantize_rows(const float* x, int64_t rows, int64_t k, int rule,
                          uint8_t* q, uint8_t* sf) {
    int64_t kb = k / 32, r, b;
    double blk[32];
    for (r = 0; r < rows; ++r) {
        for (b = 0; b < kb; ++b) {
            int i;
            for (i = 0; i < 32; ++i) blk[i] = (double)x[r * k + b * 32 + i];
            sf[r * kb + b] = oracle_quantize_block(blk, rule, q + r * k + b * 32);
        }
    }
}

/* Dequantize [rows, k] from element bytes and linear scales into doubles. */
void oracle_dequant_rows(const uint8_t* q, const uint8_t* sf, int64_t rows,
                         int64_t k, double* out) {
    int64_t kb = k / 32, r, j;
    for (r = 0; r < rows; ++r)
        for (j = 0; j < k; ++j)
            out[r * k + j] = oracle_e4m3_value(q[r * k + j]) *
                             oracle_e8m0_value(sf[r * kb + j / 32]);
}

/* ---------------------------------------------------------------- layouts */

/* Byte offset of the scale of (row m, block b) in the 8x4 layout (S6). */
int64_t oracle_offset_8x4(int64_t m, int64_t b, int64_t kb) {
    return ((m / 8) * (kb / 4) + b / 4) * 32 + (m % 8) * 4 + (b % 4);
}

int64_t oracle_act_scale_bytes(int64_t m, int64_t k) {
    int64_t kb = k / 32;
    return ((m + 7) / 8) * 8 * (((kb + 3) / 4) * 4);
}

/* Linear [m, k/32] scales -> 8x4 layout (rows >= m are zero). */
void oracle_act_scale_8x4(const uint8_t* sf_lin, int64_t m, int64_t k,
                          uint8_t* out) {
    int64_t kb = k / 32, r, b;
    memset(out, 0, (size_t)oracle_act_scale_bytes(m, k));
    for (r = 0; r < m; ++r)
        for (b = 0; b < kb; ++b)
            out[oracle_offset_8x4(r, b, kb)] = sf_lin[r * kb + b];
}

/* Byte offset of the scale of (row n, block b) in the prepared-weight scale
 * layout (S7). */
int64_t oracle_offset_w128x4(int64_t n, int64_t b, int64_t kb) {
    int64_t t = n / 128, r = n % 128;
    return (t * (kb / 4) + b / 4) * 512 + (r % 32) * 16 + (r / 32) * 4 + (b % 4);
}

/* Quantized weight [n, k] + linear scales -> padded data [n_pad, k] and
 * tiled scales [n_pad * k/32]; padding rows are zero in both. */
void oracle_weight_layout(const uint8_t* q, const uint8_t* sf_lin, int64_t n,
                          int64_t k, uint8_t* q_pad, uint8_t* sf_tiled) {
    int64_t kb = k / 32, n_pad = ((n + 127) / 128) * 128, r, b;
    memset(q_pad, 0, (size_t)(n_pad * k));
    memset(sf_tiled, 0, (size_t)(n_pad * kb));
    memcpy(q_pad, q, (size_t)(n * k));
    for (r = 0; r < n; ++r)
        for (b = 0; b < kb; ++b)
            sf_tiled[oracle_offset_w128x4(r, b, kb)] = sf_lin[r * kb + b];
}

/* ---------------------------------------------------------------- linear */

/* One output row, written as the block-scaled sum of the method:
 *   y[j] = sum_b 2^(sa[b]-127) * 2^(sw[j,b]-127) * sum_{k in b} e4m3(qa[k]) * e4m3(qw[j,k])
 * (+ bias[j]) for j < n.  Each inner 32-term sum of E4M3 products is exact in
 * double, as is its scaling by the two powers of two. */
static void linear_row(const uint8_t* qa, const uint8_t* sa, const uint8_t* wq,
                       const uint8_t* wsf, int64_t n, int64_t k,
                       const float* bias, double* y) {
    int64_t kb = k / 32, j, b, i;
    double tab[256];
    double* a = (double*)malloc(sizeof(double) * (size_t)k);
    for (i = 0; i < 256; ++i) tab[i] = oracle_e4m3_value((uint8_t)i);
    for (i = 0; i < k; ++i) a[i] = tab[qa[i]];
    for (j = 0; j < n; ++j) {
        const uint8_t* wr = wq + j * k;
        const uint8_t* ws = wsf + j * kb;
        double acc = 0.0;
        for (b = 0; b < kb; ++b) {
            double part = 0.0;
            for (i = b * 32; i < b * 32 + 32; ++i) part += a[i] * tab[wr[i]];
            acc += part * (oracle_e8m0_value(sa[b]) * oracle_e8m0_value(ws[b]));
        }
        if (bias) acc += (double)bias[j];
        y[j] = acc;
    }
    free(a);
}

/* The layer: quantize activation rows (rule A), multiply by the quantized
 * weight (given as [n, k] bytes + linear [n, k/32] scales), add bias.
 * rows_sel (nullable): compute only these rows, in this order, writing
 * y[i * n + j] for the i-th selected row; otherwise all m rows. */
void oracle_linear(const float* x, int64_t m, int64_t k, const uint8_t* wq,
                   const uint8_t* wsf, int64_t n, const float* bias,
                   const int64_t* rows_sel, int64_t n_sel, double* y) {
    int64_t cnt = rows_sel ? n_sel : m, i;
    uint8_t* qa = (uint8_t*)malloc((size_t)k);
    uint8_t* sa = (uint8_t*)malloc((size_t)(k / 32));
    for (i = 0; i < cnt; ++i) {
        int64_t r = rows_sel ? rows_sel[i] : i;
        oracle_quantize_rows(x + r * k, 1, k, 0, qa, sa);
        linear_row(qa, sa, wq, wsf, n, k, bias, y + i * n);
    }
    free(qa);
    free(sa);
}

/* Grouped (MoE gate_up) layer: rows [off[e], off[e+1]) of the expert-sorted
 * activations use expert e's weight ([e][n][k] bytes, [e][n][k/32] linear
 * scales) and bias ([e][n], nullable).  rows_sel as in oracle_linear. */
void oracle_grouped_linear(const float* x, int64_t rows, int64_t k,
                           const int32_t* off, int64_t num_experts,
                           const uint8_t* wq, const uint8_t* wsf, int64_t n,
                           const float* bias, const int64_t* rows_sel,
                           int64_t n_sel, double* y) {
    int64_t cnt = rows_sel ? n_sel : rows, i, kb = k / 32;
    uint8_t* qa = (uint8_t*)malloc((size_t)k);
    uint8_t* sa = (uint8_t*)malloc((size_t)kb);
    for (i = 0; i < cnt; ++i) {
        int64_t r = rows_sel ? rows_sel[i] : i, e = 0;
        while (e < num_experts && !(r >= off[e] && r < off[e + 1])) ++e;
        if (e == num_experts) { /* row not covered by any segment */
            int64_t j;
            for (j = 0; j < n; ++j) y[i * n + j] = NAN;
            continue;
        }
        oracle_quantize_rows(x + r * k, 1, k, 0, qa, sa);
        linear_row(qa, sa, wq + e * n * k, wsf + e * n * kb, n, k,
                   bias ? bias + e * n : NULL, y + i * n);
    }
    free(qa);
    free(sa);
}
