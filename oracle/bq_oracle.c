/*
 * Oracle for the block-quantized wire codec: a plain, slow, single-threaded CPU
 * statement of what every codec operation computes.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The GPU library shares no code, header,
 * table or helper with it, and neither side includes or links the other.
 *
 * Build flags (oracle/__init__.py): gcc -O2 -std=c11 -ffp-contract=off
 * -fno-fast-math. No a*b+c is ever contracted into a fused multiply-add, and
 * binary32 expressions are evaluated in binary32 (FLT_EVAL_METHOD == 0 on the
 * x86-64 and aarch64 hosts this runs on), so every `float` operation below is
 * one IEEE-754 binary32 operation rounded to nearest, ties to even.
 *
 * Where each rule comes from (pull-request pages on the wire codec):
 *   [I8]  "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A"
 *         - Summary: each 128-value block is 128 signed payload bytes plus one
 *           FP32 scale equal to amax/127 (132 bytes per block); owners
 *           materialize from the same final payload that is forwarded.
 *         - Implementation: the four kernels (BF16 -> INT8 quantize, INT8 -> BF16
 *           materialize, multi-source dequantize with FP32 accumulation, fused
 *           dequantize-add-requantize ring hop).
 *         - Summary of the change (the proofs list): zero blocks, the
 *           half-quantization-step error bound.
 *   [MX]  "feat(pcie_dma): add INT8 and MXFP8 wire modes"
 *         - Summary: MXFP8 = E4M3 values with one E8M0 scale per 32 values.
 *         - Review comment on mxfp8_scale_byte: an all-zero group gets scale byte
 *           127; otherwise the scale byte is the E8M0 conversion of
 *           amax / (largest finite E4M3), saturating, rounded toward +infinity.
 *   [ST]  "[II] Support staged MXFP8 linear inputs"
 *         - Behavior / Compatibility: a 128-column-aligned slice is quantized into
 *           a column offset of a wider caller-owned buffer, keeping the per-32-
 *           column groups.
 *
 * Readings taken where the pages are silent (each is listed with its reason in
 * the design notes of this repository):
 *   R1  payload rounding: q = nearest integer to fl(x / s), ties to even, then
 *       clamped to [-127, 127];
 *   R2  a block whose scale is zero (amax == 0, or an FP32 amax so small that
 *       amax/127 underflows to zero) has payload 0;
 *   R3  materialization rounds twice: fl(q * s) in binary32, then binary32 ->
 *       BF16 to nearest, ties to even;
 *   R4  accumulation is d_0 + d_1 + ... + d_{W-1} evaluated left to right in
 *       binary32, d_w = fl(q_w * s_w);
 *   R5  the "largest finite E4M3" is 448; E4M3 is the OCP format (bias 7, no
 *       infinities, 0x7F/0xFF are NaN), values are rounded to nearest, ties to
 *       even, saturated to +-448, and the sign of zero is kept;
 *   R6  the MX value fed to E4M3 is x * 2^(127 - e), which is x divided by the
 *       group's power-of-two scale;
 *   R7  inputs are finite; results for NaN or infinity are not specified (this
 *       includes an E8M0 byte of 255 and a wire element whose decoded value lies
 *       outside the binary32 range);
 *   R11 the MX all-to-all reduction follows the INT8 one with the MX codec: each
 *       source element is decoded to binary32 (exactly), the sources are added left
 *       to right in source order in binary32, and the sum is requantized group by
 *       group with the MX rules, the amax taken over the binary32 sums;
 *   R12 the MX ring hop is v = fl(decode(q_in) * 2^(e_in - 127) + x_local),
 *       requantized with the MX rules.
 * [MX] Summary names the mx_a2a and mx_ring modes on the same topologies as the
 * INT8 modes and says every mode materializes the owner shard from the payload it
 * forwards; R11 and R12 are the plainest readings of those modes.
 *   R13 the i8 mode's BF16 reduce-scatter ([I8] Summary: "i8" is a BF16
 *       reduce-scatter followed by an INT8 all-gather) sums the W ranks' BF16 shards
 *       left to right in rank order in binary32 and rounds the sum once to BF16 (the
 *       reduce-scatter's BF16 result); the all-gather payload is quant_i8 of that
 *       BF16 shard, and the owner materializes that payload;
 *   R14 the legacy E4M3 codec ([I8] Summary and Why: one E4M3 byte per value and one
 *       FP32 scale per 128-value block, 132 bytes per block) quantizes like block INT8
 *       with 448 in place of 127: s = fl(amax / 448), code = E4M3 (nearest, ties to
 *       even, saturated) of fl(x / s); a block with s == 0 has every code 0x00;
 *       materialization is BF16(fl(decode(code) * s));
 *   R15 an FP16 slice ([ST] Behavior: BF16 or FP16 feature slices) is widened
 *       exactly to binary32 and quantized with the MX rules unchanged.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define BQO_BLOCK 128   /* [I8] Summary: values per INT8 block */
#define BQO_GROUP 32    /* [MX] Summary: values per E8M0 scale */

/* ------------------------------------------------------------------------ */
/* Number formats, from their definitions.                                   */
/* ------------------------------------------------------------------------ */

/* BF16 is the upper half of a binary32 pattern, so widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Value of a non-negative BF16 code, with the infinity code 0x7F80 standing for
 * 2^128 so that it can act as the next value above the largest finite one. */
static double bf16_code_value(uint32_t code)
{
    if (code == 0x7F80u) return ldexp(1.0, 128);
    return (double)bf16_bits_to_float((uint16_t)code);
}

/* Round a real number (given exactly as a double) to BF16, to nearest, ties to
 * the even code; magnitudes at or beyond the midpoint between the largest finite
 * BF16 and 2^128 give infinity. Written as a search for the two neighbouring
 * codes, which is the definition of rounding to nearest. */
uint16_t bqo_bf16_round(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    if (a >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    /* largest code lo in [0, 0x7F80) with value(lo) <= a */
    uint32_t lo = 0, hi = 0x7F80u;
    while (hi - lo > 1) {
        uint32_t mid = lo + (hi - lo) / 2;
        if (bf16_code_value(mid) <= a) lo = mid; else hi = mid;
    }
    /* neighbours: value(lo) <= a < value(lo + 1) */
    uint32_t up = lo + 1;
    double below = a - bf16_code_value(lo);   /* exact: Sterbenz / small operands */
    double above = bf16_code_value(up) - a;
    uint32_t pick;
    if (below < above) pick = lo;
    else if (above < below) pick = up;
    else pick = (lo % 2 == 0) ? lo : up;   /* tie: even code */
    return (uint16_t)(sign | pick);
}

/* IEEE binary16: 1 sign bit, 5 exponent bits with bias 15, 10 fraction bits;
 * exponent field 0 holds the subnormals f * 2^-24. Every value is exact in
 * binary32. (Infinities and NaN are not inputs, reading R7.) */
static float f16_bits_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0) mag = ldexp((double)f, -24);
    else if (e == 31) mag = f ? NAN : INFINITY;
    else mag = ldexp(1024.0 + f, e - 25);
    return (float)(sign ? -mag : mag);
}

/* E4M3 (OCP): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 holds the subnormals m * 2^-9; 0x7F and 0xFF are NaN. */
double bqo_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if ((c & 0x7F) == 0x7F) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest E4M3 code to y, ties to the even code, saturated to +-448 ([MX]
 * review: SATFINITE), sign of zero kept (reading R5). */
uint8_t bqo_e4m3_encode(double y)
{
    uint8_t sign = signbit(y) ? 0x80u : 0u;
    double a = fabs(y);
    if (isnan(y)) return (uint8_t)(sign | 0x7Fu);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    /* codes 0x00..0x7E are the non-negative finite values, in increasing order;
     * find the largest code lo with value(lo) <= a (a < 448 = value(0x7E)) */
    int lo = 0, hi = 0x7E;
    while (hi - lo > 1) {
        int mid = lo + (hi - lo) / 2;
        if (bqo_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    int up = lo + 1;
    double below = a - bqo_e4m3_decode((uint8_t)lo);
    double above = bqo_e4m3_decode((uint8_t)up) - a;
    int pick;
    if (below < above) pick = lo;
    else if (above < below) pick = up;
    else pick = (lo % 2 == 0) ? lo : up;
    return (uint8_t)(sign | pick);
}

/* [MX] review, mxfp8_scale_byte: zero amax -> 127; otherwise the E8M0 value of
 * v = fl(amax / 448) rounded toward +infinity, i.e. the smallest power of two
 * 2^(b-127), b in [0, 254], that is >= v, saturating at b = 254. */
uint8_t bqo_e8m0_scale(float amax)
{
    if (amax == 0.0f) return 127;
    float v = amax / 448.0f;
    if (ldexp(1.0, 254 - 127) < (double)v) return 254;   /* saturate */
    /* smallest b with 2^(b-127) >= v; the predicate is monotone in b */
    int lo = -1, hi = 254;   /* pred(lo) false (or lo = -1), pred(hi) true */
    while (hi - lo > 1) {
        int mid = lo + (hi - lo) / 2;
        if (ldexp(1.0, mid - 127) >= (double)v) hi = mid; else lo = mid;
    }
    return (uint8_t)hi;
}

/* Round a binary32 value to the nearest integer, ties to even (reading R1). */
static float round_half_even(float t)
{
    float f = floorf(t);     /* exact */
    float d = t - f;         /* exact for the |t| < 2^23 that occur here */
    if (d > 0.5f) return f + 1.0f;
    if (d < 0.5f) return f;
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

/* ------------------------------------------------------------------------ */
/* Block INT8 ([I8]).                                                        */
/* ------------------------------------------------------------------------ */

/* One block: values v[0..127] are exact binary32 numbers (BF16 inputs widened,
 * or FP32 sums). Writes 128 payload bytes and the block's scale. */
static void quant_block_i8(const float *v, int8_t *q, float *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < BQO_BLOCK; i++) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;   /* [I8] Summary: scale = amax / 127, one binary32 division */
    *scale = s;
    for (int i = 0; i < BQO_BLOCK; i++) {
        if (s == 0.0f) { q[i] = 0; continue; }   /* reading R2 */
        float t = v[i] / s;                      /* binary32 quotient */
        float r = round_half_even(t);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

/* Materialize one value (reading R3): binary32 product, then BF16. */
static uint16_t materialize_i8(int8_t q, float s)
{
    float d = (float)q * s;
    return bqo_bf16_round((double)d);
}

/* BF16 [n] -> payload [n] + scales [n/128]. Returns 0, or -1 if n % 128 != 0. */
int bqo_quant_i8(const uint16_t *x, int64_t n, int8_t *q, float *scales)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    float v[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) v[i] = bf16_bits_to_float(x[b * BQO_BLOCK + i]);
        quant_block_i8(v, q + b * BQO_BLOCK, scales + b);
    }
    return 0;
}

/* payload [n] + scales [n/128] -> BF16 [n]. */
int bqo_dequant_i8(const int8_t *q, const float *scales, int64_t n, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    for (int64_t i = 0; i < n; i++) out[i] = materialize_i8(q[i], scales[i / BQO_BLOCK]);
    return 0;
}

/* [I8] Implementation, multi-source dequantize with FP32 accumulation: for
 * every element, d_w = fl(q_w * s_w) and acc = (((d_0 + d_1) + d_2) + ...) in
 * source order (reading R4); acc is requantized like quant_i8. When out is not
 * NULL it receives the materialization of the new payload ([I8] Summary: the
 * owner materializes from the payload it forwards). */
int bqo_dequant_accum_i8(const int8_t *const *q_srcs, const float *const *scale_srcs, int W,
                         int64_t n, int8_t *q_out, float *scales_out, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK || W < 1) return -1;
    float acc[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) {
            int64_t e = b * BQO_BLOCK + i;
            float a = (float)q_srcs[0][e] * scale_srcs[0][b];
            for (int w = 1; w < W; w++) {
                float d = (float)q_srcs[w][e] * scale_srcs[w][b];
                a = a + d;
            }
            acc[i] = a;
        }
        quant_block_i8(acc, q_out + b * BQO_BLOCK, scales_out + b);
    }
    if (out) bqo_dequant_i8(q_out, scales_out, n, out);
    return 0;
}

/* [I8] Implementation, fused ring hop: v = fl(fl(q_in * s_in) + x_local),
 * requantized like quant_i8; optional materialization of the new payload. */
int bqo_ring_hop_i8(const int8_t *q_in, const float *s_in, const uint16_t *x_local, int64_t n,
                    int8_t *q_out, float *s_out, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    float v[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) {
            int64_t e = b * BQO_BLOCK + i;
            float d = (float)q_in[e] * s_in[b];
            v[i] = d + bf16_bits_to_float(x_local[e]);
        }
        quant_block_i8(v, q_out + b * BQO_BLOCK, s_out + b);
    }
    if (out) bqo_dequant_i8(q_out, s_out, n, out);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* MXFP8 ([MX], [ST]).                                                       */
/* ------------------------------------------------------------------------ */

/* BF16 [rows, cols] (row stride ld_x elements) -> E4M3 [rows, cols] (row stride
 * ld_q bytes) + E8M0 [rows, cols/32] (row stride ld_s bytes). Group g of row r
 * covers columns [32g, 32g + 32). A slice is addressed by offsetting the three
 * pointers; [ST] Compatibility asks for 128-column alignment, checked here on
 * cols only because the offset is the caller's pointer arithmetic. */
static int quant_mx_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                         int64_t ld_q, uint8_t *s, int64_t ld_s, float (*widen)(uint16_t))
{
    if (rows < 0 || cols < 0 || cols % 128) return -1;
    if (ld_x < cols || ld_q < cols || ld_s < cols / BQO_GROUP) return -1;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t g = 0; g < cols / BQO_GROUP; g++) {
            const uint16_t *xg = x + r * ld_x + g * BQO_GROUP;
            float amax = 0.0f;
            for (int i = 0; i < BQO_GROUP; i++) {
                float a = fabsf(widen(xg[i]));
                if (a > amax) amax = a;
            }
            uint8_t e = bqo_e8m0_scale(amax);
            s[r * ld_s + g] = e;
            for (int i = 0; i < BQO_GROUP; i++) {
                /* reading R6: exact scaling by 2^(127-e) (in double, no rounding) */
                double y = ldexp((double)widen(xg[i]), 127 - (int)e);
                q[r * ld_q + g * BQO_GROUP + i] = bqo_e4m3_encode(y);
            }
        }
    }
    return 0;
}

int bqo_quant_mx(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                 uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s)
{
    return quant_mx_rows(x, rows, cols, ld_x, q, ld_q, s, ld_s, bf16_bits_to_float);
}

/* The same for an FP16 input slice (reading R15). */
int bqo_quant_mx_f16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                     uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s)
{
    return quant_mx_rows(x, rows, cols, ld_x, q, ld_q, s, ld_s, f16_bits_to_float);
}

/* FP16 bits -> binary32 (exposed for the pins). */
float bqo_f16_to_float(uint16_t h) { return f16_bits_to_float(h); }

/* E4M3 + E8M0 -> BF16: out = BF16(decode(byte) * 2^(e-127)); the product is a
 * 4-significant-bit number >= 2^-136 and so exact, leaving one rounding. */
int bqo_dequant_mx(const uint8_t *q, int64_t ld_q, const uint8_t *s, int64_t ld_s,
                   int64_t rows, int64_t cols, uint16_t *out, int64_t ld_out)
{
    if (rows < 0 || cols < 0 || cols % 128) return -1;
    if (ld_q < cols || ld_s < cols / BQO_GROUP || ld_out < cols) return -1;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            uint8_t e = s[r * ld_s + c / BQO_GROUP];
            double v = ldexp(bqo_e4m3_decode(q[r * ld_q + c]), (int)e - 127);
            out[r * ld_out + c] = bqo_bf16_round(v);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* MXFP8 wire reductions ([MX] Summary: mx_a2a and mx_ring).                 */
/* A flat MX wire of n values (n % 128 == 0) is E4M3 codes [n] followed by   */
/* E8M0 bytes [n/32]; group g covers elements [32g, 32g + 32).               */
/* ------------------------------------------------------------------------ */

/* One wire element as binary32: decode(code) * 2^(e - 127). The exact product
 * has at most four significant bits and magnitude >= 2^-136 (or is zero), so the
 * conversion to binary32 is exact whenever the value is in range (reading R7). */
static float mx_element(uint8_t code, uint8_t e)
{
    return (float)ldexp(bqo_e4m3_decode(code), (int)e - 127);
}

/* Requantize one group of 32 binary32 values with the rules bqo_quant_mx applies
 * to BF16 input: E8M0 byte of the group's amax, then each value scaled exactly by
 * 2^(127 - e) (reading R6, in double, no rounding) and encoded as E4M3. */
static void quant_group_mx(const float *v, uint8_t *q, uint8_t *s)
{
    float amax = 0.0f;
    for (int i = 0; i < BQO_GROUP; i++) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    uint8_t e = bqo_e8m0_scale(amax);
    *s = e;
    for (int i = 0; i < BQO_GROUP; i++) q[i] = bqo_e4m3_encode(ldexp((double)v[i], 127 - (int)e));
}

/* mx_a2a reduction (reading R11): d_w = decode(q_w) * 2^(e_w - 127) and
 * acc = (((d_0 + d_1) + d_2) + ...) in binary32, in source order; acc is
 * requantized group by group. When out is not NULL it receives the
 * materialization of the new payload (the owner's copy of what it forwards). */
int bqo_dequant_accum_mx(const uint8_t *const *q_srcs, const uint8_t *const *s_srcs, int W, int64_t n,
                         uint8_t *q_out, uint8_t *s_out, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK || W < 1) return -1;
    float acc[BQO_GROUP];
    for (int64_t g = 0; g < n / BQO_GROUP; g++) {
        for (int i = 0; i < BQO_GROUP; i++) {
            int64_t e = g * BQO_GROUP + i;
            float a = mx_element(q_srcs[0][e], s_srcs[0][g]);
            for (int w = 1; w < W; w++) {
                float d = mx_element(q_srcs[w][e], s_srcs[w][g]);
                a = a + d;
            }
            acc[i] = a;
        }
        quant_group_mx(acc, q_out + g * BQO_GROUP, s_out + g);
    }
    if (out) bqo_dequant_mx(q_out, n, s_out, n / BQO_GROUP, n ? 1 : 0, n, out, n);
    return 0;
}

/* mx_ring hop (reading R12): v = fl(decode(q_in) * 2^(e_in - 127) + x_local),
 * requantized group by group; optional materialization of the new payload. */
int bqo_ring_hop_mx(const uint8_t *q_in, const uint8_t *s_in, const uint16_t *x_local, int64_t n,
                    uint8_t *q_out, uint8_t *s_out, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    float v[BQO_GROUP];
    for (int64_t g = 0; g < n / BQO_GROUP; g++) {
        for (int i = 0; i < BQO_GROUP; i++) {
            int64_t e = g * BQO_GROUP + i;
            float d = mx_element(q_in[e], s_in[g]);
            v[i] = d + bf16_bits_to_float(x_local[e]);
        }
        quant_group_mx(v, q_out + g * BQO_GROUP, s_out + g);
    }
    if (out) bqo_dequant_mx(q_out, n, s_out, n / BQO_GROUP, n ? 1 : 0, n, out, n);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The i8 mode's BF16 reduce-scatter fused with the INT8 all-gather payload. */
/* ------------------------------------------------------------------------ */

/* Reading R13: for every element, acc = x_0 + x_1 + ... + x_{W-1} in binary32 in
 * rank order, y = BF16(acc); each 128-value block of y is quantized like
 * quant_i8; out (when not NULL) receives the materialization of the payload. */
int bqo_reduce_quant_i8(const uint16_t *const *x_srcs, int W, int64_t n, int8_t *q, float *scales,
                        uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK || W < 1) return -1;
    float y[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) {
            int64_t e = b * BQO_BLOCK + i;
            float a = bf16_bits_to_float(x_srcs[0][e]);
            for (int w = 1; w < W; w++) a = a + bf16_bits_to_float(x_srcs[w][e]);
            y[i] = bf16_bits_to_float(bqo_bf16_round((double)a));
        }
        quant_block_i8(y, q + b * BQO_BLOCK, scales + b);
    }
    if (out) bqo_dequant_i8(q, scales, n, out);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Legacy E4M3 codec (reading R14): one E4M3 byte per value, one FP32 scale  */
/* per 128-value block, the same 132-byte block as block INT8.               */
/* ------------------------------------------------------------------------ */

static void quant_block_e4m3(const float *v, uint8_t *q, float *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < BQO_BLOCK; i++) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int i = 0; i < BQO_BLOCK; i++) {
        if (s == 0.0f) {
            q[i] = 0;
            continue;
        }
        float t = v[i] / s;   /* binary32 quotient, then the E4M3 grid */
        q[i] = bqo_e4m3_encode((double)t);
    }
}

int bqo_quant_e4m3(const uint16_t *x, int64_t n, uint8_t *q, float *scales)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    float v[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) v[i] = bf16_bits_to_float(x[b * BQO_BLOCK + i]);
        quant_block_e4m3(v, q + b * BQO_BLOCK, scales + b);
    }
    return 0;
}

/* out = BF16(fl(decode(code) * s)): decode is exact in binary32, the product is
 * rounded to binary32, then to BF16 (two roundings, as for block INT8). */
int bqo_dequant_e4m3(const uint8_t *q, const float *scales, int64_t n, uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK) return -1;
    for (int64_t e = 0; e < n; e++) {
        float d = (float)bqo_e4m3_decode(q[e]);
        float p = d * scales[e / BQO_BLOCK];
        out[e] = bqo_bf16_round((double)p);
    }
    return 0;
}

/* The E4M3 all-gather mode's BF16 reduce-scatter fused with its payload: R13 with
 * the E4M3 codec in place of block INT8. */
int bqo_reduce_quant_e4m3(const uint16_t *const *x_srcs, int W, int64_t n, uint8_t *q, float *scales,
                          uint16_t *out)
{
    if (n < 0 || n % BQO_BLOCK || W < 1) return -1;
    float y[BQO_BLOCK];
    for (int64_t b = 0; b < n / BQO_BLOCK; b++) {
        for (int i = 0; i < BQO_BLOCK; i++) {
            int64_t e = b * BQO_BLOCK + i;
            float a = bf16_bits_to_float(x_srcs[0][e]);
            for (int w = 1; w < W; w++) a = a + bf16_bits_to_float(x_srcs[w][e]);
            y[i] = bf16_bits_to_float(bqo_bf16_round((double)a));
        }
        quant_block_e4m3(y, q + b * BQO_BLOCK, scales + b);
    }
    if (out) bqo_dequant_e4m3(q, scales, n, out);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tiled E8M0 scale layout for block-scaled GEMM operands.                   */
/* The staged-input page mentions scale layouts for the GEMM ("[II] Support */
/* staged MXFP8 linear inputs", Behavior: empty_input allocates MXFP8       */
/* values and scale layouts) but prints none. This is the tiled layout that */
/* Blackwell block-scaled matrix multiplies read (cuBLAS, "1D block scaling */
/* factors layout"), stated from its public description. The tests pin it   */
/* to PyTorch's independent statements of that layout (to_blocked and       */
/* from_blocked in torch's quantized-test helpers) element by element.      */
/*                                                                          */
/* The scale matrix S [rows, g] (g = cols/32) is cut into tiles of 128 rows */
/* by 4 scale columns; tile (R, C) holds rows 128R..128R+127 and columns    */
/* 4C..4C+3 and occupies 512 bytes at offset (R * (g/4) + C) * 512. Inside  */
/* the tile, row r and column c sit at byte                                  */
/*     (r % 32) * 16 + (r / 32) * 4 + c      (r in 0..127, c in 0..3),       */
/* i.e. four interleaved 32-row panels: each 16-byte line holds one row of  */
/* every panel. Rows past `rows` in the last tile row are not written.       */
/* ------------------------------------------------------------------------ */

int64_t bqo_mx_tiled_scale_offset(int64_t row, int64_t gcol, int64_t g)
{
    int64_t R = row / 128, C = gcol / 4, r = row % 128, c = gcol % 4;
    return (R * (g / 4) + C) * 512 + (r % 32) * 16 + (r / 32) * 4 + c;
}

/* Row-major E8M0 [rows][ld_s] -> tiled; g = cols/32 must be a multiple of 4. */
int bqo_mx_scales_to_tiled(const uint8_t *s, int64_t rows, int64_t g, int64_t ld_s, uint8_t *tiled)
{
    if (rows < 0 || g < 0 || g % 4 || ld_s < g) return -1;
    for (int64_t row = 0; row < rows; row++)
        for (int64_t c = 0; c < g; c++) tiled[bqo_mx_tiled_scale_offset(row, c, g)] = s[row * ld_s + c];
    return 0;
}

/* Wire size of an n-element tensor in either codec: 132 bytes per 128 values. */
int64_t bqo_wire_bytes(int64_t n) { return n + 4 * (n / BQO_BLOCK); }
