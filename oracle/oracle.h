/*
 * oracle.h -- plain, slow CPU oracle for the exact int8 (W8A8) and W4A8
 * quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's compute path may call,
 * link or load this code: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it. It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes follows the StartLux-Prism README:
 *   - "Why StartLux-Prism", bullet "Reproducible to the bit": int8 GEMMs sum
 *     exactly in int32, so results do not depend on batch composition;
 *   - "Why StartLux-Prism", bullet "The released files as they are": Q8_0
 *     weights run as int8 (W8A8) and Q4_K_M weights on their own 4-bit values
 *     (W4A8);
 *   - "How it works", bullet on int8 tensor cores with exact int32 sums.
 * The pages print no formula, byte layout, rounding rule or epilogue order;
 * the readings taken here are:
 *   - activations are quantized per token (row): s = absmax/127 (fp32,
 *     correctly rounded division), q = clamp(rint(x / s), -127, 127) with
 *     round-half-to-even; an all-zero row has s = 0 and q = 0;
 *   - Q8_0 block = {fp16 d; int8 q[32]} (34 bytes), weight = d * q;
 *   - per 32-wide K block b the integer sum isum = sum q_a * q_w is exact;
 *     the fp32 epilogue is one fused multiply-add per block in ascending b,
 *     acc = fmaf((float)isum, d_b, acc), then y = acc * s_a, then bf16
 *     round-to-nearest-even;
 *   - Q4_K super-block = 256 weights in 8 sub-blocks of 32 with 6-bit scale
 *     sc_i and 6-bit min m_i, fp16 d and dmin, weight = d*sc_i*q - dmin*m_i,
 *     q in [0, 15]; per sub-block acc = fmaf((float)isum, d*sc_i, acc) then
 *     acc = fmaf(-(float)asum, dmin*m_i, acc), asum = sum of q_a over the
 *     sub-block.
 *
 * Byte layout of the 144-byte Q4_K super-block (this library's canonical
 * packing; the pages give none):
 *   bytes 0-1   d     (fp16, little endian)
 *   bytes 2-3   dmin  (fp16, little endian)
 *   bytes 4-15  a 96-bit little-endian bit string of sixteen 6-bit fields:
 *               field f occupies bits [6f, 6f+6); fields 0..7 are sc_0..sc_7,
 *               fields 8..15 are m_0..m_7
 *   bytes 16-143 nibbles: weight j of the super-block (0..255) is the low
 *               nibble of byte 16 + j/2 when j is even, the high nibble when
 *               j is odd.
 */
#ifndef QG_ORACLE_H
#define QG_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* IEEE 754 binary16 -> binary32, exact. */
float orc_f16_to_f32(uint16_t h);
/* binary32 -> bfloat16 bits, round to nearest, ties to even. */
uint16_t orc_f32_to_bf16(float f);
/* bfloat16 bits -> binary32, exact. */
float orc_bf16_to_f32(uint16_t b);

/* Per-token activation quantization.
 * x: [M][K] row-major, fp32 values (x_is_bf16 = 0) or bf16 bits (x_is_bf16 = 1).
 * q: [M][K] int8 out; s: [M] fp32 out; bsum: [M][K/32] int32 out or NULL.
 * K must be a multiple of 32 when bsum is not NULL. */
void orc_quantize_act(const void* x, int x_is_bf16, int64_t M, int64_t K,
                      int8_t* q, float* s, int32_t* bsum);

/* Activation quantization with given (calibrated) scales: row m uses
 * s = s_in[m * s_stride] (s_stride 0: one scale for every row);
 * q = clamp(rint(x / s), -127, 127) with the correctly rounded division,
 * q = 0 when s == 0. Values beyond the calibrated range saturate. */
void orc_quantize_act_static(const void* x, int x_is_bf16, int64_t M, int64_t K,
                             const float* s_in, int64_t s_stride, int8_t* q, int32_t* bsum);

/* W8A8 with Q8_0 weights.
 * qa: [M][K] int8, sa: [M] fp32, blocks: [N][K/32] x 34 bytes.
 * y: [M][N] fp32 out (the value before bf16 rounding) or NULL;
 * out: [M][N] bf16 bits out or NULL. */
void orc_gemm_w8a8_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                        const uint8_t* blocks, int64_t N, float* y, uint16_t* out);

/* Exact int32 block sums isum[m][n][b] for W8A8. */
void orc_block_sums_q8_0(const int8_t* qa, int64_t M, int64_t K,
                         const uint8_t* blocks, int64_t N, int32_t* isum);

/* Q4_K decode of one super-block into 256 weights as the pages define them,
 * in fp64 (exact: d*sc*q and dmin*m are exact products), plus the fields. */
void orc_q4k_decode(const uint8_t* sb, double* w, float* d, float* dmin,
                    uint8_t* sc, uint8_t* mn, uint8_t* q);

/* W4A8 with Q4_K weights.
 * qa: [M][K] int8, sa: [M] fp32, sblocks: [N][K/256] x 144 bytes. */
void orc_gemm_w4a8_q4k(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                       const uint8_t* sblocks, int64_t N, float* y, uint16_t* out);

/* Exact int32 sums for W4A8: isum[m][n][b] = sum q_a*q, asum[m][b] = sum q_a. */
void orc_block_sums_q4k(const int8_t* qa, int64_t M, int64_t K,
                        const uint8_t* sblocks, int64_t N, int32_t* isum, int32_t* asum);

/* Number of OpenMP threads the GEMM loops use (1 without OpenMP). */
int orc_num_threads(void);

/* MXFP4 weights from Q8_0 (README, "Supported models and GPUs" and "Blackwell
 * MXFP4": --precision mxfp4 runs the MLP's projections in MXFP4 from a Q8_0
 * file, at lower precision). The pages give no conversion rule; the reading
 * taken (the OCP microscaling format): 32-element blocks along K share an
 * 8-bit exponent E, scale X = 2^(E-127); elements are E2M1 codes (sign bit 3,
 * exponent bits 2..1 with bias 1, mantissa bit 0: magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6). For a block of Q8_0 values w = d*q: E = floor(log2(max|w|)) -
 * 2 + 127 (clamped to [0, 254]; an all-zero block takes E = 127), and each
 * w/X goes to the nearest E2M1 value, ties to the even mantissa, magnitudes
 * above 6 saturating at 6.
 * codes: [N][K] one code per weight (0..15); E: [N][K/32]. */
void orc_mxfp4_from_q8_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* codes,
                         uint8_t* E);
/* The value of an E2M1 code. */
double orc_e2m1_value(int code);
/* W4A8 with MXFP4 weights: per K block the exact sum isum = sum q_a * (2v)
 * (2v in -12..12, an integer), then acc = fmaf((float)isum, 2^(E-128), acc)
 * in ascending blocks, y = acc * s_a, bf16 round-to-nearest-even: the W8A8
 * chain with integer weights 2v and block scales X/2. */
void orc_gemm_w4a8_mxfp4(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                         const uint8_t* codes, const uint8_t* E, int64_t N, float* y,
                         uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
