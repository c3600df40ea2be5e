/*
 * oracle.c -- plain CPU oracle (test infrastructure only; see oracle.h).
 *
 * Written for a reader checking it against the StartLux-Prism README
 * ("Why StartLux-Prism": "Reproducible to the bit", "The released files as
 * they are"; "How it works": int8 tensor cores with exact int32 sums) and the
 * readings listed in oracle.h. No blocking, fusion or reordering: every loop
 * is the definition written out. Build with -ffp-contract=off so that the only
 * fused multiply-adds are the explicit fmaf calls.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QBLK 32   /* weights per Q8_0 block and per Q4_K sub-block */
#define Q8_0_BYTES 34
#define Q4K_WEIGHTS 256
#define Q4K_BYTES 144

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  float v;
  if (e == 0) {
    v = ldexpf((float)f, -24);               /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexpf((float)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round to nearest, ties to even, on the 16 dropped low bits. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
    return (uint16_t)((u >> 16) | 0x40);     /* keep NaN a quiet NaN */
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
    upper += 1;                               /* carries into the exponent correctly */
  return (uint16_t)upper;
}

/* ---------------------------------------------------------------------- */
/* Per-token activation quantization                                       */
/* ---------------------------------------------------------------------- */
void orc_quantize_act(const void* x, int x_is_bf16, int64_t M, int64_t K,
                      int8_t* q, float* s, int32_t* bsum) {
  for (int64_t m = 0; m < M; ++m) {
    /* absmax over the row */
    float absmax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float v = x_is_bf16 ? orc_bf16_to_f32(((const uint16_t*)x)[m * K + k])
                          : ((const float*)x)[m * K + k];
      float a = fabsf(v);
      if (a > absmax) absmax = a;
    }
    float scale = absmax / 127.0f;            /* one correctly rounded division */
    s[m] = scale;
    for (int64_t k = 0; k < K; ++k) {
      float v = x_is_bf16 ? orc_bf16_to_f32(((const uint16_t*)x)[m * K + k])
                          : ((const float*)x)[m * K + k];
      int qi = 0;
      if (absmax != 0.0f) {
        float r = rintf(v / scale);           /* IEEE division, then ties-to-even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        qi = (int)r;
      }
      q[m * K + k] = (int8_t)qi;
    }
    if (bsum) {
      int64_t B = K / QBLK;
      for (int64_t b = 0; b < B; ++b) {
        int32_t acc = 0;
        for (int j = 0; j < QBLK; ++j) acc += q[m * K + b * QBLK + j];
        bsum[m * B + b] = acc;
      }
    }
  }
}

void orc_quantize_act_static(const void* x, int x_is_bf16, int64_t M, int64_t K,
                             const float* s_in, int64_t s_stride, int8_t* q, int32_t* bsum) {
  for (int64_t m = 0; m < M; ++m) {
    float scale = s_in[m * s_stride];
    for (int64_t k = 0; k < K; ++k) {
      float v = x_is_bf16 ? orc_bf16_to_f32(((const uint16_t*)x)[m * K + k])
                          : ((const float*)x)[m * K + k];
      int qi = 0;
      if (scale != 0.0f) {
        float r = rintf(v / scale);           /* IEEE division, then ties-to-even */
        if (r > 127.0f) r = 127.0f;           /* saturate outside the calibrated range */
        if (r < -127.0f) r = -127.0f;
        qi = (int)r;
      }
      q[m * K + k] = (int8_t)qi;
    }
    if (bsum) {
      int64_t B = K / QBLK;
      for (int64_t b = 0; b < B; ++b) {
        int32_t acc = 0;
        for (int j = 0; j < QBLK; ++j) acc += q[m * K + b * QBLK + j];
        bsum[m * B + b] = acc;
      }
    }
  }
}

/* ---------------------------------------------------------------------- */
/* W8A8, Q8_0 weights                                                      */
/* ---------------------------------------------------------------------- */
static const uint8_t* q8_0_block(const uint8_t* blocks, int64_t B, int64_t n, int64_t b) {
  return blocks + (n * B + b) * Q8_0_BYTES;
}

static float q8_0_scale(const uint8_t* blk) {
  uint16_t h = (uint16_t)(blk[0] | (blk[1] << 8));
  return orc_f16_to_f32(h);
}

static int32_t q8_0_isum(const int8_t* qa_row, const uint8_t* blk, int64_t b) {
  const int8_t* qw = (const int8_t*)(blk + 2);
  int32_t acc = 0;
  for (int j = 0; j < QBLK; ++j) acc += (int32_t)qa_row[b * QBLK + j] * (int32_t)qw[j];
  return acc;
}

void orc_block_sums_q8_0(const int8_t* qa, int64_t M, int64_t K,
                         const uint8_t* blocks, int64_t N, int32_t* isum) {
  int64_t B = K / QBLK;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t b = 0; b < B; ++b)
        isum[(m * N + n) * B + b] = q8_0_isum(qa + m * K, q8_0_block(blocks, B, n, b), b);
}

void orc_gemm_w8a8_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                        const uint8_t* blocks, int64_t N, float* y, uint16_t* out) {
  int64_t B = K / QBLK;
  for (int64_t m = 0; m < M; ++m) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      for (int64_t b = 0; b < B; ++b) {          /* ascending K blocks */
        const uint8_t* blk = q8_0_block(blocks, B, n, b);
        int32_t is = q8_0_isum(qa + m * K, blk, b);  /* exact */
        acc = fmaf((float)is, q8_0_scale(blk), acc);
      }
      float v = acc * sa[m];
      if (y) y[m * N + n] = v;
      if (out) out[m * N + n] = orc_f32_to_bf16(v);
    }
  }
}

/* ---------------------------------------------------------------------- */
/* W4A8, Q4_K weights                                                      */
/* ---------------------------------------------------------------------- */
static int q4k_field(const uint8_t* sb, int f) {
  /* bits [6f, 6f+6) of the 96-bit little-endian string at bytes 4..15 */
  int v = 0;
  for (int bit = 0; bit < 6; ++bit) {
    int pos = 6 * f + bit;
    int byte = sb[4 + pos / 8];
    v |= ((byte >> (pos % 8)) & 1) << bit;
  }
  return v;
}

static int q4k_nibble(const uint8_t* sb, int j) {
  int byte = sb[16 + j / 2];
  return (j % 2 == 0) ? (byte & 0xf) : (byte >> 4);
}

void orc_q4k_decode(const uint8_t* sb, double* w, float* d, float* dmin,
                    uint8_t* sc, uint8_t* mn, uint8_t* q) {
  float dd = orc_f16_to_f32((uint16_t)(sb[0] | (sb[1] << 8)));
  float dm = orc_f16_to_f32((uint16_t)(sb[2] | (sb[3] << 8)));
  if (d) *d = dd;
  if (dmin) *dmin = dm;
  for (int i = 0; i < 8; ++i) {
    int s_i = q4k_field(sb, i), m_i = q4k_field(sb, 8 + i);
    if (sc) sc[i] = (uint8_t)s_i;
    if (mn) mn[i] = (uint8_t)m_i;
    for (int j = 0; j < QBLK; ++j) {
      int qq = q4k_nibble(sb, i * QBLK + j);
      if (q) q[i * QBLK + j] = (uint8_t)qq;
      if (w) w[i * QBLK + j] = (double)dd * s_i * qq - (double)dm * m_i;
    }
  }
}

void orc_block_sums_q4k(const int8_t* qa, int64_t M, int64_t K,
                        const uint8_t* sblocks, int64_t N, int32_t* isum, int32_t* asum) {
  int64_t B = K / QBLK, J = K / Q4K_WEIGHTS;
  for (int64_t m = 0; m < M; ++m) {
    if (asum)
      for (int64_t b = 0; b < B; ++b) {
        int32_t acc = 0;
        for (int j = 0; j < QBLK; ++j) acc += qa[m * K + b * QBLK + j];
        asum[m * B + b] = acc;
      }
    if (isum)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < B; ++b) {
          const uint8_t* sb = sblocks + (n * J + b / 8) * Q4K_BYTES;
          int i = (int)(b % 8);
          int32_t acc = 0;
          for (int j = 0; j < QBLK; ++j)
            acc += (int32_t)qa[m * K + b * QBLK + j] * q4k_nibble(sb, i * QBLK + j);
          isum[(m * N + n) * B + b] = acc;
        }
  }
}

void orc_gemm_w4a8_q4k(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                       const uint8_t* sblocks, int64_t N, float* y, uint16_t* out) {
  int64_t B = K / QBLK, J = K / Q4K_WEIGHTS;
  for (int64_t m = 0; m < M; ++m) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      for (int64_t b = 0; b < B; ++b) {          /* ascending sub-blocks */
        const uint8_t* sb = sblocks + (n * J + b / 8) * Q4K_BYTES;
        int i = (int)(b % 8);
        float d = orc_f16_to_f32((uint16_t)(sb[0] | (sb[1] << 8)));
        float dmin = orc_f16_to_f32((uint16_t)(sb[2] | (sb[3] << 8)));
        float ds = d * (float)q4k_field(sb, i);       /* exact product */
        float dm = dmin * (float)q4k_field(sb, 8 + i); /* exact product */
        int32_t is = 0, as = 0;
        for (int j = 0; j < QBLK; ++j) {
          int32_t a = qa[m * K + b * QBLK + j];
          is += a * q4k_nibble(sb, i * QBLK + j);
          as += a;
        }
        acc = fmaf((float)is, ds, acc);
        acc = fmaf(-(float)as, dm, acc);
      }
      float v = acc * sa[m];
      if (y) y[m * N + n] = v;
      if (out) out[m * N + n] = orc_f32_to_bf16(v);
    }
  }
}
