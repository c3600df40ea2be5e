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

/* ---------------------------------------------------------------------- */
/* MXFP4 weights converted from Q8_0 (the README's "Blackwell MXFP4":    */
/* the MLP's projections in MXFP4 from a Q8_0 file, lower precision)     */
/* ---------------------------------------------------------------------- */
/* E2M1 element: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
double orc_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* nearest E2M1 code to v, ties to the even mantissa, magnitudes beyond 6
 * saturate to 6; a zero magnitude is code 0 */
static int e2m1_round(double v) {
  double a = fabs(v);
  int best = 0;
  double best_err = a;  /* code 0: magnitude 0 */
  for (int c = 1; c < 8; ++c) {
    double err = fabs(a - orc_e2m1_value(c));
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  if (best == 0) return 0;
  return (v < 0) ? (best | 8) : best;
}

void orc_mxfp4_from_q8_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* codes,
                         uint8_t* E) {
  int64_t B = K / QBLK;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < B; ++b) {
      const uint8_t* blk = q8_0_block(blocks, B, n, b);
      float d = q8_0_scale(blk);
      double w[QBLK], amax = 0.0;
      for (int j = 0; j < QBLK; ++j) {
        w[j] = (double)d * (double)(int8_t)blk[2 + j];  /* exact */
        if (fabs(w[j]) > amax) amax = fabs(w[j]);
      }
      int e = 127;  /* an all-zero block: X = 1 */
      if (amax > 0.0) {
        int p;
        frexp(amax, &p);         /* amax = f * 2^p, f in [0.5, 1) */
        e = (p - 1) - 2 + 127;   /* floor(log2(amax)) - emax(E2M1) + bias */
        if (e < 0) e = 0;
        if (e > 254) e = 254;
      }
      E[n * B + b] = (uint8_t)e;
      double X = ldexp(1.0, e - 127);
      for (int j = 0; j < QBLK; ++j) codes[n * K + b * QBLK + j] = (uint8_t)e2m1_round(w[j] / X);
    }
}

void orc_gemm_w4a8_mxfp4(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                         const uint8_t* codes, const uint8_t* E, int64_t N, float* y,
                         uint16_t* out) {
  int64_t B = K / QBLK;
  for (int64_t m = 0; m < M; ++m) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      for (int64_t b = 0; b < B; ++b) {  /* ascending K blocks */
        int32_t is = 0;                    /* exact: |2v| <= 12 */
        for (int j = 0; j < QBLK; ++j) {
          int c2 = (int)lrint(2.0 * orc_e2m1_value(codes[n * K + b * QBLK + j]));
          is += (int32_t)qa[m * K + b * QBLK + j] * c2;
        }
        /* weight = (2v) * X / 2: the block scale as an exact fp32 power of two */
        acc = fmaf((float)is, ldexpf(1.0f, (int)E[n * B + b] - 128), acc);
      }
      float v = acc * sa[m];
      if (y) y[m * N + n] = v;
      if (out) out[m * N + n] = orc_f32_to_bf16(v);
    }
  }
}
