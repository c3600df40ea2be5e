// pack.cu -- one-time rearrangement of Q8_0 blocks / Q4_K super-blocks into
// the library's packed layout (see qg_common.cuh). No value is changed: the
// int8 / 4-bit weights and fp16 scales reach the GEMMs bit for bit (the
// StartLux-Prism README, "Why StartLux-Prism": the released files run "as
// they are", with no conversion step). Not on the hot path.
#include "qg_common.cuh"

namespace qg {

// ------------------------------------------------------------------ Q8_0
__device__ __forceinline__ int8_t q8_val(const uint8_t* blocks, int64_t B, int64_t N, int64_t n,
                                         int64_t k) {
  if (n >= N) return 0;
  return (int8_t)blocks[(n * B + k / kBlk) * kQ8Bytes + 2 + (k % kBlk)];
}
__device__ __forceinline__ uint16_t q8_dbits(const uint8_t* blocks, int64_t B, int64_t N,
                                             int64_t n, int64_t b) {
  if (n >= N || b >= B) return 0;
  const uint8_t* p = blocks + (n * B + b) * kQ8Bytes;
  return (uint16_t)(p[0] | (p[1] << 8));
}

// Value sources of the decode stream and fp16 scale packers: Q8_0 blocks, or
// the fp16 copy and fp32 scales already written into a packed buffer (the
// MXFP4 conversion below writes those first).
struct Q8Src {
  const uint8_t* blocks;
  int64_t B, N;
  __device__ int8_t val(int64_t n, int64_t k) const { return q8_val(blocks, B, N, n, k); }
  __device__ uint16_t dbits(int64_t n, int64_t b) const { return q8_dbits(blocks, B, N, n, b); }
};
struct PackedSrc {
  const __half* q16;  // [N][K]
  const float* d32;   // [N][B4]
  int64_t B, B4, N, K;
  __device__ int8_t val(int64_t n, int64_t k) const {
    return n < N ? (int8_t)__half2int_rn(q16[n * K + k]) : (int8_t)0;
  }
  __device__ uint16_t dbits(int64_t n, int64_t b) const {
    return (n < N && b < B) ? __half_as_ushort(__float2half_rn(d32[n * B4 + b])) : (uint16_t)0;
  }
};

// one thread per (group g, block b, chunk t): 16 of the block's int8 values
// as signed bytes. Chunk t = 16*h + (r ^ 4h) holds q[16g+r][32b+16h ..
// +15]: the decode kernel's integer dot products read a row's 32 values as
// chunks (0, r) and (1, r); its 16-row fp16 MMA tiles read 8 bytes of rows
// r and r+8, and the XOR keeps those half-warp reads free of bank conflicts.
template <class Src>
__global__ void pack_q8_0_stream(const Src src, int64_t B, int64_t G, uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * B * 32) return;
  const int t = (int)(i % 32);
  const int64_t b = (i / 32) % B, g = i / 32 / B;
  const int h = t >> 4, r = (t & 15) ^ (h << 2);
  const int64_t n = 16 * g + r, k0 = 32 * b + 16 * h;
  uint32_t w[4];
  for (int x = 0; x < 4; ++x) {
    w[x] = 0;
    for (int e = 0; e < 4; ++e) w[x] |= (uint32_t)(uint8_t)src.val(n, k0 + 4 * x + e) << (8 * e);
  }
  reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

// one thread per (group g, block quad p, row r in 0..7)
template <class Src>
__global__ void pack_q8_0_dsc(const Src src, int64_t B4, int64_t G, uint16_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t P = B4 / 4;
  if (i >= G * P * 8) return;
  const int r = (int)(i % 8);
  const int64_t p = (i / 8) % P, g = i / 8 / P;
  for (int j = 0; j < 4; ++j) {
    out[i * 8 + j] = src.dbits(16 * g + r, 4 * p + j);
    out[i * 8 + 4 + j] = src.dbits(16 * g + r + 8, 4 * p + j);
  }
}

// one thread per (n, b4): fp16 copy of the block's 32 values and fp32 scale
__global__ void pack_q8_0_mma(const uint8_t* __restrict__ blocks, int64_t N, int64_t B,
                              int64_t B4, __half* __restrict__ q16, float* __restrict__ d32) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= N * B4) return;
  const int64_t b = i % B4, n = i / B4;
  d32[n * B4 + b] = __half2float(__ushort_as_half(q8_dbits(blocks, B, N, n, b)));
  if (b < B) {
    const int64_t K = B * kBlk;
    for (int j = 0; j < kBlk; ++j)
      q16[n * K + b * kBlk + j] = __int2half_rn(q8_val(blocks, B, N, n, b * kBlk + j));
  }
}

// ------------------------------------------------------------ MXFP4 weights
// (StartLux-Prism README, "Supported models and GPUs": --precision mxfp4 runs
// the MLP's projections in MXFP4 from a Q8_0 file, at lower precision.)
// Twice the E2M1 magnitude nearest to a >= 0 (an integer 0..12): the
// thresholds are the midpoints of 0, 0.5, 1, 1.5, 2, 3, 4, 6, a midpoint
// going to the neighbour whose mantissa bit is 0 (0, 1, 2, 4), and anything
// above 6 saturating at 6.
__device__ __forceinline__ int e2m1_twice(float a) {
  if (a > 5.0f) return 12;
  if (a >= 3.5f) return 8;
  if (a > 2.5f) return 6;
  if (a >= 1.75f) return 4;
  if (a > 1.25f) return 3;
  if (a >= 0.75f) return 2;
  if (a > 0.25f) return 1;
  return 0;
}

// one thread per (n, b4): the block's values w = d*q (exact in fp32), its
// shared exponent E = floor(log2 max|w|) - 2 + 127 (clamped to [0, 254]; an
// all-zero block takes 127), and each w / 2^(E-127) rounded to E2M1. The
// fp16 copy holds the integer 2v and the fp32 scale 2^(E-128), so the W8A8
// kernels compute with the weight 2v * 2^(E-128) = v * X exactly. A block
// whose 2^(E-128) lies outside fp16's range (the decode kernels' scales)
// sets the range bit of the error word.
__global__ void pack_mxfp4_mma(const uint8_t* __restrict__ blocks, int64_t N, int64_t B,
                               int64_t B4, __half* __restrict__ q16, float* __restrict__ d32,
                               uint32_t* err) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= N * B4) return;
  const int64_t b = i % B4, n = i / B4;
  if (b >= B) {
    d32[n * B4 + b] = 0.0f;
    return;
  }
  const uint8_t* p = blocks + (n * B + b) * kQ8Bytes;
  const float d = __half2float(__ushort_as_half((uint16_t)(p[0] | (p[1] << 8))));
  float w[kBlk];
  float amax = 0.0f;
  for (int j = 0; j < kBlk; ++j) {
    w[j] = d * (float)(int8_t)p[2 + j];  // exact: 11 x 8 significant bits
    amax = fmaxf(amax, fabsf(w[j]));
  }
  int e = 127;
  if (amax > 0.0f) {  // a normal fp32 (|w| >= 2^-24): floor(log2) from its exponent bits
    const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
    e = min(254, max(0, ex - 2 + 127));
  }
  const float inv = ldexpf(1.0f, 127 - e);  // 1 / X, a power of two
  const int64_t K = B * kBlk;
  for (int j = 0; j < kBlk; ++j) {
    const float r = w[j] * inv;  // exact: |r| >= 4/127 for w != 0
    const int c = e2m1_twice(fabsf(r));
    q16[n * K + b * kBlk + j] = __int2half_rn(r < 0.0f ? -c : c);
  }
  d32[n * B4 + b] = ldexpf(1.0f, e - 128);
  if (e - 128 < -24 || e - 128 > 15) set_error(err, kErrRange);
}

// ------------------------------------------------------------------ Q4_K
__device__ __forceinline__ int q4_nib(const uint8_t* sb, int64_t J, int64_t N, int64_t n,
                                      int64_t k) {
  if (n >= N) return 0;
  const uint8_t* p = sb + (n * J + k / kQ4kWeights) * kQ4kBytes;
  const int j = (int)(k % kQ4kWeights);
  const uint8_t byte = p[16 + j / 2];
  return (j & 1) ? (byte >> 4) : (byte & 0xF);
}

// 6-bit field f of the 96-bit little-endian string that starts at p
__device__ __forceinline__ int q4_field(const uint8_t* p, int f) {
  const int pos = 6 * f, byte = pos >> 3, sh = pos & 7;
  uint32_t v = p[byte];
  if (sh > 2) v |= (uint32_t)p[byte + 1] << 8;
  return (int)((v >> sh) & 63u);
}

// one thread per (group g, block b, row r): the row's 32 values of the block
// in 16 bytes, [g][b][r][16 B]. Word x (0..3) holds k = 32b + 8x .. 8x+7:
// byte e's low nibble is q[k = 32b + 8x + e], its high nibble q[32b + 8x + 4
// + e], so masking a word with 0x0F0F0F0F / 0xF0F0F0F0 gives four bytes that
// pair with four consecutive activation bytes in an integer dot product.
__global__ void pack_q4k_stream(const uint8_t* __restrict__ sb, int64_t N, int64_t J,
                                int64_t B, int64_t G, uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * B * 16) return;
  const int r = (int)(i % 16);
  const int64_t b = (i / 16) % B, g = i / 16 / B;
  const int64_t n = 16 * g + r;
  uint32_t w[4];
  for (int x = 0; x < 4; ++x) {
    w[x] = 0;
    for (int e = 0; e < 4; ++e) {
      const int64_t k = 32 * b + 8 * x + e;
      const uint32_t lo = (uint32_t)q4_nib(sb, J, N, n, k), hi = (uint32_t)q4_nib(sb, J, N, n, k + 4);
      w[x] |= (lo | (hi << 4)) << (8 * e);
    }
  }
  reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

// one thread per (group g, super-block j, row r in 0..15): a 16-byte header,
// [G][J][16 rows][16 B]: d and dmin (bytes 0-3, as in the super-block), then
// a 96-bit little-endian string of eight 12-bit units, unit i at bits [12i,
// 12i+12) = sc_i | m_i << 6, so that one funnel shift brings a sub-block's
// two fields together.
__global__ void pack_q4k_shdr(const uint8_t* __restrict__ sb, int64_t N, int64_t J, int64_t G,
                              uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * J * 16) return;
  const int r = (int)(i % 16);
  const int64_t j = (i / 16) % J, g = i / 16 / J;
  const int64_t n = 16 * g + r;
  uint8_t h[16] = {};
  if (n < N) {
    const uint8_t* p = sb + (n * J + j) * kQ4kBytes;
    for (int x = 0; x < 4; ++x) h[x] = p[x];
    uint64_t lo = 0;  // units 0..4 (bits 0..59) and the low 4 bits of unit 5
    uint32_t hi = 0;  // bits 64..95
    for (int u = 0; u < 8; ++u) {
      const uint64_t unit = (uint64_t)(q4_field(p + 4, u) | (q4_field(p + 4, 8 + u) << 6));
      const int pos = 12 * u;
      if (pos + 12 <= 64) {
        lo |= unit << pos;
      } else if (pos >= 64) {
        hi |= (uint32_t)(unit << (pos - 64));
      } else {
        lo |= unit << pos;
        hi |= (uint32_t)(unit >> (64 - pos));
      }
    }
    for (int x = 0; x < 8; ++x) h[4 + x] = (uint8_t)(lo >> (8 * x));
    for (int x = 0; x < 4; ++x) h[12 + x] = (uint8_t)(hi >> (8 * x));
  }
  for (int x = 0; x < 16; ++x) out[i * 16 + x] = h[x];
}

// one thread per (n, b): fp16 copy of the sub-block's 4-bit values, d*sc, dmin*m
__global__ void pack_q4k_mma(const uint8_t* __restrict__ sb, int64_t N, int64_t J, int64_t B,
                             __half* __restrict__ q16, float* __restrict__ ds32,
                             float* __restrict__ dm32) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= N * B) return;
  const int64_t b = i % B, n = i / B;
  const uint8_t* p = sb + (n * J + b / 8) * kQ4kBytes;
  const float d = __half2float(__ushort_as_half((uint16_t)(p[0] | (p[1] << 8))));
  const float dmin = __half2float(__ushort_as_half((uint16_t)(p[2] | (p[3] << 8))));
  const int sub = (int)(b % 8);
  ds32[n * B + b] = d * (float)q4_field(p + 4, sub);        // exact product
  dm32[n * B + b] = dmin * (float)q4_field(p + 4, 8 + sub); // exact product
  const int64_t K = B * kBlk;
  for (int j = 0; j < kBlk; ++j)
    q16[n * K + b * kBlk + j] = __int2half_rn(q4_nib(sb, J, N, n, b * kBlk + j));
}

static unsigned grid_for(int64_t n, int threads) { return (unsigned)ceil_div(n, threads); }

cudaError_t launch_pack_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                             cudaStream_t st) {
  const Q8Layout L(N, K);
  auto* base = reinterpret_cast<uint8_t*>(packed);
  const auto* in = reinterpret_cast<const uint8_t*>(blocks);
  const Q8Src src{in, L.B, N};
  pack_q8_0_stream<<<grid_for(L.G * L.B * 32, 256), 256, 0, st>>>(src, L.B, L.G,
                                                                    base + L.off_stream);
  pack_q8_0_dsc<<<grid_for(L.G * (L.B4 / 4) * 8, 256), 256, 0, st>>>(
      src, L.B4, L.G, reinterpret_cast<uint16_t*>(base + L.off_dsc));
  pack_q8_0_mma<<<grid_for(N * L.B4, 256), 256, 0, st>>>(
      in, N, L.B, L.B4, reinterpret_cast<__half*>(base + L.off_q16),
      reinterpret_cast<float*>(base + L.off_d32));
  return cudaGetLastError();
}

cudaError_t launch_pack_mxfp4_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                                   uint32_t* err, cudaStream_t st) {
  const Q8Layout L(N, K);
  auto* base = reinterpret_cast<uint8_t*>(packed);
  auto* q16 = reinterpret_cast<__half*>(base + L.off_q16);
  auto* d32 = reinterpret_cast<float*>(base + L.off_d32);
  pack_mxfp4_mma<<<grid_for(N * L.B4, 256), 256, 0, st>>>(
      reinterpret_cast<const uint8_t*>(blocks), N, L.B, L.B4, q16, d32, err);
  // the decode stream and fp16 scales from the sections just written
  const PackedSrc src{q16, d32, L.B, L.B4, N, K};
  pack_q8_0_stream<<<grid_for(L.G * L.B * 32, 256), 256, 0, st>>>(src, L.B, L.G,
                                                                    base + L.off_stream);
  pack_q8_0_dsc<<<grid_for(L.G * (L.B4 / 4) * 8, 256), 256, 0, st>>>(
      src, L.B4, L.G, reinterpret_cast<uint16_t*>(base + L.off_dsc));
  return cudaGetLastError();
}

cudaError_t launch_pack_q4k(const void* sblocks, int64_t N, int64_t K, void* packed,
                            cudaStream_t st) {
  const Q4kLayout L(N, K);
  auto* base = reinterpret_cast<uint8_t*>(packed);
  const auto* in = reinterpret_cast<const uint8_t*>(sblocks);
  pack_q4k_stream<<<grid_for(L.G * L.B * 16, 256), 256, 0, st>>>(in, N, L.J, L.B, L.G,
                                                                   base + L.off_stream);
  pack_q4k_shdr<<<grid_for(L.G * L.J * 16, 256), 256, 0, st>>>(in, N, L.J, L.G,
                                                                base + L.off_shdr);
  pack_q4k_mma<<<grid_for(N * L.B, 256), 256, 0, st>>>(
      in, N, L.J, L.B, reinterpret_cast<__half*>(base + L.off_q16),
      reinterpret_cast<float*>(base + L.off_ds32), reinterpret_cast<float*>(base + L.off_dm32));
  return cudaGetLastError();
}

}  // namespace qg
