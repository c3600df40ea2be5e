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

// one thread per (group g, block b, lane t): the 16 A-fragment bytes of the
// decode kernel's two fp16 MMAs for this block, stored biased (q + 128 as an
// unsigned byte) so that two byte permutes and one packed subtract turn four
// of them into exact fp16 values
__global__ void pack_q8_0_stream(const uint8_t* __restrict__ blocks, int64_t N, int64_t B,
                                 int64_t G, uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * B * 32) return;
  const int t = (int)(i % 32);
  const int64_t b = (i / 32) % B, g = i / 32 / B;
  const int r = t / 4, c = t % 4;
  const int64_t n0 = 16 * g + r, n1 = n0 + 8, k0 = 32 * b + 8 * c;
  uint8_t v[16];
  for (int j = 0; j < 4; ++j) {
    v[j] = (uint8_t)(q8_val(blocks, B, N, n0, k0 + j) + 128);
    v[4 + j] = (uint8_t)(q8_val(blocks, B, N, n1, k0 + j) + 128);
    v[8 + j] = (uint8_t)(q8_val(blocks, B, N, n0, k0 + 4 + j) + 128);
    v[12 + j] = (uint8_t)(q8_val(blocks, B, N, n1, k0 + 4 + j) + 128);
  }
  uint4 w;
  w.x = v[0] | (v[1] << 8) | (v[2] << 16) | ((uint32_t)v[3] << 24);
  w.y = v[4] | (v[5] << 8) | (v[6] << 16) | ((uint32_t)v[7] << 24);
  w.z = v[8] | (v[9] << 8) | (v[10] << 16) | ((uint32_t)v[11] << 24);
  w.w = v[12] | (v[13] << 8) | (v[14] << 16) | ((uint32_t)v[15] << 24);
  reinterpret_cast<uint4*>(out)[i] = w;
}

// one thread per (group g, block quad p, row r in 0..7)
__global__ void pack_q8_0_dsc(const uint8_t* __restrict__ blocks, int64_t N, int64_t B,
                              int64_t B4, int64_t G, uint16_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t P = B4 / 4;
  if (i >= G * P * 8) return;
  const int r = (int)(i % 8);
  const int64_t p = (i / 8) % P, g = i / 8 / P;
  for (int j = 0; j < 4; ++j) {
    out[i * 8 + j] = q8_dbits(blocks, B, N, 16 * g + r, 4 * p + j);
    out[i * 8 + 4 + j] = q8_dbits(blocks, B, N, 16 * g + r + 8, 4 * p + j);
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

// one thread per (group g, block b, lane t): two words of nibbles, one per
// 16-wide half h of the block's 32 k (k = 32b + 8c + 4h + j, j = 0..3): rows
// r and r+8 interleaved so that shift-and-mask yields fp16 pairs directly:
//   bits 0-3 q[r][j0], 16-19 q[r][j1], 4-7 q[r+8][j0], 20-23 q[r+8][j1],
//   8-11 q[r][j2], 24-27 q[r][j3], 12-15 q[r+8][j2], 28-31 q[r+8][j3]
__global__ void pack_q4k_stream(const uint8_t* __restrict__ sb, int64_t N, int64_t J,
                                int64_t B, int64_t G, uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * B * 32) return;
  const int t = (int)(i % 32);
  const int64_t b = (i / 32) % B, g = i / 32 / B;
  const int r = t / 4, c = t % 4;
  const int64_t n0 = 16 * g + r, n1 = n0 + 8;
  uint32_t w[2];
  for (int h = 0; h < 2; ++h) {
    const int64_t k = 32 * b + 8 * c + 4 * h;
    uint32_t a[4], e[4];
    for (int j = 0; j < 4; ++j) {
      a[j] = (uint32_t)q4_nib(sb, J, N, n0, k + j);
      e[j] = (uint32_t)q4_nib(sb, J, N, n1, k + j);
    }
    w[h] = a[0] | (a[1] << 16) | (e[0] << 4) | (e[1] << 20) | (a[2] << 8) | (a[3] << 24) |
           (e[2] << 12) | (e[3] << 28);
  }
  // [g][b/2][lane][16 B]: block 2p in bytes 0-7, block 2p+1 in bytes 8-15
  const int64_t off = (((g * (B / 2) + b / 2) * 32 + t) * 16) + (b & 1) * 8;
  *reinterpret_cast<uint2*>(out + off) = make_uint2(w[0], w[1]);
}

// one thread per (group g, super-block j, row r in 0..15): the 16-byte header
__global__ void pack_q4k_shdr(const uint8_t* __restrict__ sb, int64_t N, int64_t J, int64_t G,
                              uint8_t* __restrict__ out) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= G * J * 16) return;
  const int r = (int)(i % 16);
  const int64_t j = (i / 16) % J, g = i / 16 / J;
  const int64_t n = 16 * g + r;
  for (int x = 0; x < 16; ++x) out[i * 16 + x] = (n < N) ? sb[(n * J + j) * kQ4kBytes + x] : 0;
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
  pack_q8_0_stream<<<grid_for(L.G * L.B * 32, 256), 256, 0, st>>>(in, N, L.B, L.G,
                                                                    base + L.off_stream);
  pack_q8_0_dsc<<<grid_for(L.G * (L.B4 / 4) * 8, 256), 256, 0, st>>>(
      in, N, L.B, L.B4, L.G, reinterpret_cast<uint16_t*>(base + L.off_dsc));
  pack_q8_0_mma<<<grid_for(N * L.B4, 256), 256, 0, st>>>(
      in, N, L.B, L.B4, reinterpret_cast<__half*>(base + L.off_q16),
      reinterpret_cast<float*>(base + L.off_d32));
  return cudaGetLastError();
}

cudaError_t launch_pack_q4k(const void* sblocks, int64_t N, int64_t K, void* packed,
                            cudaStream_t st) {
  const Q4kLayout L(N, K);
  auto* base = reinterpret_cast<uint8_t*>(packed);
  const auto* in = reinterpret_cast<const uint8_t*>(sblocks);
  pack_q4k_stream<<<grid_for(L.G * L.B * 32, 256), 256, 0, st>>>(in, N, L.J, L.B, L.G,
                                                                   base + L.off_stream);
  pack_q4k_shdr<<<grid_for(L.G * L.J * 16, 256), 256, 0, st>>>(in, N, L.J, L.G,
                                                                base + L.off_shdr);
  pack_q4k_mma<<<grid_for(N * L.B, 256), 256, 0, st>>>(
      in, N, L.J, L.B, reinterpret_cast<__half*>(base + L.off_q16),
      reinterpret_cast<float*>(base + L.off_ds32), reinterpret_cast<float*>(base + L.off_dm32));
  return cudaGetLastError();
}

}  // namespace qg
