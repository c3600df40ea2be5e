// gemm_small.cu -- decode (small-M) GEMMs that stream the packed weights once.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and a fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit" and "The released files as they
// are"; "How it works": int8 tensor cores with exact int32 sums).
//
// Design. For M <= 64 the layer is bound by reading the weights from HBM
// (1.0625 B/weight for Q8_0, 0.5625 B/weight for Q4_K). Each warp owns one
// group of 16 weight rows and walks all K blocks in ascending order:
//   * one 16-byte streaming load per lane per block brings that block's
//     A-fragment of an m16n8k32 int8 MMA (the packed layout stores the bytes
//     in register order; Q4_K nibbles are widened with two masks);
//   * the tokens are the MMA's 8-wide N side (T = ceil(M/8) MMAs per block),
//     read as 8-byte loads from the row-major int8 activations (L1/L2
//     resident);
//   * the MMA accumulates exactly in int32, starting from the bit pattern of
//     1.5*2^23 so that the result reads back as a float with one FADD;
//   * per (row, token) the epilogue applies acc = fmaf(isum, d, acc) (Q4_K:
//     then fmaf(-asum, dmin*m, acc)) in block order, the same chain as the
//     prefill kernel, so both paths give identical bits.
#include "qg_common.cuh"

namespace qg {

constexpr int kSmallWarps = 2;  // warps per CTA (one 16-row group each)
constexpr int kUnroll = 8;      // blocks of weights in flight per lane

template <int T, bool kQ4K, bool kDebug>
__global__ void __launch_bounds__(kSmallWarps * 32) decode_gemm_kernel(
    const int8_t* __restrict__ qa, const float* __restrict__ sa,
    const int32_t* __restrict__ asum_g, int M, int K, int N, int64_t G,
    const uint8_t* __restrict__ wstream, const uint8_t* __restrict__ wscale, void* __restrict__ out,
    int out_f32, int64_t ldo, int32_t* __restrict__ dbg) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = (int64_t)blockIdx.x * kSmallWarps + warp;
  if (g >= G) return;
  const int r = lane >> 2, c = lane & 3;
  const int n0 = (int)(16 * g + r), n1 = n0 + 8;
  const int B = K / kBlk;

  float acc[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

  const int magic4[4] = {kMagicBits, kMagicBits, kMagicBits, kMagicBits};

  // activation rows of this lane's B fragments: token 8t + r
  const int8_t* arow[T];
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const int m = 8 * t + r;
    arow[t] = (m < M) ? qa + (int64_t)m * K + 8 * c : nullptr;
  }

  // Q8_0: fragment stream [G][B][32][16]; scales [G][B4/4][8][16 B]
  // Q4_K: nibble stream [G][B/2][32][16]; headers [G][J][16][16 B]
  const int B4 = (B + 3) & ~3;

  for (int b0 = 0; b0 < B; b0 += kUnroll) {
    int4 wv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int b = b0 + u;
      if (!kQ4K) {
        if (b < B) wv[u] = ldg_stream(wstream + (((int64_t)g * B + b) * 32 + lane) * 16);
      } else if ((u & 1) == 0) {
        if (b < B) wv[u] = ldg_stream(wstream + (((int64_t)g * (B / 2) + b / 2) * 32 + lane) * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int b = b0 + u;
      if (b >= B) break;
      int a[4];
      float d0, d1, m0 = 0.f, m1 = 0.f;
      if (!kQ4K) {
        a[0] = wv[u].x; a[1] = wv[u].y; a[2] = wv[u].z; a[3] = wv[u].w;
        // fp16 scales of rows n0, n1 for this block
        const uint4 sc = __ldg(reinterpret_cast<const uint4*>(
            wscale + (((int64_t)g * (B4 / 4) + b / 4) * 8 + r) * 16));
        const uint32_t w0 = (b & 2) ? sc.y : sc.x;  // d[n0][4p..4p+3] in x, y
        const uint32_t w1 = (b & 2) ? sc.w : sc.z;  // d[n1][4p..4p+3] in z, w
        d0 = __half2float(__ushort_as_half((uint16_t)((b & 1) ? (w0 >> 16) : (w0 & 0xFFFF))));
        d1 = __half2float(__ushort_as_half((uint16_t)((b & 1) ? (w1 >> 16) : (w1 & 0xFFFF))));
      } else {
        const int4 v = wv[u & ~1];
        const uint32_t x0 = (u & 1) ? (uint32_t)v.z : (uint32_t)v.x;
        const uint32_t x1 = (u & 1) ? (uint32_t)v.w : (uint32_t)v.y;
        a[0] = (int)(x0 & 0x0F0F0F0Fu);
        a[1] = (int)((x0 >> 4) & 0x0F0F0F0Fu);
        a[2] = (int)(x1 & 0x0F0F0F0Fu);
        a[3] = (int)((x1 >> 4) & 0x0F0F0F0Fu);
        // headers of rows n0, n1 for super-block b/8
        const int J = B / 8;
        const uint8_t* h0 = wscale + (((int64_t)g * J + b / 8) * 16 + r) * 16;
        const uint8_t* h1 = h0 + 8 * 16;
        const uint4 H0 = __ldg(reinterpret_cast<const uint4*>(h0));
        const uint4 H1 = __ldg(reinterpret_cast<const uint4*>(h1));
        const int sub = b & 7;
        auto field = [](const uint4& H, int f) -> float {
          // 96-bit string in words y, z, w (bytes 4..15)
          const uint64_t lo = (uint64_t)H.y | ((uint64_t)H.z << 32);
          const int pos = 6 * f;
          uint32_t v;
          if (pos + 6 <= 64) v = (uint32_t)(lo >> pos);
          else if (pos >= 64) v = H.w >> (pos - 64);
          else v = (uint32_t)(lo >> pos) | (H.w << (64 - pos));
          return (float)(v & 63u);
        };
        const float dd0 = __half2float(__ushort_as_half((uint16_t)(H0.x & 0xFFFF)));
        const float dm0 = __half2float(__ushort_as_half((uint16_t)(H0.x >> 16)));
        const float dd1 = __half2float(__ushort_as_half((uint16_t)(H1.x & 0xFFFF)));
        const float dm1 = __half2float(__ushort_as_half((uint16_t)(H1.x >> 16)));
        d0 = dd0 * field(H0, sub);       // exact products
        d1 = dd1 * field(H1, sub);
        m0 = dm0 * field(H0, 8 + sub);
        m1 = dm1 * field(H1, 8 + sub);
      }
#pragma unroll
      for (int t = 0; t < T; ++t) {
        int2 bb = make_int2(0, 0);
        if (arow[t]) bb = __ldg(reinterpret_cast<const int2*>(arow[t] + (int64_t)b * kBlk));
        int d[4];
        mma_s8_16832(d, a, bb.x, bb.y, magic4);
        // d[0]: (n0, token 8t+2c), d[1]: (n0, 8t+2c+1), d[2]: (n1, 8t+2c), d[3]: (n1, 8t+2c+1)
        const int mt0 = 8 * t + 2 * c;
        if (kDebug) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int m = mt0 + (i & 1), n = (i < 2) ? n0 : n1;
            if (m < M && n < N) dbg[((int64_t)m * N + n) * B + b] = d[i] - kMagicBits;
          }
        }
        if (!kQ4K) {
          acc[t][0] = fmaf(magic_to_float(d[0]), d0, acc[t][0]);
          acc[t][1] = fmaf(magic_to_float(d[1]), d0, acc[t][1]);
          acc[t][2] = fmaf(magic_to_float(d[2]), d1, acc[t][2]);
          acc[t][3] = fmaf(magic_to_float(d[3]), d1, acc[t][3]);
        } else {
          float as0 = 0.f, as1 = 0.f;
          if (mt0 < M) as0 = (float)__ldg(asum_g + (int64_t)mt0 * B + b);
          if (mt0 + 1 < M) as1 = (float)__ldg(asum_g + (int64_t)(mt0 + 1) * B + b);
          acc[t][0] = fmaf(-as0, m0, fmaf(magic_to_float(d[0]), d0, acc[t][0]));
          acc[t][1] = fmaf(-as1, m0, fmaf(magic_to_float(d[1]), d0, acc[t][1]));
          acc[t][2] = fmaf(-as0, m1, fmaf(magic_to_float(d[2]), d1, acc[t][2]));
          acc[t][3] = fmaf(-as1, m1, fmaf(magic_to_float(d[3]), d1, acc[t][3]));
        }
      }
    }
  }

  if (kDebug) return;
#pragma unroll
  for (int t = 0; t < T; ++t) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = 8 * t + 2 * c + (i & 1), n = (i < 2) ? n0 : n1;
      if (m < M && n < N) {
        const float y = acc[t][i] * __ldg(sa + m);
        if (out_f32)
          reinterpret_cast<float*>(out)[(int64_t)m * ldo + n] = y;
        else
          reinterpret_cast<uint16_t*>(out)[(int64_t)m * ldo + n] = f32_to_bf16_rne(y);
      }
    }
  }
}

template <bool kQ4K, bool kDebug>
static cudaError_t launch_decode_t(int T, const int8_t* qa, const float* sa, const int32_t* asum,
                                   int M, int K, int N, int64_t G, const uint8_t* ws,
                                   const uint8_t* wsc, void* out, int out_f32, int64_t ldo,
                                   int32_t* dbg, cudaStream_t st) {
  dim3 grid((unsigned)ceil_div(G, kSmallWarps)), block(kSmallWarps * 32);
#define QG_DECODE_CASE(TT)                                                                  \
  case TT:                                                                                  \
    decode_gemm_kernel<TT, kQ4K, kDebug><<<grid, block, 0, st>>>(qa, sa, asum, M, K, N, G, \
                                                                 ws, wsc, out, out_f32, ldo, \
                                                                 dbg);                      \
    break;
  switch (T) {
    QG_DECODE_CASE(1)
    QG_DECODE_CASE(2)
    QG_DECODE_CASE(4)
    QG_DECODE_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef QG_DECODE_CASE
  return cudaGetLastError();
}

static int token_tiles(int M) {
  const int t = (M + 7) / 8;
  return t <= 1 ? 1 : t <= 2 ? 2 : t <= 4 ? 4 : 8;
}

cudaError_t launch_decode_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                               const void* packed, int64_t N, void* out, bool out_f32,
                               int64_t ldo, int32_t* dbg, cudaStream_t st) {
  const Q8Layout L(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  const int T = token_tiles((int)M);
  if (dbg)
    return launch_decode_t<false, true>(T, qa, sa, nullptr, (int)M, (int)K, (int)N, L.G,
                                        base + L.off_stream, base + L.off_dsc, out, out_f32, ldo,
                                        dbg, st);
  return launch_decode_t<false, false>(T, qa, sa, nullptr, (int)M, (int)K, (int)N, L.G,
                                       base + L.off_stream, base + L.off_dsc, out, out_f32, ldo,
                                       nullptr, st);
}

cudaError_t launch_decode_q4k(const int8_t* qa, const float* sa, const int32_t* asum, int64_t M,
                              int64_t K, const void* packed, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int32_t* dbg, cudaStream_t st) {
  const Q4kLayout L(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  const int T = token_tiles((int)M);
  if (dbg)
    return launch_decode_t<true, true>(T, qa, sa, asum, (int)M, (int)K, (int)N, L.G,
                                       base + L.off_stream, base + L.off_shdr, out, out_f32, ldo,
                                       dbg, st);
  return launch_decode_t<true, false>(T, qa, sa, asum, (int)M, (int)K, (int)N, L.G,
                                      base + L.off_stream, base + L.off_shdr, out, out_f32, ldo,
                                      nullptr, st);
}

}  // namespace qg
