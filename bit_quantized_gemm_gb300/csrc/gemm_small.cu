// gemm_small.cu -- decode (small-M) GEMMs that stream the packed weights once.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and a fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit" and "The released files as they
// are"; "How it works": int8 tensor cores with exact int32 sums).
//
// Design. For M <= 64 the layer is bound by reading the weights from HBM
// (1.0625 B/weight for Q8_0, 0.5625 B/weight for Q4_K). A CTA owns R groups
// of 16 weight rows and walks all K blocks in ascending order:
//   * one producer thread streams, per stage of 16 blocks, the row groups'
//     contiguous fragment-order weights and scales and the activation rows
//     into a shared-memory ring with 1-D bulk copies (cp.async.bulk +
//     mbarrier transaction counts), keeping tens of KB in flight per SM
//     with no registers tied up;
//   * each consumer warp owns one (row group, 8-token tile) pair: per block
//     one 16-byte shared load gives the A fragments of two m16n8k16 fp16
//     MMAs (biased int8 bytes widened to exact fp16 by byte permutes and one
//     packed subtract; Q4_K nibbles by shift-and-mask), one 8-byte load the
//     token fragment (int8 rows padded to 544 bytes: conflict-free), and the
//     two MMAs sum the block exactly in fp32 from zero (|sum| < 2^20). This
//     GPU runs legacy fp16 MMAs at 4x the rate of legacy int8 MMAs (which
//     are no faster than dp4a), so int8 values travel as fp16 here;
//   * acc = fmaf(isum, d, acc) (Q4_K: then fmaf(-asum, dmin*m, acc)) per
//     block in order with packed f32x2 FMAs -- the same chain as the prefill
//     kernel, so both paths give identical bits.
#include "qg_common.cuh"

namespace qg {

constexpr int kSBlk = 16;          // K blocks per pipeline stage
constexpr int kARow = 544;         // bytes per activation row in a stage (512 + 32 pad)

__device__ __forceinline__ void bulk_copy(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int R, int TT, bool kQ4K>
struct DecodeSmem {
  static constexpr int kWBytes = R * kSBlk * (kQ4K ? 256 : 512);  // weights per stage
  static constexpr int kSBytes = R * 512;                          // scales / headers
  static constexpr int kABytes = TT * 8 * kARow;                   // activation rows
  static constexpr int kBBytes = kQ4K ? TT * 8 * kSBlk * 4 : 0;    // block sums (W4A8)
  static constexpr int kStage = kWBytes + kSBytes + kABytes + kBBytes;
  static constexpr int kNst = (R == 1) ? 6 : 3;
  static constexpr int kBarOff = kNst * kStage;
  static constexpr int kTotal = kBarOff + 2 * kNst * 8;
};

struct DecodeArgs {
  const int8_t* qa;        // [M][K]
  const float* sa;         // [M]
  const int32_t* bsum;     // [M][B] (W4A8)
  const uint8_t* wstream;  // packed stream section
  const uint8_t* wscale;   // packed scale / header section
  void* out;
  int64_t ldo;
  int32_t* dbg;
  uint32_t* err;
  int M, K, N, G;
  int out_f32;
};

template <int R, int TT, bool kQ4K, bool kDebug>
__global__ void __launch_bounds__(32 * (1 + R * TT), 1) decode_gemm_kernel(const DecodeArgs a) {
  using L = DecodeSmem<R, TT, kQ4K>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + L::kNst;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.K / kBlk;
  const int B4 = (B + 3) & ~3;
  const int J = B / 8;
  const int nstages = (B + kSBlk - 1) / kSBlk;
  const int g0 = blockIdx.x * R;
  const int M = a.M;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], R * TT);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int st = 0;
    uint32_t ph = 0;
    for (int s = 0; s < nstages; ++s) {
      const int blk0 = s * kSBlk;
      const int nb = min(kSBlk, B - blk0);
      uint8_t* base = smem + st * L::kStage;
      uint32_t bytes = 0;
      int ngroups = 0;
      for (int r = 0; r < R; ++r)
        if (g0 + r < a.G) ++ngroups;
      if (!kQ4K)
        bytes = ngroups * (nb * 512 + ((nb + 3) / 4) * 128);
      else
        bytes = ngroups * (nb * 256 + (nb / 8) * 256);
      const int mrows = min(M, TT * 8);
      bytes += mrows * nb * 32;
      if (kQ4K) bytes += mrows * nb * 4;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&empty[st], ph ^ 1, a.err);
        if (ok) mbar_arrive_expect_tx(&full[st], bytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        for (int r = 0; r < ngroups; ++r) {
          const int64_t g = g0 + r;
          if (!kQ4K) {
            bulk_copy(base + r * kSBlk * 512, a.wstream + (g * B + blk0) * 512, nb * 512, &full[st]);
            bulk_copy(base + L::kWBytes + r * 512,
                      a.wscale + (g * (B4 / 4) + blk0 / 4) * 128, ((nb + 3) / 4) * 128, &full[st]);
          } else {
            bulk_copy(base + r * kSBlk * 256, a.wstream + (g * (B / 2) + blk0 / 2) * 512,
                      nb * 256, &full[st]);
            bulk_copy(base + L::kWBytes + r * 512, a.wscale + (g * J + blk0 / 8) * 256,
                      (nb / 8) * 256, &full[st]);
          }
        }
      }
      for (int m = lane; m < mrows; m += 32) {
        bulk_copy(base + L::kWBytes + L::kSBytes + m * kARow,
                  a.qa + (int64_t)m * a.K + (int64_t)blk0 * kBlk, nb * 32, &full[st]);
        if (kQ4K)
          bulk_copy(base + L::kWBytes + L::kSBytes + L::kABytes + m * (kSBlk * 4),
                    a.bsum + (int64_t)m * B + blk0, nb * 4, &full[st]);
      }
      if (++st == L::kNst) { st = 0; ph ^= 1; }
    }
    // drain: every stage released before the CTA exits
    if (lane == 0) {
      for (int i = 0; i < L::kNst; ++i) {
        if (!mbar_wait(&empty[st], ph ^ 1, a.err)) break;
        if (++st == L::kNst) { st = 0; ph ^= 1; }
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int r = cw / TT, t = cw % TT;
  const int64_t g = g0 + r;
  const bool gvalid = g < a.G;
  const int gr = lane >> 2, c = lane & 3;
  const int n0 = (int)(16 * g + gr), n1 = n0 + 8;
  const int mrow = 8 * t + gr;                 // token of this lane's B fragment
  const int mc0 = 8 * t + 2 * c, mc1 = mc0 + 1;  // tokens of this lane's accumulators
  const bool tile_live = gvalid && (8 * t < M);
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

  float2 acc0 = make_float2(0.f, 0.f);  // row n0: tokens mc0, mc1
  float2 acc1 = make_float2(0.f, 0.f);  // row n1: tokens mc0, mc1

  int st = 0;
  uint32_t ph = 0;
  for (int s = 0; s < nstages; ++s) {
    const int blk0 = s * kSBlk;
    const int nb = min(kSBlk, B - blk0);
    if (!mbar_wait(&full[st], ph, a.err)) break;
    const uint8_t* base = smem + st * L::kStage;
    if (tile_live) {
      const uint8_t* wb = base + r * kSBlk * (kQ4K ? 256 : 512);
      const uint8_t* sb = base + L::kWBytes + r * 512;
      const uint8_t* ab = base + L::kWBytes + L::kSBytes + mrow * kARow + c * 8;
      const int32_t* bb = reinterpret_cast<const int32_t*>(base + L::kWBytes + L::kSBytes + L::kABytes);
      // blocks in groups of kG (a quad of Q8_0 scales / one Q4_K super-block),
      // each group fully unrolled so per-group scale arrays stay in registers
      constexpr int kG = kQ4K ? 8 : 4;
      for (int j0 = 0; j0 < nb; j0 += kG) {
        float dA[kG], dB[kG], mA[kG], mB[kG];
        if (!kQ4K) {
          const uint4 sc = *reinterpret_cast<const uint4*>(sb + (j0 >> 2) * 128 + gr * 16);
          const __half2* h = reinterpret_cast<const __half2*>(&sc);
          const float2 f0 = __half22float2(h[0]), f1 = __half22float2(h[1]);
          const float2 f2 = __half22float2(h[2]), f3 = __half22float2(h[3]);
          dA[0] = f0.x; dA[1] = f0.y; dA[2] = f1.x; dA[3] = f1.y;
          dB[0] = f2.x; dB[1] = f2.y; dB[2] = f3.x; dB[3] = f3.y;
        } else {
          const uint4 H0 = *reinterpret_cast<const uint4*>(sb + (j0 >> 3) * 256 + gr * 16);
          const uint4 H1 = *reinterpret_cast<const uint4*>(sb + (j0 >> 3) * 256 + (gr + 8) * 16);
          // 6-bit fields: a 96-bit string in words y, z, w (bytes 4..15)
          auto field = [](const uint4& H, int f) -> float {
            const uint64_t lo = (uint64_t)H.y | ((uint64_t)H.z << 32);
            const int pos = 6 * f;
            uint32_t v;
            if (pos + 6 <= 64) v = (uint32_t)(lo >> pos);
            else if (pos >= 64) v = H.w >> (pos - 64);
            else v = (uint32_t)(lo >> pos) | (H.w << (64 - pos));
            return (float)(v & 63u);
          };
          const float2 dd0 = __half22float2(*reinterpret_cast<const __half2*>(&H0.x));
          const float2 dd1 = __half22float2(*reinterpret_cast<const __half2*>(&H1.x));
#pragma unroll
          for (int u = 0; u < kG; ++u) {
            dA[u] = dd0.x * field(H0, u);   // exact products
            dB[u] = dd1.x * field(H1, u);
            mA[u] = -(dd0.y * field(H0, 8 + u));
            mB[u] = -(dd1.y * field(H1, 8 + u));
          }
        }
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const int j = j0 + u;
          if (j >= nb) break;
          // A fragments for the block's two 16-wide halves h = 0, 1
          uint32_t a0[4], a1[4];
          if (!kQ4K) {
            const uint4 w = *reinterpret_cast<const uint4*>(wb + j * 512 + lane * 16);
            // x: row n0 k 8c..+3, y: row n1 k 8c..+3, z: n0 k 8c+4..+7, w: n1 k 8c+4..+7
            biased_u8x4_to_f16x4(w.x, a0[0], a0[2]);
            biased_u8x4_to_f16x4(w.y, a0[1], a0[3]);
            biased_u8x4_to_f16x4(w.z, a1[0], a1[2]);
            biased_u8x4_to_f16x4(w.w, a1[1], a1[3]);
          } else {
            const uint2 w =
                *reinterpret_cast<const uint2*>(wb + (j >> 1) * 512 + lane * 16 + (j & 1) * 8);
            a0[0] = nib_pair_to_f16x2<0>(w.x);
            a0[1] = nib_pair_to_f16x2<4>(w.x);
            a0[2] = nib_pair_to_f16x2<8>(w.x);
            a0[3] = nib_pair_to_f16x2<12>(w.x);
            a1[0] = nib_pair_to_f16x2<0>(w.y);
            a1[1] = nib_pair_to_f16x2<4>(w.y);
            a1[2] = nib_pair_to_f16x2<8>(w.y);
            a1[3] = nib_pair_to_f16x2<12>(w.y);
          }
          uint32_t b00 = 0, b01 = 0, b10 = 0, b11 = 0;  // token k 8c+0..1, +2..3, +4..5, +6..7
          if (mrow < M) {
            const uint2 bv = *reinterpret_cast<const uint2*>(ab + j * 32);
            biased_u8x4_to_f16x4(bv.x ^ 0x80808080u, b00, b01);
            biased_u8x4_to_f16x4(bv.y ^ 0x80808080u, b10, b11);
          }
          float d[4];
          mma_f16_16816(d, a0, b00, b01, zero4);
          mma_f16_16816(d, a1, b10, b11, d);
          // d[0]: (n0, mc0), d[1]: (n0, mc1), d[2]: (n1, mc0), d[3]: (n1, mc1), exact
          if (kDebug) {
            const int b = blk0 + j;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int m = (i & 1) ? mc1 : mc0, n = (i < 2) ? n0 : n1;
              if (m < M && n < a.N) a.dbg[((int64_t)m * a.N + n) * B + b] = __float2int_rn(d[i]);
            }
          }
          acc0 = __ffma2_rn(make_float2(d[0], d[1]), make_float2(dA[u], dA[u]), acc0);
          acc1 = __ffma2_rn(make_float2(d[2], d[3]), make_float2(dB[u], dB[u]), acc1);
          if (kQ4K) {
            const float as0 = (mc0 < M) ? (float)bb[mc0 * kSBlk + j] : 0.f;
            const float as1 = (mc1 < M) ? (float)bb[mc1 * kSBlk + j] : 0.f;
            const float2 as = make_float2(as0, as1);
            acc0 = __ffma2_rn(as, make_float2(mA[u], mA[u]), acc0);
            acc1 = __ffma2_rn(as, make_float2(mB[u], mB[u]), acc1);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (++st == L::kNst) { st = 0; ph ^= 1; }
  }

  if (kDebug || !tile_live) return;
  const float accs[4] = {acc0.x, acc0.y, acc1.x, acc1.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = (i & 1) ? mc1 : mc0, n = (i < 2) ? n0 : n1;
    if (m < M && n < a.N) {
      const float y = accs[i] * __ldg(a.sa + m);
      if (a.out_f32)
        reinterpret_cast<float*>(a.out)[(int64_t)m * a.ldo + n] = y;
      else
        reinterpret_cast<uint16_t*>(a.out)[(int64_t)m * a.ldo + n] = f32_to_bf16_rne(y);
    }
  }
}

template <int R, int TT, bool kQ4K, bool kDebug>
static cudaError_t launch_decode_cfg(const DecodeArgs& a, cudaStream_t st) {
  using L = DecodeSmem<R, TT, kQ4K>;
  auto kern = decode_gemm_kernel<R, TT, kQ4K, kDebug>;
  static bool configured = false;  // once per process (idempotent if raced)
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((unsigned)ceil_div(a.G, R)), block(32 * (1 + R * TT));
  kern<<<grid, block, L::kTotal, st>>>(a);
  return cudaGetLastError();
}

template <bool kQ4K, bool kDebug>
static cudaError_t launch_decode_m(const DecodeArgs& a, cudaStream_t st) {
  if (a.M <= 8) return launch_decode_cfg<1, 1, kQ4K, kDebug>(a, st);
  if (a.M <= 16) return launch_decode_cfg<1, 2, kQ4K, kDebug>(a, st);
  if (a.M <= 32) return launch_decode_cfg<2, 4, kQ4K, kDebug>(a, st);
  return launch_decode_cfg<2, 8, kQ4K, kDebug>(a, st);
}

cudaError_t launch_decode_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                               const void* packed, int64_t N, void* out, bool out_f32,
                               int64_t ldo, int32_t* dbg, uint32_t* err, cudaStream_t st) {
  const Q8Layout Lq(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  DecodeArgs a{};
  a.qa = qa; a.sa = sa; a.bsum = nullptr;
  a.wstream = base + Lq.off_stream;
  a.wscale = base + Lq.off_dsc;
  a.out = out; a.ldo = ldo; a.dbg = dbg; a.err = err;
  a.M = (int)M; a.K = (int)K; a.N = (int)N; a.G = (int)Lq.G;
  a.out_f32 = out_f32 ? 1 : 0;
  return dbg ? launch_decode_m<false, true>(a, st) : launch_decode_m<false, false>(a, st);
}

cudaError_t launch_decode_q4k(const int8_t* qa, const float* sa, const int32_t* asum, int64_t M,
                              int64_t K, const void* packed, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int32_t* dbg, uint32_t* err, cudaStream_t st) {
  const Q4kLayout Lq(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  DecodeArgs a{};
  a.qa = qa; a.sa = sa; a.bsum = asum;
  a.wstream = base + Lq.off_stream;
  a.wscale = base + Lq.off_shdr;
  a.out = out; a.ldo = ldo; a.dbg = dbg; a.err = err;
  a.M = (int)M; a.K = (int)K; a.N = (int)N; a.G = (int)Lq.G;
  a.out_f32 = out_f32 ? 1 : 0;
  return dbg ? launch_decode_m<true, true>(a, st) : launch_decode_m<true, false>(a, st);
}

}  // namespace qg
