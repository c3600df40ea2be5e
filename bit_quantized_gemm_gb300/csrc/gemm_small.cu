// gemm_small.cu -- decode (small-M) GEMMs that stream the packed weights once.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and a fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit" and "The released files as they
// are"; "How it works": int8 tensor cores with exact int32 sums).
//
// Design. For M <= 16 the layer is bound by reading the weights from HBM
// (1.0625 B/weight for Q8_0, 0.5625 B/weight for Q4_K). A CTA owns one group
// of 16 weight rows and all of K; K is cut into stages of 16 or 32 blocks.
// Two kernels share that frame:
//   * warp 0 (one thread) streams each stage into a shared-memory ring -- the
//     group's contiguous weights and scales with 1-D bulk copies
//     (cp.async.bulk), the stage's slice of every activation row (and for
//     W4A8 of every block-sum row) as one 2-D TMA box -- with mbarrier
//     transaction counts;
//   * warps 1..8 compute the stage's exact block sums into a shared stash:
//     - up to 4 rows, decode_dp4a_kernel: one lane per
//       weight row and block, eight dp4a per token on the row's 32 int8
//       values (W4A8: its 32 nibbles masked into low and high bytes), no
//       widening; the W4A8 lane also decodes its row's d*sc and dmin*m;
//     - more rows, decode_gemm_kernel: one legacy int8 m16n8k32 MMA per
//       block and 8-token tile on the stored bytes (nibbles masked into
//       unsigned bytes). That MMA runs at a quarter of the legacy fp16 rate,
//       but 16 rows need only ~18 us of it for a 5120 x 17408 matrix, and
//       nothing is widened (the fp16-MMA variant, which widens weights and
//       activations in registers, is kept behind a build switch); every sum
//       is below 2^20, exact in int32 and in fp32;
//     and once a warp has read the stage (and copied into the stash what the
//     chain needs from it: Q8_0 scales, MMA tiles' Q4_K block sums) it hands
//     its part of the stage back to the producer;
//   * warp 9 applies acc = fmaf(isum, d, acc) (Q4_K: then
//     fmaf(-asum, dmin*m, acc)) over the stage's blocks in ascending order
//     with packed f32x2 FMAs -- the same chain as the prefill kernel, so both
//     paths give identical bits -- reading the stash alone.
// K-parallel compute with a sequential fp32 chain keeps ten warps busy per
// 16-row group, which small N (few groups) needs to reach HBM rate.
// As the GEMM of the layer call the kernel is a programmatic dependent of the
// quantize kernel: it starts while the rows are quantized, requests its first
// weight stages, and copies activations only once the quantize grid is done.
#include <cuda.h>

#include <cstring>

#include "qg_common.cuh"

namespace qg {

// from gemm_large.cu: rows of row_bytes bytes as 8-byte words, box_words x box_rows
bool make_tmap_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                    uint32_t box_words, uint32_t box_rows);

constexpr int kCompWarps = 8;      // compute warps per CTA

// 5..16 rows: block sums by the legacy int8 MMA on the stored bytes (1) or by
// fp16 MMAs on weights and activations widened in registers (0)
#ifndef QG_DEC_IMMA
#define QG_DEC_IMMA 1
#endif

// K blocks per pipeline stage. MMA tiles: 16 for Q8_0 (8 KB of weights per
// 16-row group; 32 measured 8-35 % slower at 4-16 rows); Q4_K 32 with one
// 8-token tile (8 KB of nibbles: 5-8 rows 6-21 % faster than 16) and 16
// with two, whose larger stash would leave too few stages in flight (32
// measured 35 % slower at 12 and 16 rows). Integer dot products: 32 for both
// (16 KB of Q8_0, 8 KB of Q4_K nibbles per stage): shorter stages are too
// short for the fixed per-stage work (barrier waits, hand-over) of every
// warp (Q8_0 at 16: 17408 -> 5120 M = 1 20.7 against 19.0 us), longer ones
// leave too few stages in flight (Q4_K at 48 or 64: 18.7 against 16.6 us).
#ifndef QG_DEC_SBLK_Q8
#define QG_DEC_SBLK_Q8 16
#endif
#ifndef QG_DEC_SBLK_Q4K
#define QG_DEC_SBLK_Q4K 16
#endif
#ifndef QG_DEC_SBLK_Q4K_TT1
#define QG_DEC_SBLK_Q4K_TT1 32
#endif
#ifndef QG_DEC_SBLK_DP4A_Q8
#define QG_DEC_SBLK_DP4A_Q8 32
#endif
#ifndef QG_DEC_SBLK_DP4A_Q4K
#define QG_DEC_SBLK_DP4A_Q4K 32
#endif
template <int TT, bool kQ4K, bool kDp4a>
__host__ __device__ constexpr int sblk() {
  return kDp4a ? (kQ4K ? QG_DEC_SBLK_DP4A_Q4K : QG_DEC_SBLK_DP4A_Q8)
               : (kQ4K ? (TT == 1 ? QG_DEC_SBLK_Q4K_TT1 : QG_DEC_SBLK_Q4K) : QG_DEC_SBLK_Q8);
}
// CTAs of 320 threads resident per SM (registers and shared memory are
// budgeted for it)
// (kKind: 0 the dp4a kernel, 1 / 2 the MMA kernel with one / two token
// tiles). W4A8 on one MMA token tile (5-8 rows) runs two per SM with a deeper
// ring: at 8 rows 5120 -> 17408 29.1 -> 25.0 us and 17408 -> 5120 37.6 ->
// 33.2 us (at 5-6 rows 1-4 % slower); the dp4a kernel with two per SM
// measured slower (17408 -> 5120 at 1 row 19.0 -> 21.1 us)
#ifndef QG_DEC_CTAS_Q4K
#define QG_DEC_CTAS_Q4K 3
#endif
#ifndef QG_DEC_CTAS_Q4K_TT1
#define QG_DEC_CTAS_Q4K_TT1 2
#endif
#ifndef QG_DEC_CTAS_Q4K_TT2
#define QG_DEC_CTAS_Q4K_TT2 3
#endif
#ifndef QG_DEC_CTAS_Q8
#define QG_DEC_CTAS_Q8 3
#endif
#ifndef QG_DEC_CTAS_Q8_TT1
#define QG_DEC_CTAS_Q8_TT1 3
#endif
template <bool kQ4K, int kKind>
__host__ __device__ constexpr int dec_ctas() {
  return kQ4K ? (kKind == 1 ? QG_DEC_CTAS_Q4K_TT1 : kKind == 2 ? QG_DEC_CTAS_Q4K_TT2 : QG_DEC_CTAS_Q4K)
              : (kKind == 1 ? QG_DEC_CTAS_Q8_TT1 : QG_DEC_CTAS_Q8);
}
template <bool kQ4K, int kKind>
constexpr int dec_smem_budget() { return dec_ctas<kQ4K, kKind>() == 2 ? 110 * 1024 : 70 * 1024; }
// MMA tiles: blocks whose sums the chain warp loads before their FMAs: 4 for
// Q8_0, one at a time for Q4_K (whose sub-block terms need the registers).
#ifndef QG_DEC_HB_Q4K
#define QG_DEC_HB_Q4K 1
#endif
template <bool kQ4K>
__host__ __device__ constexpr int dec_hbatch() { return kQ4K ? QG_DEC_HB_Q4K : 4; }
// Rows up to which the integer dot-product kernel runs (one lane per weight
// row; each token's 32 activation bytes of a block are loaded by every row's
// lane) rather than MMA tiles (activations loaded once per 8-token tile); at
// most kDp4aMaxM. Measured on GB300 (both kernels releasing stages from
// their compute warps): 4 rows tie at 5120 -> 17408 for both formats and
// favour the integer kernel at 17408 -> 5120 for W8A8 (24.9 vs 25.7 us);
// W4A8 ties there too (28.9 us).
constexpr int kDp4aMaxM = 4;
#ifndef QG_DEC_DP4A_MAX_Q8
#define QG_DEC_DP4A_MAX_Q8 4
#endif
#ifndef QG_DEC_DP4A_MAX_Q4K
#define QG_DEC_DP4A_MAX_Q4K 4
#endif
template <bool kQ4K>
constexpr int dec_dp4a_max_m() { return kQ4K ? QG_DEC_DP4A_MAX_Q4K : QG_DEC_DP4A_MAX_Q8; }
static_assert(QG_DEC_DP4A_MAX_Q8 <= kDp4aMaxM && QG_DEC_DP4A_MAX_Q4K <= kDp4aMaxM,
              "the integer kernel's stash and chain hold at most four tokens");
#ifndef QG_DEC_BUDGET_TT2_KB
#define QG_DEC_BUDGET_TT2_KB 70
#endif
#ifndef QG_DEC_EARLY
#define QG_DEC_EARLY 1  // the compute warps, not the chain warp, release each stage
#endif
#ifndef QG_DEC_CHAIN_UNROLL
#define QG_DEC_CHAIN_UNROLL 1  // chain warp: a full stage's block quads unrolled
#endif


// Shared-memory layout (offsets depend on M, fixed at launch):
//   NW weight stages, each: weights | scales | M activation rows | (W4A8) M
//   block-sum rows -- released by the chain warp;
//   2 stash slots between compute and chain warps: exact block sums, and for
//   W4A8 the rows' d*sc, dmin*m (and, integer kernel, -asum per token);
//   barriers full[NW], empty[NW], xfull[2], xempty[2].
// Stash sums: MMA tiles keep an m16n8 accumulator fragment per block and
// 8-token tile ([block][tile][lane][4], W4A8 scales [block][row]); the
// integer kernel keeps, per block, token pair and row, the two sums (W8A8)
// or the two sums with the row's d*sc and dmin*m (W4A8, one 16-byte load
// for the chain), and for W4A8 -asum per block and token.
template <int TT, bool kQ4K, bool kDp4a, int kPairs = 2>
struct DecodeSmem {
  static constexpr int kSBlk = sblk<TT, kQ4K, kDp4a>();
  // bytes per activation row in a stage: 32 per block + 32 of padding, so the
  // eight rows one 8-byte load touches fall in distinct banks
  static constexpr int kARow = kSBlk * 32 + 32;
  static constexpr int kWBytes = kSBlk * (kQ4K ? 256 : 512);  // weights per stage
  static constexpr int kSBytes = kQ4K ? kSBlk / 8 * 256 : kSBlk / 4 * 128;  // scales / headers
  static constexpr int kXBytes =
      kDp4a ? kSBlk * kPairs * 16 * (kQ4K ? 16 : 8) : kSBlk * TT * 32 * 16;
  static constexpr int kScBytes = (kQ4K && !kDp4a) ? kSBlk * 16 * 8 : 0;
  static constexpr int kAsBytes = (kQ4K && kDp4a) ? kSBlk * kDp4aMaxM * 4 : 0;
  // The chain warp's inputs that arrive with the stage (Q8_0 scales; MMA
  // tiles' Q4_K activation block sums of up to TT*8 rows), copied into the
  // stash by the compute warps so that they, not the chain, release the stage
  static constexpr bool kEarly = QG_DEC_EARLY != 0;
  // (the integer kernel's Q4_K chain reads its stash alone)
  static constexpr int kCdBytes =
      kEarly ? (kQ4K ? (kDp4a ? 0 : TT * 8 * kSBlk * 4) : kSBytes) : 0;
  static constexpr int kCdOff = kXBytes + kScBytes + kAsBytes;
  static constexpr int kSlotBytes = kXBytes + kScBytes + kAsBytes + kCdBytes;
  static constexpr int kMaxNw = 8;
  // the activation rows and the block sums are TMA destinations: each starts
  // on a 128-byte boundary of the stage (stages are 128-byte multiples)
  static_assert((kWBytes + kSBytes) % 128 == 0, "activation rows 128-byte aligned");
  static __host__ __device__ int stage_bytes(int mrows) {
    return (int)align_up(bsum_off(mrows) + (kQ4K ? mrows * kSBlk * 4 : 0), 128);
  }
  static __host__ __device__ int act_off() { return kWBytes + kSBytes; }
  static __host__ __device__ int bsum_off(int mrows) {
    return (int)align_up(kWBytes + kSBytes + mrows * kARow, 128);
  }
  // weight stages that fit in `budget` bytes next to the stash and barriers
  static int num_stages(int mrows, int budget) {
    const int fixed = 2 * kSlotBytes + 2 * (kMaxNw + 2) * 8;
    int nw = (budget - fixed) / stage_bytes(mrows);
    return nw < 2 ? 2 : (nw > kMaxNw ? kMaxNw : nw);
  }
  static __host__ __device__ int total(int mrows, int nw) {
    return nw * stage_bytes(mrows) + 2 * kSlotBytes + 2 * (nw + 2) * 8;
  }
};

// Exact integer dot products of four byte pairs (dp4a): both operands signed,
// or unsigned weights with signed activations.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Sub-block i's scales of a packed Q4_K row header (d, dmin, then 12-bit
// units sc_i | m_i << 6 at bits [12i, 12i+12) of words y, z, w): d*sc_i and
// dmin*m_i, exact products.
// A 6-bit field f enters as the float 2^23 + f (its bits or'ed into the
// mantissa of 2^23); fmaf(d, 2^23 + f, -d * 2^23) rounds the exact value d*f,
// which fits in fp32 (11 + 6 significant bits), so it is d*f exactly.
__device__ __forceinline__ float2 q4k_scales(const uint4& H, int i) {
  const uint32_t lo = i < 3 ? H.y : (i < 6 ? H.z : H.w);
  const uint32_t hi = i < 3 ? H.z : H.w;
  const uint32_t u = __funnelshift_r(lo, hi, (12 * i) & 31);
  const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&H.x));
  const float sc = __uint_as_float((u & 63u) | 0x4B000000u);
  const float mn = __uint_as_float(((u >> 6) & 63u) | 0x4B000000u);
  return make_float2(fmaf(dd.x, sc, dd.x * -8388608.0f), fmaf(dd.y, mn, dd.y * -8388608.0f));
}

// An integer of magnitude below 2^22 as fp32 (exact): added to the bits of
// 1.5 * 2^23 it lands in the mantissa, and subtracting 1.5 * 2^23 leaves it.
__device__ __forceinline__ float small_int_to_f32(int v) {
  return __int_as_float(v + 0x4B400000) - 12582912.0f;
}

// Eight 4-bit values of a packed Q4_K word (byte e: low nibble k = e, high
// nibble k = 4 + e) as exact fp16 pairs: p0 = (k0, k2), p8 = (k1, k3), p4 =
// (k4, k6), p12 = (k5, k7). A nibble or'ed into the mantissa of 1024 gives
// 1024 + q (minus 1024); one in mantissa bits 4..7 gives 1024 + 16q, which
// one fused multiply-add by 1/16 minus 64 brings back to q.
__device__ __forceinline__ void nib_word_to_f16(uint32_t w, uint32_t& p0, uint32_t& p8,
                                                uint32_t& p4, uint32_t& p12) {
  const uint32_t w8 = w >> 8;
  const uint32_t l0 = (w & 0x000F000Fu) | 0x64006400u, h0 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t l8 = (w8 & 0x000F000Fu) | 0x64006400u, h8 = (w8 & 0x00F000F0u) | 0x64006400u;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(p0) : "r"(l0), "r"(0x64006400u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(p8) : "r"(l8), "r"(0x64006400u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(p4) : "r"(h0), "r"(0x2C002C00u), "r"(0xD400D400u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(p12) : "r"(h8), "r"(0x2C002C00u), "r"(0xD400D400u));
}

// Four biased bytes (q + 128) as exact fp16 pairs of bytes (0, 2) and (1, 3).
__device__ __forceinline__ void biased_u8x4_to_f16x4_even_odd(uint32_t u, uint32_t& lo,
                                                              uint32_t& hi) {
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4240;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4341;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

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
  int nw;           // weight stages in the ring
  int pdl;          // launched as a programmatic dependent of the quantize kernel
};

// Warp 0 of a decode CTA: streams stage after stage of the CTA's groups into
// the ring (weights and scales, then the activation rows and, for W4A8,
// their block sums), and at the end waits until every stage has been handed
// back.
template <class L, bool kQ4K>
__device__ __forceinline__ void decode_produce(const DecodeArgs& a, const CUtensorMap* tmX,
                                               const CUtensorMap* tmS, uint8_t* smem, int SBY,
                                               int mrows, uint64_t* full, uint64_t* empty,
                                               int lane) {
  constexpr int kSBlk = L::kSBlk;
  constexpr int kARow = L::kARow;
  const int NW = a.nw;
  const int B = a.K / kBlk;
  const int B4 = (B + 3) & ~3;
  const int J = B / 8;
  const int nstages = (B + kSBlk - 1) / kSBlk;
  // The activation rows (and W4A8 block sums) of stage r into ring slot
  // `slot`: one 2-D copy each, all rows at once, landing at the stage's row
  // pitch (the box's rows carry the pitch's padding, read from the next
  // stage or as zeros past K, never used)
  auto copy_acts = [&](int r, int slot) {
    if (lane == 0) {
      uint8_t* base = smem + slot * SBY;
      tma_load_2d(base + L::act_off(), tmX, &full[slot], r * kSBlk * (kBlk / 8), 0);
      if (kQ4K) tma_load_2d(base + L::bsum_off(mrows), tmS, &full[slot], r * kSBlk / 2, 0);
    }
  };
  // Launched as a programmatic dependent, the weights and scales of the
  // first P stages are requested before any activation: the quantize kernel
  // may still be writing the activations, and griddep_wait() returns once it
  // has completed. P is at most 3: every CTA's first three stages are ~1 us
  // of HBM time, about what a decode-sized quantize lasts; more would still
  // be arriving when the activations are requested, and stage 0's
  // activations would queue behind them. An ordinary launch requests each
  // stage's activations right after its weights.
  // The CTA's groups are g = blockIdx.x, + gridDim.x, ... (grid capped at the
  // resident CTAs): the ring streams from one group into the next without
  // draining. The activation slices are the same for every group.
  const int P = a.pdl ? min(min(nstages, NW), 3) : 1;
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  bool first = true;
  for (int64_t g = blockIdx.x; g < a.G && ok; g += gridDim.x, first = false) {
    for (int s = 0; s < nstages; ++s) {
      const int blk0 = s * kSBlk;
      const int nb = min(kSBlk, B - blk0);
      uint8_t* base = smem + st * SBY;
      uint32_t bytes = !kQ4K ? nb * 512 + ((nb + 3) / 4) * 128 : nb * 256 + (nb / 8) * 256;
      bytes += mrows * kARow;                   // whole boxes (zero-filled past K)
      if (kQ4K) bytes += mrows * kSBlk * 4;
      if (lane == 0) {
        ok = mbar_wait(&empty[st], ph ^ 1, a.err);
        if (ok) {
          // the consumers read the slot through the generic proxy; the copies
          // below rewrite it through the async proxy, ordered after those
          // reads (which the wait made visible) only by this fence
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[st], bytes);
          if (!kQ4K) {
            bulk_copy_g2s(base, a.wstream + (g * B + blk0) * 512, nb * 512, &full[st]);
            bulk_copy_g2s(base + L::kWBytes, a.wscale + (g * (B4 / 4) + blk0 / 4) * 128,
                      ((nb + 3) / 4) * 128, &full[st]);
          } else {
            bulk_copy_g2s(base, a.wstream + (g * B + blk0) * 256, nb * 256, &full[st]);
            bulk_copy_g2s(base + L::kWBytes, a.wscale + (g * J + blk0 / 8) * 256, (nb / 8) * 256,
                      &full[st]);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (first && s + 1 == P) {
        // the first group's first P stages are slots 0..P-1 of the first round
        if (a.pdl) griddep_wait();
        for (int r = 0; r < P; ++r) copy_acts(r, r);
      } else if (!first || s >= P) {
        copy_acts(s, st);
      }
      if (++st == NW) { st = 0; ph ^= 1; }
    }
  }
  // drain: every stage released before the CTA exits
  if (lane == 0) {
    for (int i = 0; i < NW; ++i) {
      if (!mbar_wait(&empty[st], ph ^ 1, a.err)) break;
      if (++st == NW) { st = 0; ph ^= 1; }
    }
  }
}

// Decode GEMM on legacy MMA tiles of 16 weight rows x 8 tokens (TT tiles):
// int8 m16n8k32 on the stored bytes, or (build switch) fp16 m16n8k16 on
// values widened in registers.
template <int TT, bool kQ4K, bool kDebug>
__global__ void __launch_bounds__(32 * (kCompWarps + 2), dec_ctas<kQ4K, TT>())
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmS, const DecodeArgs a) {
  using L = DecodeSmem<TT, kQ4K, false>;
  constexpr int kSBlk = L::kSBlk;
  constexpr int kARow = L::kARow;
  constexpr int kBlkPerWarp = kSBlk / kCompWarps;
  // (W4A8: each half-warp decodes the scales of every other one of the
  // warp's blocks)
  static_assert(!kQ4K || kBlkPerWarp % 2 == 0, "an even number of blocks per compute warp");
  extern __shared__ __align__(128) uint8_t smem[];
  const int NW = a.nw;
  const int mrows = min(a.M, TT * 8);
  const int SBY = L::stage_bytes(mrows);
  float* stash_base = reinterpret_cast<float*>(smem + NW * SBY);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NW * SBY + 2 * L::kSlotBytes);
  uint64_t* empty = full + NW;    // weight stage consumed (compute warps, or the chain warp)
  uint64_t* xfull = empty + NW;   // stash slot written (count: compute warps)
  uint64_t* xempty = xfull + 2;   // stash slot read by the chain warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.K / kBlk;
  const int nstages = (B + kSBlk - 1) / kSBlk;
  const int M = a.M;
  const int gr = lane >> 2, c = lane & 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], L::kEarly ? kCompWarps : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xfull[i], kCompWarps);
      mbar_init(&xempty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    decode_produce<L, kQ4K>(a, &tmX, &tmS, smem, SBY, mrows, full, empty, lane);
    return;
  }

  if (warp <= kCompWarps) {
    // ------------------------------------------------------ compute warps
    const int cw = warp - 1;
    int st = 0, xs = 0;
    uint32_t ph = 0, xph = 0;
    bool ok = true;
    for (int64_t g = blockIdx.x; g < a.G && ok; g += gridDim.x) {
    for (int s = 0; s < nstages; ++s) {
      const int blk0 = s * kSBlk;
      const int nb = min(kSBlk, B - blk0);
      ok = mbar_wait(&full[st], ph, a.err) && mbar_wait(&xempty[xs], xph ^ 1, a.err);
      if (!ok) break;
      const uint8_t* base = smem + st * SBY;
      float* stash = stash_base + xs * (L::kSlotBytes / 4);
      if constexpr (QG_DEC_IMMA != 0) {
        // one int8 m16n8k32 MMA per block and 8-token tile, on the stored
        // bytes: lane (gr, c) gives k 8c..8c+7 of rows gr and gr+8 (a0/a2,
        // a1/a3) and of its token (b0/b1), the same k on both operands; Q4_K
        // nibbles are masked into unsigned bytes (low: k 8c..8c+3, high:
        // 8c+4..8c+7). The int32 sums are exact; |sum| < 2^20 makes them
        // exact in fp32 for the chain warp.
        uint32_t af[kBlkPerWarp][4];
#pragma unroll
        for (int u = 0; u < kBlkPerWarp; ++u) {
          const int j = cw * kBlkPerWarp + u;
          if (!kQ4K) {
            const int q = c >> 1;
            const uint8_t* wp = base + j * 512 + 8 * (c & 1);
            const uint2 xa = *reinterpret_cast<const uint2*>(wp + (q * 16 + (gr ^ (q << 2))) * 16);
            const uint2 xb =
                *reinterpret_cast<const uint2*>(wp + (q * 16 + ((gr + 8) ^ (q << 2))) * 16);
            af[u][0] = xa.x; af[u][2] = xa.y;
            af[u][1] = xb.x; af[u][3] = xb.y;
          } else {
            const uint8_t* wp = base + j * 256 + 4 * c;
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(wp + gr * 16);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(wp + (gr + 8) * 16);
            af[u][0] = wa & 0x0F0F0F0Fu; af[u][2] = (wa >> 4) & 0x0F0F0F0Fu;
            af[u][1] = wb & 0x0F0F0F0Fu; af[u][3] = (wb >> 4) & 0x0F0F0F0Fu;
          }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const int mrow = 8 * t + gr;  // token of this lane's B fragment
#pragma unroll
          for (int u = 0; u < kBlkPerWarp; ++u) {
            const int j = cw * kBlkPerWarp + u;
            uint2 bv = make_uint2(0u, 0u);
            if (mrow < M)
              bv = *reinterpret_cast<const uint2*>(base + L::act_off() + mrow * kARow + c * 8 + j * 32);
            int d[4];
            mma_i8_16832<kQ4K>(d, af[u], bv.x, bv.y);
            // d: (n0, tok 8t+2c), (n0, 8t+2c+1), (n1, 8t+2c), (n1, 8t+2c+1)
            if (j < nb)
              *reinterpret_cast<float4*>(stash + ((j * TT + t) * 32 + lane) * 4) =
                  make_float4(small_int_to_f32(d[0]), small_int_to_f32(d[1]),
                              small_int_to_f32(d[2]), small_int_to_f32(d[3]));
            if (kDebug && j < nb) {
              const int b = blk0 + j;
              const int n0 = (int)(16 * g + gr), mc0 = 8 * t + 2 * c;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int m = mc0 + (i & 1), n = n0 + ((i < 2) ? 0 : 8);
                if (m < M && n < a.N) a.dbg[((int64_t)m * a.N + n) * B + b] = d[i];
              }
            }
          }
        }
      } else {
        // two m16n8k16 fp16 MMAs per block and 8-token tile (this warp's
        // blocks 2cw, 2cw+1; their fragments first, so the blocks' load and
        // MMA latencies overlap)
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a0[kBlkPerWarp][4], a1[kBlkPerWarp][4];  // A fragments
#pragma unroll
        for (int u = 0; u < kBlkPerWarp; ++u) {
          const int j = cw * kBlkPerWarp + u;
          if (!kQ4K) {
            // rows gr and gr+8, k 8c .. 8c+7 (chunk c/2 of each row)
            const int q = c >> 1;
            const uint8_t* wp = base + j * 512 + 8 * (c & 1);
            const uint2 xa = *reinterpret_cast<const uint2*>(wp + (q * 16 + (gr ^ (q << 2))) * 16);
            const uint2 xb =
                *reinterpret_cast<const uint2*>(wp + (q * 16 + ((gr + 8) ^ (q << 2))) * 16);
            biased_u8x4_to_f16x4(xa.x ^ 0x80808080u, a0[u][0], a0[u][2]);
            biased_u8x4_to_f16x4(xb.x ^ 0x80808080u, a0[u][1], a0[u][3]);
            biased_u8x4_to_f16x4(xa.y ^ 0x80808080u, a1[u][0], a1[u][2]);
            biased_u8x4_to_f16x4(xb.y ^ 0x80808080u, a1[u][1], a1[u][3]);
          } else {
            // word c of rows gr and gr+8: k 8c .. 8c+7; the MMA's k slots
            // (2c, 2c+1) / (2c+8, 2c+9) take k (8c, 8c+2) / (8c+1, 8c+3) and,
            // in the second MMA, (8c+4, 8c+6) / (8c+5, 8c+7)
            const uint8_t* wp = base + j * 256 + 4 * c;
            nib_word_to_f16(*reinterpret_cast<const uint32_t*>(wp + gr * 16), a0[u][0], a0[u][2],
                            a1[u][0], a1[u][2]);
            nib_word_to_f16(*reinterpret_cast<const uint32_t*>(wp + (gr + 8) * 16), a0[u][1],
                            a0[u][3], a1[u][1], a1[u][3]);
          }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const int mrow = 8 * t + gr;  // token of this lane's B fragment
#pragma unroll
          for (int u = 0; u < kBlkPerWarp; ++u) {
            const int j = cw * kBlkPerWarp + u;
            uint32_t b00 = 0, b01 = 0, b10 = 0, b11 = 0;
            if (mrow < M) {
              const uint2 bv = *reinterpret_cast<const uint2*>(
                  base + L::act_off() + mrow * kARow + c * 8 + j * 32);
              if (!kQ4K) {
                biased_u8x4_to_f16x4(bv.x ^ 0x80808080u, b00, b01);
                biased_u8x4_to_f16x4(bv.y ^ 0x80808080u, b10, b11);
              } else {
                biased_u8x4_to_f16x4_even_odd(bv.x ^ 0x80808080u, b00, b01);
                biased_u8x4_to_f16x4_even_odd(bv.y ^ 0x80808080u, b10, b11);
              }
            }
            float d[4];
            mma_f16_16816(d, a0[u], b00, b01, zero4);
            mma_f16_16816(d, a1[u], b10, b11, d);
            // d: (n0, tok 8t+2c), (n0, 8t+2c+1), (n1, 8t+2c), (n1, 8t+2c+1): exact sums
            if (j < nb)
              *reinterpret_cast<float4*>(stash + ((j * TT + t) * 32 + lane) * 4) =
                  make_float4(d[0], d[1], d[2], d[3]);
            if (kDebug && j < nb) {
              const int b = blk0 + j;
              const int n0 = (int)(16 * g + gr), mc0 = 8 * t + 2 * c;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int m = mc0 + (i & 1), n = n0 + ((i < 2) ? 0 : 8);
                if (m < M && n < a.N) a.dbg[((int64_t)m * a.N + n) * B + b] = __float2int_rn(d[i]);
              }
            }
          }
        }
      }
      if (kQ4K) {
        // lane (r, hh): row r's d*sc and dmin*m of the warp's blocks hh, hh + 2, ...
        const int r = lane & 15;
#pragma unroll
        for (int v = 0; v < kBlkPerWarp / 2; ++v) {
          const int j = cw * kBlkPerWarp + 2 * v + (lane >> 4);
          if (j < nb) {
            const uint4 H =
                *reinterpret_cast<const uint4*>(base + L::kWBytes + (j >> 3) * 256 + r * 16);
            float2* scw = reinterpret_cast<float2*>(stash + L::kXBytes / 4);
            scw[j * 16 + r] = q4k_scales(H, j & 7);
          }
        }
      }
      if constexpr (L::kEarly) {
        // the chain's inputs from the stage into the stash, 16 bytes a lane
        const int nchunk = (kQ4K ? mrows * kSBlk * 4 : L::kSBytes) / 16;
        const uint8_t* src = base + (kQ4K ? L::bsum_off(mrows) : L::kWBytes);
        uint8_t* dst = reinterpret_cast<uint8_t*>(stash) + L::kCdOff;
        for (int i = cw * 32 + lane; i < nchunk; i += kCompWarps * 32)
          *reinterpret_cast<uint4*>(dst + 16 * i) = *reinterpret_cast<const uint4*>(src + 16 * i);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&xfull[xs]);
        if (L::kEarly) mbar_arrive(&empty[st]);  // this warp's reads of the stage are done
      }
      if (++st == NW) { st = 0; ph ^= 1; }
      if (++xs == 2) { xs = 0; xph ^= 1; }
    }
    }
    return;
  }

  // ----------------------------------------------------------- chain warp
  bool ok = true;
  int st = 0, xs = 0;
  uint32_t ph = 0, xph = 0;
  for (int64_t g = blockIdx.x; g < a.G && ok; g += gridDim.x) {
  const int n0 = (int)(16 * g + gr), n1 = n0 + 8;
  float2 acc[TT][2];  // [tile][row n0 / n1]: tokens 8t+2c, 8t+2c+1
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = make_float2(0.f, 0.f);
  for (int s = 0; s < nstages && ok; ++s) {
    const int blk0 = s * kSBlk;
    const int nb = min(kSBlk, B - blk0);
    ok = mbar_wait(&xfull[xs], xph, a.err);
    if (!ok) break;
    const uint8_t* base = smem + st * SBY;
    const float* stash = stash_base + xs * (L::kSlotBytes / 4);
    const uint8_t* cd = reinterpret_cast<const uint8_t*>(stash) + L::kCdOff;
    const uint8_t* sb = L::kEarly ? cd : base + L::kWBytes;
    const int32_t* bb = reinterpret_cast<const int32_t*>(L::kEarly ? cd : base + L::bsum_off(mrows));
    const float2* scs = reinterpret_cast<const float2*>(stash + L::kXBytes / 4);  // [block][row]
    // blocks in groups of kG (a quad of Q8_0 scales); a full stage's quads
    // are unrolled so that later quads' shared loads overlap earlier FMAs
    constexpr int kG = 4;
    auto quad = [&](const int j0) {
      float dA[kG], dB[kG], mA[kG], mB[kG];
      if (!kQ4K) {
        const uint4 sc = *reinterpret_cast<const uint4*>(sb + (j0 >> 2) * 128 + gr * 16);
        const __half2* h = reinterpret_cast<const __half2*>(&sc);
        const float2 f0 = __half22float2(h[0]), f1 = __half22float2(h[1]);
        const float2 f2 = __half22float2(h[2]), f3 = __half22float2(h[3]);
        dA[0] = f0.x; dA[1] = f0.y; dA[2] = f1.x; dA[3] = f1.y;
        dB[0] = f2.x; dB[1] = f2.y; dB[2] = f3.x; dB[3] = f3.y;
      } else {
        // decoded by the compute warps: rows gr and gr+8 of each block
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const float2 s0 = scs[(j0 + u) * 16 + gr], s1 = scs[(j0 + u) * 16 + gr + 8];
          dA[u] = s0.x;
          dB[u] = s1.x;
          mA[u] = -s0.y;
          mB[u] = -s1.y;
        }
      }
      // the exact sums of kH blocks (and for W4A8 their activation sums)
      // are loaded before their FMAs, so one shared-memory latency covers kH
      // blocks (blocks past nb are loaded, never used; a per-block load
      // right before its FMAs cost ~90 cycles a block)
      constexpr int kH = dec_hbatch<kQ4K>();
#pragma unroll
      for (int h = 0; h < kG; h += kH) {
        float4 x[kH][TT];
        float2 as[kH][TT];
#pragma unroll
        for (int u = 0; u < kH; ++u) {
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            const int j = j0 + h + u;
            x[u][t] = *reinterpret_cast<const float4*>(stash + ((j * TT + t) * 32 + lane) * 4);
            if (kQ4K) {
              const int mc0 = 8 * t + 2 * c, mc1 = mc0 + 1;
              as[u][t] = make_float2((mc0 < M) ? (float)bb[mc0 * kSBlk + j] : 0.f,
                                     (mc1 < M) ? (float)bb[mc1 * kSBlk + j] : 0.f);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kH; ++u) {
          if (j0 + h + u < nb) {
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              const float4& xv = x[u][t];
              const int uu = h + u;
              acc[t][0] = __ffma2_rn(make_float2(xv.x, xv.y), make_float2(dA[uu], dA[uu]), acc[t][0]);
              acc[t][1] = __ffma2_rn(make_float2(xv.z, xv.w), make_float2(dB[uu], dB[uu]), acc[t][1]);
              if (kQ4K) {
                acc[t][0] = __ffma2_rn(as[u][t], make_float2(mA[uu], mA[uu]), acc[t][0]);
                acc[t][1] = __ffma2_rn(as[u][t], make_float2(mB[uu], mB[uu]), acc[t][1]);
              }
            }
          }
        }
      }
    
    };
    if (QG_DEC_CHAIN_UNROLL && nb == kSBlk) {
#pragma unroll
      for (int j0 = 0; j0 < kSBlk; j0 += kG) quad(j0);
    } else {
      for (int j0 = 0; j0 < nb; j0 += kG) quad(j0);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&xempty[xs]);
      if (!L::kEarly) mbar_arrive(&empty[st]);
    }
    if (++st == NW) { st = 0; ph ^= 1; }
    if (++xs == 2) { xs = 0; xph ^= 1; }
  }

  if (kDebug || !ok) continue;
  griddep_wait();  // the activation scales come from the preceding quantize kernel
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const float accs[4] = {acc[t][0].x, acc[t][0].y, acc[t][1].x, acc[t][1].y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = 8 * t + 2 * c + (i & 1), n = (i < 2) ? n0 : n1;
      if (m < M && n < a.N) {
        const float y = accs[i] * __ldg(a.sa + m);
        if (a.out_f32)
          reinterpret_cast<float*>(a.out)[(int64_t)m * a.ldo + n] = y;
        else
          reinterpret_cast<uint16_t*>(a.out)[(int64_t)m * a.ldo + n] = f32_to_bf16_rne(y);
      }
    }
  }
  }
}

// Decode GEMM for at most four rows on integer dot products. Compute warps:
// half-warp hh of warp cw takes blocks cw + 8*hh (+ 16, + 32 ... within the
// stage), one lane per weight row: two 16-byte loads of the row's 32 int8
// values of the block (W4A8: one load of its 32 nibbles, masked into low
// and high bytes), two of each token's 32 activation bytes, eight dp4a per
// token, and the exact int32 sum goes to the stash as fp32 (|sum| < 2^20).
// For W4A8 the lane also decodes its row's d*sc and dmin*m (exact products;
// the block's sub-block index is cw for every lane of the warp), and lanes r
// < M store token r's -asum of the block. No value is widened to fp16 and no
// lane idles at one token. Chain warp: lane (r, tp) carries weight row r and
// tokens 2tp, 2tp+1 as one packed pair, applying per block, in ascending
// order, acc = fmaf(isum, d, acc) (W4A8: fmaf(isum, d*sc, acc) then
// fmaf(-asum, dmin*m, acc)): the same operations in the same order as the
// MMA kernel and the prefill kernel.
template <bool kQ4K, int kM, bool kDebug>
__global__ void __launch_bounds__(32 * (kCompWarps + 2), dec_ctas<kQ4K, 0>())
    decode_dp4a_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmS, const DecodeArgs a) {
  constexpr int kPairs = (kM + 1) / 2;  // token pairs
  using L = DecodeSmem<1, kQ4K, true, kPairs>;
  constexpr int kSBlk = L::kSBlk;
  constexpr int kARow = L::kARow;
  constexpr int kPer = kSBlk / (2 * kCompWarps);  // blocks per lane and stage
  static_assert(kSBlk % (2 * kCompWarps) == 0 && kCompWarps == 8,
                "a warp's blocks share their sub-block index");
  extern __shared__ __align__(128) uint8_t smem[];
  const int NW = a.nw;
  static_assert(kM >= 1 && kM <= kDp4aMaxM, "rows of the integer kernel");
  constexpr int M = kM;  // == a.M
  const int SBY = L::stage_bytes(M);
  float* stash_base = reinterpret_cast<float*>(smem + NW * SBY);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NW * SBY + 2 * L::kSlotBytes);
  uint64_t* empty = full + NW;    // weight stage consumed (compute warps, or the chain warp)
  uint64_t* xfull = empty + NW;   // stash slot written (count: compute warps)
  uint64_t* xempty = xfull + 2;   // stash slot read by the chain warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.K / kBlk;
  const int nstages = (B + kSBlk - 1) / kSBlk;
  const int r = lane & 15, hh = lane >> 4;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], L::kEarly ? kCompWarps : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xfull[i], kCompWarps);
      mbar_init(&xempty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    decode_produce<L, kQ4K>(a, &tmX, &tmS, smem, SBY, M, full, empty, lane);
    return;
  }

  if (warp <= kCompWarps) {
    // ------------------------------------------------------ compute warps
    const int cw = warp - 1;
    int st = 0, xs = 0;
    uint32_t ph = 0, xph = 0;
    bool ok = true;
    for (int64_t g = blockIdx.x; g < a.G && ok; g += gridDim.x) {
      const int64_t n = 16 * g + r;
      for (int s = 0; s < nstages; ++s) {
        const int blk0 = s * kSBlk;
        const int nb = min(kSBlk, B - blk0);
        ok = mbar_wait(&full[st], ph, a.err) && mbar_wait(&xempty[xs], xph ^ 1, a.err);
        if (!ok) break;
        const uint8_t* base = smem + st * SBY;
        float* xsum = stash_base + xs * (L::kSlotBytes / 4);  // [block][pair][row][2 or 4]
        float* asn = xsum + L::kXBytes / 4;                    // [block][token]
        const int32_t* bb = reinterpret_cast<const int32_t*>(base + L::bsum_off(M));
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int j = cw + kCompWarps * hh + 2 * kCompWarps * u;
          const uint8_t* act = base + L::act_off() + j * 32;
          int isum[kM];
          if (!kQ4K) {
            const uint8_t* wp = base + j * 512;
            const uint4 w0 = *reinterpret_cast<const uint4*>(wp + r * 16);             // k 0..15
            const uint4 w1 = *reinterpret_cast<const uint4*>(wp + (16 + (r ^ 4)) * 16);  // k 16..31
#pragma unroll
            for (int m = 0; m < kM; ++m) {
              const uint4 x0 = *reinterpret_cast<const uint4*>(act + m * kARow);
              const uint4 x1 = *reinterpret_cast<const uint4*>(act + m * kARow + 16);
              int s0 = dp4a_ss(w0.x, x0.x, 0), s1 = dp4a_ss(w1.x, x1.x, 0);
              s0 = dp4a_ss(w0.y, x0.y, s0);
              s1 = dp4a_ss(w1.y, x1.y, s1);
              s0 = dp4a_ss(w0.z, x0.z, s0);
              s1 = dp4a_ss(w1.z, x1.z, s1);
              s0 = dp4a_ss(w0.w, x0.w, s0);
              s1 = dp4a_ss(w1.w, x1.w, s1);
              isum[m] = s0 + s1;
            }
          } else {
            // word x of the row: low nibbles k = 8x..8x+3, high nibbles
            // 8x+4..8x+7; the high nibbles stay in place (16 q), and their
            // sum is shifted back once (exact: a multiple of 16)
            const uint4 w = *reinterpret_cast<const uint4*>(base + j * 256 + r * 16);
            const uint32_t l0 = w.x & 0x0F0F0F0Fu, h0 = w.x & 0xF0F0F0F0u;
            const uint32_t l1 = w.y & 0x0F0F0F0Fu, h1 = w.y & 0xF0F0F0F0u;
            const uint32_t l2 = w.z & 0x0F0F0F0Fu, h2 = w.z & 0xF0F0F0F0u;
            const uint32_t l3 = w.w & 0x0F0F0F0Fu, h3 = w.w & 0xF0F0F0F0u;
#pragma unroll
            for (int m = 0; m < kM; ++m) {
              const uint4 x0 = *reinterpret_cast<const uint4*>(act + m * kARow);       // k 0..15
              const uint4 x1 = *reinterpret_cast<const uint4*>(act + m * kARow + 16);  // k 16..31
              int sl = dp4a_us(l0, x0.x, 0), sh = dp4a_us(h0, x0.y, 0);
              sl = dp4a_us(l1, x0.z, sl);
              sh = dp4a_us(h1, x0.w, sh);
              sl = dp4a_us(l2, x1.x, sl);
              sh = dp4a_us(h2, x1.y, sh);
              sl = dp4a_us(l3, x1.z, sl);
              sh = dp4a_us(h3, x1.w, sh);
              isum[m] = sl + (sh >> 4);
            }
          }
          if (j < nb) {
            float xf[2 * kPairs];
#pragma unroll
            for (int m = 0; m < 2 * kPairs; ++m) {
              xf[m] = m < kM ? small_int_to_f32(isum[m < kM ? m : 0]) : 0.f;
              if (kDebug && m < kM && n < a.N)
                a.dbg[((int64_t)m * a.N + n) * B + blk0 + j] = isum[m < kM ? m : 0];
            }
            if (!kQ4K) {
#pragma unroll
              for (int p = 0; p < kPairs; ++p)
                *reinterpret_cast<float2*>(xsum + ((j * kPairs + p) * 16 + r) * 2) =
                    make_float2(xf[2 * p], xf[2 * p + 1]);
            } else {
              const uint4 H =
                  *reinterpret_cast<const uint4*>(base + L::kWBytes + (j >> 3) * 256 + r * 16);
              const float2 sc = q4k_scales(H, cw);
#pragma unroll
              for (int p = 0; p < kPairs; ++p)
                *reinterpret_cast<float4*>(xsum + ((j * kPairs + p) * 16 + r) * 4) =
                    make_float4(xf[2 * p], xf[2 * p + 1], sc.x, sc.y);
              if (r < M) asn[j * kDp4aMaxM + r] = small_int_to_f32(-bb[r * kSBlk + j]);
            }
          }
        }
        if constexpr (L::kEarly && !kQ4K) {
          // the stage's scales into the stash for the chain, 16 bytes a lane
          const uint8_t* src = base + L::kWBytes;
          uint8_t* dst = reinterpret_cast<uint8_t*>(xsum) + L::kCdOff;
          for (int i = cw * 32 + lane; i < L::kSBytes / 16; i += kCompWarps * 32)
            *reinterpret_cast<uint4*>(dst + 16 * i) = *reinterpret_cast<const uint4*>(src + 16 * i);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&xfull[xs]);
          if (L::kEarly) mbar_arrive(&empty[st]);  // this warp's reads of the stage are done
        }
        if (++st == NW) { st = 0; ph ^= 1; }
        if (++xs == 2) { xs = 0; xph ^= 1; }
      }
    }
    return;
  }

  // ----------------------------------------------------------- chain warp
  const int tp = hh;                          // tokens 2tp, 2tp+1
  const int tpc = tp < kPairs ? tp : 0;       // (lanes past the last pair repeat pair 0)
  bool ok = true;
  int st = 0, xs = 0;
  uint32_t ph = 0, xph = 0;
  for (int64_t g = blockIdx.x; g < a.G && ok; g += gridDim.x) {
    const int64_t n = 16 * g + r;
    float2 acc = make_float2(0.f, 0.f);
    for (int s = 0; s < nstages && ok; ++s) {
      const int blk0 = s * kSBlk;
      const int nb = min(kSBlk, B - blk0);
      ok = mbar_wait(&xfull[xs], xph, a.err);
      if (!ok) break;
      const uint8_t* base = smem + st * SBY;
      const float* xsum = stash_base + xs * (L::kSlotBytes / 4);
      const float* asn = xsum + L::kXBytes / 4;
      const uint8_t* sbase =
          L::kEarly ? reinterpret_cast<const uint8_t*>(xsum) + L::kCdOff : base + L::kWBytes;
      // four blocks at a time: their operands are loaded before their FMAs
      auto quad = [&](const int j0) {
        if (!kQ4K) {
          float2 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            x[u] = *reinterpret_cast<const float2*>(xsum + (((j0 + u) * kPairs + tpc) * 16 + r) * 2);
          // fp16 scales of rows r&7 and (r&7)+8 for blocks j0..j0+3
          const uint2 dq = *reinterpret_cast<const uint2*>(sbase + (j0 >> 2) * 128 +
                                                           (r & 7) * 16 + (r >> 3) * 8);
          const float2 d01 = __half22float2(*reinterpret_cast<const __half2*>(&dq.x));
          const float2 d23 = __half22float2(*reinterpret_cast<const __half2*>(&dq.y));
          const float d[4] = {d01.x, d01.y, d23.x, d23.y};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (j0 + u < nb) acc = __ffma2_rn(x[u], make_float2(d[u], d[u]), acc);
        } else {
          float4 v[4];
          float2 as[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            v[u] = *reinterpret_cast<const float4*>(xsum + (((j0 + u) * kPairs + tpc) * 16 + r) * 4);
            as[u] = *reinterpret_cast<const float2*>(asn + (j0 + u) * kDp4aMaxM + 2 * tpc);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (j0 + u < nb) {
              acc = __ffma2_rn(make_float2(v[u].x, v[u].y), make_float2(v[u].z, v[u].z), acc);
              acc = __ffma2_rn(as[u], make_float2(v[u].w, v[u].w), acc);
            }
          }
        }
      };
      if (nb == kSBlk) {
#pragma unroll
        for (int j0 = 0; j0 < kSBlk; j0 += 4) quad(j0);
      } else {
        for (int j0 = 0; j0 < nb; j0 += 4) quad(j0);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&xempty[xs]);
        if (!L::kEarly) mbar_arrive(&empty[st]);
      }
      if (++st == NW) { st = 0; ph ^= 1; }
      if (++xs == 2) { xs = 0; xph ^= 1; }
    }
    if (kDebug || !ok) continue;
    griddep_wait();  // the activation scales come from the preceding quantize kernel
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int m = 2 * tp + i;
      if (m < M && n < a.N) {
        const float y = (i ? acc.y : acc.x) * __ldg(a.sa + m);
        if (a.out_f32)
          reinterpret_cast<float*>(a.out)[(int64_t)m * a.ldo + n] = y;
        else
          reinterpret_cast<uint16_t*>(a.out)[(int64_t)m * a.ldo + n] = f32_to_bf16_rne(y);
      }
    }
  }
}

// Launch of either decode kernel with layout L over `mrows` activation rows.
template <class L, bool kQ4K, class Kern>
static cudaError_t launch_decode(Kern kern, std::atomic<uint64_t>& attr_set, const DecodeArgs& a,
                                 int mrows, int budget, int ctas, bool pdl, cudaStream_t st) {
  // the attribute only caps the launch size; occupancy follows the size passed at launch
  {
    const cudaError_t e = smem_attr_once_per_device(kern, 200 * 1024, attr_set);
    if (e != cudaSuccess) return e;
  }
  DecodeArgs b = a;
  b.nw = L::num_stages(mrows, budget);
  b.pdl = pdl ? 1 : 0;
  // persistent: at most the CTAs that are resident at once; each walks
  // groups blockIdx.x, + gridDim.x, ...
  const int64_t slots = (int64_t)num_sms() * ctas;
  // with pdl, the CTAs may start while the previous kernel on the stream
  // (the quantize kernel) runs, streaming their first weight stages meanwhile
  const dim3 grid((unsigned)(a.G < slots ? a.G : slots)), block(32 * (kCompWarps + 2));
  // the activation rows and (W4A8) block sums of a stage, one box each
  CUtensorMap tx, ts;
  memset(&ts, 0, sizeof(ts));
  if (!make_tmap_rows(&tx, a.qa, a.M, a.K, L::kARow / 8, (uint32_t)mrows))
    return cudaErrorNotSupported;
  if (kQ4K && !make_tmap_rows(&ts, a.bsum, a.M, (int64_t)(a.K / kBlk) * 4, L::kSBlk / 2,
                              (uint32_t)mrows))
    return cudaErrorNotSupported;
  return launch_kernel(kern, grid, block, (size_t)L::total(mrows, b.nw), st, pdl, tx, ts, b);
}

template <int TT, bool kQ4K, bool kDebug>
static cudaError_t launch_decode_mma(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  using L = DecodeSmem<TT, kQ4K, false>;
  // two-tile kernels (9..16 rows) carry twice the activation rows and stash
  constexpr int kBudget = (TT == 2 && dec_ctas<kQ4K, TT>() != 2) ? QG_DEC_BUDGET_TT2_KB * 1024
                                                                  : dec_smem_budget<kQ4K, TT>();
  static std::atomic<uint64_t> attr_set{0};
  return launch_decode<L, kQ4K>(decode_gemm_kernel<TT, kQ4K, kDebug>, attr_set, a,
                                a.M < TT * 8 ? a.M : TT * 8, kBudget, dec_ctas<kQ4K, TT>(), pdl,
                                st);
}

template <bool kQ4K, int kM, bool kDebug>
static cudaError_t launch_decode_dp4a_m(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  using L = DecodeSmem<1, kQ4K, true, (kM + 1) / 2>;
  static std::atomic<uint64_t> attr_set{0};
  return launch_decode<L, kQ4K>(decode_dp4a_kernel<kQ4K, kM, kDebug>, attr_set, a, kM,
                                dec_smem_budget<kQ4K, 0>(), dec_ctas<kQ4K, 0>(), pdl, st);
}

template <bool kQ4K, bool kDebug>
static cudaError_t launch_decode_dp4a(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  static_assert(kDp4aMaxM == 4, "one instantiation per row count");
  switch (a.M) {
    case 1: return launch_decode_dp4a_m<kQ4K, 1, kDebug>(a, pdl, st);
    case 2: return launch_decode_dp4a_m<kQ4K, 2, kDebug>(a, pdl, st);
    case 3: return launch_decode_dp4a_m<kQ4K, 3, kDebug>(a, pdl, st);
    default: return launch_decode_dp4a_m<kQ4K, 4, kDebug>(a, pdl, st);
  }
}

template <bool kQ4K, bool kDebug>
static cudaError_t launch_decode_m(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  if (a.M <= dec_dp4a_max_m<kQ4K>()) return launch_decode_dp4a<kQ4K, kDebug>(a, pdl, st);
  if (a.M <= 8) return launch_decode_mma<1, kQ4K, kDebug>(a, pdl, st);
  return launch_decode_mma<2, kQ4K, kDebug>(a, pdl, st);
}

cudaError_t launch_decode_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                               const void* packed, int64_t N, void* out, bool out_f32,
                               int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                               cudaStream_t st) {
  const Q8Layout Lq(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  DecodeArgs a{};
  a.qa = qa; a.sa = sa; a.bsum = nullptr;
  a.wstream = base + Lq.off_stream;
  a.wscale = base + Lq.off_dsc;
  a.out = out; a.ldo = ldo; a.dbg = dbg; a.err = err;
  a.M = (int)M; a.K = (int)K; a.N = (int)N; a.G = (int)Lq.G;
  a.out_f32 = out_f32 ? 1 : 0;
  return dbg ? launch_decode_m<false, true>(a, false, st) : launch_decode_m<false, false>(a, pdl, st);
}

cudaError_t launch_decode_q4k(const int8_t* qa, const float* sa, const int32_t* asum, int64_t M,
                              int64_t K, const void* packed, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                              cudaStream_t st) {
  const Q4kLayout Lq(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  DecodeArgs a{};
  a.qa = qa; a.sa = sa; a.bsum = asum;
  a.wstream = base + Lq.off_stream;
  a.wscale = base + Lq.off_shdr;
  a.out = out; a.ldo = ldo; a.dbg = dbg; a.err = err;
  a.M = (int)M; a.K = (int)K; a.N = (int)N; a.G = (int)Lq.G;
  a.out_f32 = out_f32 ? 1 : 0;
  return dbg ? launch_decode_m<true, true>(a, false, st) : launch_decode_m<true, false>(a, pdl, st);
}

}  // namespace qg
