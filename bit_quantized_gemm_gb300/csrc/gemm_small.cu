// gemm_small.cu -- decode (small-M) GEMMs that stream the packed weights once.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and a fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit" and "The released files as they
// are"; "How it works": int8 tensor cores with exact int32 sums).
//
// Design. For M <= 16 the layer is bound by reading the weights from HBM
// (1.0625 B/weight for Q8_0, 0.5625 B/weight for Q4_K). A CTA owns one group
// of 16 weight rows and all of K; K is cut into stages of 16 blocks.
//   * warp 0 (one thread) streams each stage -- the group's contiguous
//     fragment-order weights and scales, the activation rows (and for W4A8
//     their block sums) -- into a shared-memory ring with 1-D bulk copies
//     (cp.async.bulk + mbarrier transaction counts);
//   * warps 1..8 split the stage's blocks (two each): per block one 16-byte
//     shared load gives the A fragments of two m16n8k16 fp16 MMAs (biased
//     int8 bytes widened to exact fp16 by byte permutes and one packed
//     subtract; Q4_K nibbles by shift-and-mask), one 8-byte load per 8-token
//     tile the token fragment (int8 rows padded to 544 bytes:
//     conflict-free), and the two MMAs sum the block exactly in fp32 from
//     zero (|sum| < 2^20). The exact block sums go to a shared stash. (This
//     GPU runs legacy fp16 MMAs at 4x the rate of legacy int8 MMAs, which
//     are no faster than dp4a, so int8 values travel as fp16 here);
//   * warp 9 applies acc = fmaf(isum, d, acc) (Q4_K: then
//     fmaf(-asum, dmin*m, acc)) over the stage's blocks in ascending order
//     with packed f32x2 FMAs -- the same chain as the prefill kernel, so both
//     paths give identical bits -- and hands the stage back to the producer.
// K-parallel compute with a sequential fp32 chain keeps ten warps busy per
// 16-row group, which small N (few groups) needs to reach HBM rate.
// As the GEMM of the layer call the kernel is a programmatic dependent of the
// quantize kernel: it starts while the rows are quantized, requests its first
// weight stages, and copies activations only once the quantize grid is done.
#include "qg_common.cuh"

namespace qg {

constexpr int kCompWarps = 8;      // compute warps per CTA

// K blocks per pipeline stage: 16 for both formats (8 KB of Q8_0 weights,
// 4 KB of Q4_K nibbles per 16-row group). Q4_K once took 32 to halve the
// per-stage overhead, but its stash then left room for two stages in
// flight: 16 blocks measured 43 % faster at 16 rows, equal at 1 and 8.
#ifndef QG_DEC_SBLK_Q8
#define QG_DEC_SBLK_Q8 16
#endif
// CTAs of 320 threads resident per SM (registers and shared memory are
// budgeted for it)
#ifndef QG_DEC_CTAS_Q4K
#define QG_DEC_CTAS_Q4K 3
#endif
template <bool kQ4K>
__host__ __device__ constexpr int dec_ctas() { return kQ4K ? QG_DEC_CTAS_Q4K : 3; }
template <bool kQ4K>
constexpr int dec_smem_budget() { return dec_ctas<kQ4K>() == 2 ? 110 * 1024 : 70 * 1024; }
// Blocks a compute warp converts before their MMAs, and blocks whose sums the
// chain warp loads before their FMAs: all of a warp's blocks / 4 for Q8_0,
// one at a time for Q4_K (whose conversions and sub-block terms need the
// registers; batching measured slower there).
#ifndef QG_DEC_CB_Q4K
#define QG_DEC_CB_Q4K 1
#endif
template <bool kQ4K>
__host__ __device__ constexpr int dec_cbatch() { return kQ4K ? QG_DEC_CB_Q4K : 32; }
#ifndef QG_DEC_HB_Q4K
#define QG_DEC_HB_Q4K 1
#endif
template <bool kQ4K>
__host__ __device__ constexpr int dec_hbatch() { return kQ4K ? QG_DEC_HB_Q4K : 4; }
#ifndef QG_DEC_BUDGET_TT2_KB
#define QG_DEC_BUDGET_TT2_KB 70
#endif
#ifndef QG_DEC_CHAIN_UNROLL
#define QG_DEC_CHAIN_UNROLL 1  // chain warp: a full stage's block quads unrolled
#endif
#ifndef QG_DEC_SBLK_Q4K
#define QG_DEC_SBLK_Q4K 16
#endif
template <bool kQ4K>
__host__ __device__ constexpr int sblk() { return kQ4K ? QG_DEC_SBLK_Q4K : QG_DEC_SBLK_Q8; }
// bytes per activation row in a stage: 32 per block + 32 of padding, so the
// eight rows one 8-byte load touches fall in distinct banks
template <bool kQ4K>
__host__ __device__ constexpr int arow() { return sblk<kQ4K>() * 32 + 32; }

__device__ __forceinline__ void bulk_copy(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory layout (offsets depend on M, fixed at launch):
//   NW weight stages, each: weights | scales | M activation rows | (W4A8) M
//   block-sum rows -- released by the chain warp;
//   2 stash slots of exact block sums between compute and chain warps;
//   barriers full[NW], empty[NW], xfull[2], xempty[2].
template <int TT, bool kQ4K>
struct DecodeSmem {
  static constexpr int kSBlk = sblk<kQ4K>();
  static constexpr int kARow = arow<kQ4K>();
  static constexpr int kWBytes = kSBlk * (kQ4K ? 256 : 512);  // weights per stage
  static constexpr int kSBytes = kQ4K ? kSBlk / 8 * 256 : kSBlk / 4 * 128;  // scales / headers
  static constexpr int kXBytes = kSBlk * TT * 32 * 16;          // exact sums of a stash slot
  // Q4_K: the exact sub-block scales (d*sc, dmin*m) of the 16 rows, per block,
  // decoded by the compute warps so the chain warp only loads them
  static constexpr int kScBytes = kQ4K ? kSBlk * 16 * 8 : 0;
  static constexpr int kSlotBytes = kXBytes + kScBytes;
  static constexpr int kMaxNw = 8;
  static __host__ __device__ int stage_bytes(int mrows) {
    return (int)align_up(kWBytes + kSBytes + mrows * kARow + (kQ4K ? mrows * kSBlk * 4 : 0), 128);
  }
  static __host__ __device__ int act_off() { return kWBytes + kSBytes; }
  static __host__ __device__ int bsum_off(int mrows) { return kWBytes + kSBytes + mrows * kARow; }
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

// 6-bit field f (0..15: sc_0..7 then m_0..7) of a Q4_K super-block header
// held as 16 bytes (d, dmin, then a 96-bit little-endian string of fields in
// words y, z, w), as a float (exact)
__device__ __forceinline__ float q4k_field(const uint4& H, int f) {
  const uint64_t lo = (uint64_t)H.y | ((uint64_t)H.z << 32);
  const int pos = 6 * f;
  uint32_t v;
  if (pos + 6 <= 64) v = (uint32_t)(lo >> pos);
  else if (pos >= 64) v = H.w >> (pos - 64);
  else v = (uint32_t)(lo >> pos) | (H.w << (64 - pos));
  return (float)(v & 63u);
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

template <int TT, bool kQ4K, bool kDebug>
__global__ void __launch_bounds__(32 * (kCompWarps + 2), dec_ctas<kQ4K>()) decode_gemm_kernel(const DecodeArgs a) {
  using L = DecodeSmem<TT, kQ4K>;
  constexpr int kSBlk = L::kSBlk;
  constexpr int kARow = L::kARow;
  constexpr int kBlkPerWarp = kSBlk / kCompWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  const int NW = a.nw;
  const int mrows = min(a.M, TT * 8);
  const int SBY = L::stage_bytes(mrows);
  float* stash_base = reinterpret_cast<float*>(smem + NW * SBY);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NW * SBY + 2 * L::kSlotBytes);
  uint64_t* empty = full + NW;    // weight stage consumed by the chain warp
  uint64_t* xfull = empty + NW;   // stash slot written (count: compute warps)
  uint64_t* xempty = xfull + 2;   // stash slot read by the chain warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.K / kBlk;
  const int B4 = (B + 3) & ~3;
  const int J = B / 8;
  const int nstages = (B + kSBlk - 1) / kSBlk;
  const int M = a.M;
  const int gr = lane >> 2, c = lane & 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xfull[i], kCompWarps);
      mbar_init(&xempty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    // The activation rows (and W4A8 block sums) of stage r into ring slot `slot`.
    auto copy_acts = [&](int r, int slot) {
      const int blk0 = r * kSBlk;
      const int nb = min(kSBlk, B - blk0);
      uint8_t* base = smem + slot * SBY;
      for (int m = lane; m < mrows; m += 32) {
        bulk_copy(base + L::act_off() + m * kARow,
                  a.qa + (int64_t)m * a.K + (int64_t)blk0 * kBlk, nb * 32, &full[slot]);
        if (kQ4K)
          bulk_copy(base + L::bsum_off(mrows) + m * (kSBlk * 4), a.bsum + (int64_t)m * B + blk0,
                    nb * 4, &full[slot]);
      }
    };
    // Launched as a programmatic dependent, the weights and scales of the
    // first P stages are requested before any activation: the quantize
    // kernel may still be writing the activations, and griddep_wait()
    // returns once it has completed. P is at most 3: every CTA's first three
    // stages are ~1 us of HBM time, about what a decode-sized quantize
    // lasts; more would still be arriving when the activations are
    // requested, and stage 0's activations would queue behind them. An
    // ordinary launch requests each stage's activations right after its
    // weights.
    // The CTA's groups are g = blockIdx.x, + gridDim.x, ... (grid capped at
    // the resident CTAs): the ring streams from one group into the next
    // without draining. The activation slices are the same for every group.
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
      bytes += mrows * nb * 32;
      if (kQ4K) bytes += mrows * nb * 4;
      if (lane == 0) {
        ok = mbar_wait(&empty[st], ph ^ 1, a.err);
        if (ok) {
          mbar_arrive_expect_tx(&full[st], bytes);
          if (!kQ4K) {
            bulk_copy(base, a.wstream + (g * B + blk0) * 512, nb * 512, &full[st]);
            bulk_copy(base + L::kWBytes, a.wscale + (g * (B4 / 4) + blk0 / 4) * 128,
                      ((nb + 3) / 4) * 128, &full[st]);
          } else {
            bulk_copy(base, a.wstream + (g * (B / 2) + blk0 / 2) * 512, nb * 256, &full[st]);
            bulk_copy(base + L::kWBytes, a.wscale + (g * J + blk0 / 8) * 256, (nb / 8) * 256,
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
    return;
  }

  if (warp <= kCompWarps) {
    // ------------------------------------------------------ compute warps
    const int cw = warp - 1;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
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
      // this warp's blocks: fragments of all of them first (rows past nb
      // of a short last stage compute unused sums that are never stored),
      // so the blocks' load and MMA latencies overlap
      constexpr int kCB = dec_cbatch<kQ4K>() < kBlkPerWarp ? dec_cbatch<kQ4K>() : kBlkPerWarp;
#pragma unroll
      for (int u0 = 0; u0 < kBlkPerWarp; u0 += kCB) {
      uint32_t a0[kCB][4], a1[kCB][4];  // A fragments, k 0-15 / 16-31
#pragma unroll
      for (int u = 0; u < kCB; ++u) {
        const int j = cw * kBlkPerWarp + u0 + u;
        if (!kQ4K) {
          const uint4 w = *reinterpret_cast<const uint4*>(base + j * 512 + lane * 16);
          // x: row n0 k 8c..+3, y: row n1 k 8c..+3, z: n0 k 8c+4..+7, w: n1 k 8c+4..+7
          biased_u8x4_to_f16x4(w.x, a0[u][0], a0[u][2]);
          biased_u8x4_to_f16x4(w.y, a0[u][1], a0[u][3]);
          biased_u8x4_to_f16x4(w.z, a1[u][0], a1[u][2]);
          biased_u8x4_to_f16x4(w.w, a1[u][1], a1[u][3]);
        } else {
          const uint2 w =
              *reinterpret_cast<const uint2*>(base + (j >> 1) * 512 + lane * 16 + (j & 1) * 8);
          a0[u][0] = nib_pair_to_f16x2<0>(w.x);
          a0[u][1] = nib_pair_to_f16x2<4>(w.x);
          a0[u][2] = nib_pair_to_f16x2<8>(w.x);
          a0[u][3] = nib_pair_to_f16x2<12>(w.x);
          a1[u][0] = nib_pair_to_f16x2<0>(w.y);
          a1[u][1] = nib_pair_to_f16x2<4>(w.y);
          a1[u][2] = nib_pair_to_f16x2<8>(w.y);
          a1[u][3] = nib_pair_to_f16x2<12>(w.y);
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const int mrow = 8 * t + gr;  // token of this lane's B fragment
#pragma unroll
        for (int u = 0; u < kCB; ++u) {
          const int j = cw * kBlkPerWarp + u0 + u;
          uint32_t b00 = 0, b01 = 0, b10 = 0, b11 = 0;
          if (mrow < M) {
            const uint2 bv = *reinterpret_cast<const uint2*>(
                base + L::act_off() + mrow * kARow + c * 8 + j * 32);
            biased_u8x4_to_f16x4(bv.x ^ 0x80808080u, b00, b01);
            biased_u8x4_to_f16x4(bv.y ^ 0x80808080u, b10, b11);
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
      if (kQ4K && lane < 16) {
        // this warp's blocks: row `lane`'s d*sc and dmin*m (exact products)
        float2* scw = reinterpret_cast<float2*>(stash + L::kXBytes / 4);
#pragma unroll
        for (int u = 0; u < kBlkPerWarp; ++u) {
          const int j = cw * kBlkPerWarp + u;
          if (j < nb) {
            const uint4 H = *reinterpret_cast<const uint4*>(base + L::kWBytes + (j >> 3) * 256 +
                                                            lane * 16);
            const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&H.x));
            scw[j * 16 + lane] = make_float2(dd.x * q4k_field(H, j & 7), dd.y * q4k_field(H, 8 + (j & 7)));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xfull[xs]);
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
    const uint8_t* sb = base + L::kWBytes;
    const int32_t* bb = reinterpret_cast<const int32_t*>(base + L::bsum_off(mrows));
    const float* stash = stash_base + xs * (L::kSlotBytes / 4);
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
      mbar_arrive(&empty[st]);
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

template <int TT, bool kQ4K, bool kDebug>
static cudaError_t launch_decode_cfg(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  using L = DecodeSmem<TT, kQ4K>;
  // two-tile kernels (9..16 rows) carry twice the activation rows and stash
  constexpr int kBudget = TT == 2 ? QG_DEC_BUDGET_TT2_KB * 1024 : dec_smem_budget<kQ4K>();
  auto kern = decode_gemm_kernel<TT, kQ4K, kDebug>;
  // the attribute only caps the launch size; occupancy follows the size passed at launch
  static std::atomic<uint64_t> attr_set{0};
  {
    const cudaError_t e = smem_attr_once_per_device(kern, 200 * 1024, attr_set);
    if (e != cudaSuccess) return e;
  }
  DecodeArgs b = a;
  const int mrows = a.M < TT * 8 ? a.M : TT * 8;
  b.nw = L::num_stages(mrows, kBudget);
  b.pdl = pdl ? 1 : 0;
  // persistent: at most the CTAs that are resident at once; each walks
  // groups blockIdx.x, + gridDim.x, ...
  const int64_t slots = (int64_t)num_sms() * dec_ctas<kQ4K>();
  dim3 grid((unsigned)(a.G < slots ? a.G : slots)), block(32 * (kCompWarps + 2));
  if (!pdl) {
    kern<<<grid, block, L::total(mrows, b.nw), st>>>(b);
    return cudaGetLastError();
  }
  // programmatic dependent launch: the CTAs may start while the previous
  // kernel on the stream (the quantize kernel) runs, streaming their first
  // weight stages meanwhile
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = (size_t)L::total(mrows, b.nw);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, b);
}

template <bool kQ4K, bool kDebug>
static cudaError_t launch_decode_m(const DecodeArgs& a, bool pdl, cudaStream_t st) {
  if (a.M <= 8) return launch_decode_cfg<1, kQ4K, kDebug>(a, pdl, st);
  return launch_decode_cfg<2, kQ4K, kDebug>(a, pdl, st);
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
