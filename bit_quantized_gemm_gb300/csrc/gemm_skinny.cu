// gemm_skinny.cu -- W8A8 and W4A8 GEMM tiles of 16 weight rows on legacy fp16 MMA.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and the fixed ascending-block fp32 epilogue (StartLux-Prism README,
// "Why StartLux-Prism": "Reproducible to the bit"; "How it works": int8
// tensor cores with exact int32 sums, W4A8 as 4-bit weights against 8-bit
// activations) -- the same chain as the other kernels, so all give identical
// bits: W8A8 one fma(isum, d, acc) per block, W4A8 fma(isum, d*sc, acc) then
// fma(-asum, dmin*m, acc) per 32-wide sub-block.
//
// Use: work that the tensor-memory kernel can only cut into narrow tiles --
// the weight rows left over after whole waves of 256-token tiles, and GEMMs
// whose weight-row tiles cannot fill the SMs. There each 32-block step of a
// narrow tile pays a fixed barrier round trip (~400 cycles). Here a CTA owns
// 16 weight rows x TB tokens, and every compute warp owns 16 tokens (32 in
// 64-token tiles). Each warp sums a block exactly with two m16n8k16 fp16 MMAs
// per 8 tokens and applies that block's FMAs at once, in registers: no
// accumulator hand-off at all.
//   * operands: the fp16 copies of the weights ([N][K], from the packed
//     buffer; Q4_K: the 4-bit values) and activations (q16 [M][K]) arrive by
//     TMA, 64 K (two blocks) per stage, 128-byte swizzle; fragments come out
//     with ldmatrix;
//   * one producer warp (lane 0) runs the ring; the compute warps hand each
//     stage back per thread (no warp-wide operation on the path);
//   * per-block operands of the FMAs -- weight scales d[n][b] (W4A8: d*sc and
//     dmin*m) from the fp32 scale rows and, for W4A8, the activation block
//     sums of the lane's four tokens -- a stage's two blocks per 8-byte load,
//     fetched several stages ahead into fixed register slots (one stage ahead
//     left the loads' latency exposed).
#include <cuda.h>

#include <cstring>

#include "qg_common.cuh"

namespace qg {

// from gemm_large.cu
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows);
bool make_tmap_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                    uint32_t box_words, uint32_t box_rows);

constexpr int kSkRows = 16;  // weight rows per CTA (the MMA's M)
constexpr int kSkBK = 64;    // K per stage: two blocks, one 128-byte swizzle row

// kTT = n8 token tiles per compute warp: 4 (32 tokens) in the 64-token tile
// of a GEMM of at most 64 tokens (each weight fragment feeds four MMAs: fewer
// fragment loads per token on the L1 data pipe that bounds these tiles;
// 17408 -> 5120 at 64 tokens 82.5 -> 78.0 us), else 2 (16 tokens: a 32-token
// tile with one warp, 128-token tiles, and the 256 64-token CTAs of the 4B
// down projection's tail all measured slower with 32-token warps)
template <int TB, bool kQ4K, int kTT>
struct SkinnyCfg {
  static_assert(TB % 16 == 0 && TB >= 16 && TB <= 256, "token tile");
  static_assert(kTT == 2 || kTT == 4, "token tiles per warp");
  static constexpr int kWarps = TB / (8 * kTT);  // compute warps, 8 * kTT tokens each
  static constexpr int kThreads = 32 * (kWarps + 1);
  static constexpr uint32_t kABytes = kSkRows * kSkBK * 2;  // 2 KB
  static constexpr uint32_t kBBytes = TB * kSkBK * 2;
  static constexpr uint32_t kTileBytes = kABytes + kBBytes;  // multiple of 1024 (swizzle atoms)
  // every even stage also brings the per-block FMA operands of four blocks
  // (its own two and the next stage's), 16 bytes per row: the 16 weight rows'
  // scales d (W4A8: d*sc, and dmin*m) and, W4A8, the TB tokens' activation
  // block sums; they land in the stage's operand slot, kept apart from the
  // tiles (slots 128-byte aligned, each box 128-byte aligned in its slot)
  static constexpr uint32_t kSdOff = 0;
  static constexpr uint32_t kSmOff = 256;
  static constexpr uint32_t kSsOff = 512;
  static constexpr uint32_t kSBytes = kQ4K ? 512 + TB * 16 : 256;
  static constexpr uint32_t kSSlot = (kSBytes + 127) / 128 * 128;
  static constexpr uint32_t kPerStage = kTileBytes + kSSlot;
  // resident CTAs per SM: three of 64 tokens (a shallower ring: 7 stages),
  // else two; 17408 -> 5120 at 33-64 tokens (320 CTAs) then runs as one wave
  static constexpr int kCtas = TB == 64 ? 3 : 2;
  static constexpr int kBudget = kCtas == 3 ? 74 * 1024 : 96 * 1024;
  static constexpr int kStages = kBudget / (int)kPerStage > 8 ? 8 : kBudget / (int)kPerStage;
  static constexpr size_t kSmem = kStages * kPerStage + 2 * kStages * 8 + 1024;
  static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kStages >= 2, "ring depth");
};

struct SkinnyArgs {
  const float* d32;  // [N][ldd] fp32 weight scales (rows padded to whole quads); W4A8: d*sc
  const float* dm32;     // W4A8: dmin*m [N][ldd]
  const int32_t* bsum;   // W4A8: [M][K/32] activation block sums
  const float* sa;   // [M] activation scales
  void* out;
  int64_t ldo, ldd;
  int M, N, K;
  int out_f32;
  int pdl;  // launched as a programmatic dependent of the quantize kernel
  uint32_t* err;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// byte offset of the 16-byte chunk holding element k of row r in a tile of
// 128-byte rows written by TMA with 128-byte swizzle (chunk index ^ row % 8)
__device__ __forceinline__ uint32_t sw128(int r, int k) {
  return (uint32_t)(r * 128 + ((((k >> 3) ^ r) & 7) << 4));
}

template <int TB, bool kQ4K, int kTT>
__global__ void __launch_bounds__(SkinnyCfg<TB, kQ4K, kTT>::kThreads, SkinnyCfg<TB, kQ4K, kTT>::kCtas)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD,
                       const __grid_constant__ CUtensorMap tmM,
                       const __grid_constant__ CUtensorMap tmS, const SkinnyArgs args) {
  using C = SkinnyCfg<TB, kQ4K, kTT>;
  constexpr int kW = C::kWarps;
  constexpr int kS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* const sops = sm + kS * C::kTileBytes;  // the stages' operand slots
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kS * C::kPerStage);
  uint64_t* empty = full + kS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = args.M, N = args.N, K = args.K;
  const int n0 = blockIdx.x * kSkRows, m0 = blockIdx.y * TB;
  const int NB = K / kBlk, NS = (NB + 1) / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kW * 32);  // every compute thread hands the stage back
    }
    fence_barrier_init();
  }
  if (warp == kW && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    if (kQ4K) {
      tma_prefetch_desc(&tmM);
      tma_prefetch_desc(&tmS);
    }
  }
  __syncthreads();

  if (warp == kW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      // as a programmatic dependent of the quantize kernel: the weight tiles
      // of the first P stages before the wait for its grid, their activation
      // tiles after it (W4A8 stages carry activation block sums: wait first)
      const int P = (args.pdl && !kQ4K) ? min(min(NS, kS), 3) : 0;
      if (kQ4K && args.pdl) griddep_wait();
      for (int s = 0; s < NS && ok; ++s) {
        ok = mbar_wait(&empty[st], ph ^ 1, args.err);
        if (!ok) break;
        // the compute warps read the slot through the generic proxy
        // (ldmatrix); the TMA loads below rewrite it through the async proxy.
        // Without this fence such a load could land before those reads
        // (measured: wrong sums for a warp in a few CTAs when three CTAs
        // shared an SM)
        fence_proxy_async_smem();
        uint8_t* a_s = sm + st * C::kTileBytes;
        uint8_t* o_s = sops + st * C::kSSlot;
        const bool ops = (s & 1) == 0;  // this stage brings four blocks' FMA operands
        // whole boxes (zero-filled edges)
        mbar_arrive_expect_tx(&full[st], C::kABytes + C::kBBytes + (ops ? C::kSBytes : 0));
        tma_load_2d(a_s, &tmA, &full[st], s * kSkBK, n0);
        if (ops) {
          // x in 8-byte words: blocks 2s..2s+3 start at word s (even: 16-byte aligned)
          tma_load_2d(o_s + C::kSdOff, &tmD, &full[st], s, n0);
          if (kQ4K) {
            tma_load_2d(o_s + C::kSmOff, &tmM, &full[st], s, n0);
            tma_load_2d(o_s + C::kSsOff, &tmS, &full[st], s, m0);
          }
        }
        if (s >= P) tma_load_2d(a_s + C::kABytes, &tmB, &full[st], s * kSkBK, m0);
        if (s + 1 == P) {
          griddep_wait();
          for (int r = 0; r < P; ++r)
            tma_load_2d(sm + r * C::kTileBytes + C::kABytes, &tmB, &full[r], r * kSkBK, m0);
        }
        if (++st == kS) { st = 0; ph ^= 1; }
      }
      // every stage handed back before the CTA exits (no copy in flight)
      for (int i = 0; i < kS && ok; ++i) {
        if (!mbar_wait(&empty[st], ph ^ 1, args.err)) break;
        if (++st == kS) { st = 0; ph ^= 1; }
      }
    }
    return;
  }

  // ------------------------------------------------------------- compute
  const int g = lane >> 2, t = lane & 3;
  const int nA = n0 + g, nB = n0 + g + 8;  // this lane's two weight rows
  // ldmatrix row addresses: lane l serves row l % 8 of matrix l / 8
  const int mi = lane >> 3, ri = lane & 7;
  const int a_row = ri + 8 * (mi & 1), a_k = 8 * (mi >> 1);      // A: rows 0-15, k 0-15
  // B: 16 tokens per x4 load (matrices 2, 3: tokens 8-15; 1, 3: k 8-15)
  const int b_row = 8 * kTT * warp + ri + 8 * (mi >> 1), b_k = 8 * (mi & 1);
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  float2 acc[kTT][2];  // [token tile][row nA / nB]: tokens 2t, 2t+1 of the tile
#pragma unroll
  for (int i = 0; i < kTT; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

  // Per stage (two blocks): wait for the slot, sum each block exactly with
  // four MMAs, read the FMA operands that came with an even stage (this
  // lane's rows g, g+8 and tokens: four blocks, 16-byte loads, one wavefront
  // each), hand the slot back, then the blocks' FMAs in block order.
  float4 sdA = make_float4(0.f, 0.f, 0.f, 0.f), sdB = sdA, smA = sdA, smB = sdA;
  int4 ssv[kTT][2];  // [token tile][token 2t + e]: activation block sums of four blocks
  const int tl = 8 * kTT * warp + 2 * t;  // this lane's first token in the tile (then +1, +8, ...)
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int s = 0; s < NS && ok; ++s) {
    ok = mbar_wait(&full[st], ph, args.err);
    if (!ok) break;
    // both blocks' sums first (a missing second block of a K tail reads the
    // zero-filled box and is never used)
    float d[2][kTT][4];  // [block][token tile]: (nA, 2t), (nA, 2t+1), (nB, 2t), (nB, 2t+1)
    const uint8_t* sb = sm + st * C::kTileBytes;
    const uint8_t* ob = sops + st * C::kSSlot;
    {
      const uint32_t a_s = smem_u32(sb);
      const uint32_t b_s = a_s + C::kABytes;
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const int kc = jb * 32 + kh * 16;
          uint32_t af[4], bfr[kTT / 2][4];
          ldsm_x4(a_s + sw128(a_row, kc + a_k), af);
#pragma unroll
          for (int h = 0; h < kTT / 2; ++h) ldsm_x4(b_s + sw128(b_row + 16 * h, kc + b_k), bfr[h]);
          // bfr[h]: tile 2h (k 0-7, 8-15), tile 2h+1 (k 0-7, 8-15); a fresh sum per block
          float(&dd)[kTT][4] = d[jb];
#pragma unroll
          for (int tt = 0; tt < kTT; ++tt) {
            const uint32_t* bp = &bfr[tt / 2][2 * (tt & 1)];
            if (kh == 0)
              mma_f16_16816(dd[tt], af, bp[0], bp[1], zero4);
            else
              mma_f16_16816(dd[tt], af, bp[0], bp[1], dd[tt]);
          }
        }
      }
    }
    if ((s & 1) == 0) {
      sdA = *reinterpret_cast<const float4*>(ob + C::kSdOff + g * 16);
      sdB = *reinterpret_cast<const float4*>(ob + C::kSdOff + (g + 8) * 16);
      if constexpr (kQ4K) {
        smA = *reinterpret_cast<const float4*>(ob + C::kSmOff + g * 16);
        smB = *reinterpret_cast<const float4*>(ob + C::kSmOff + (g + 8) * 16);
#pragma unroll
        for (int tt = 0; tt < kTT; ++tt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            ssv[tt][e] = *reinterpret_cast<const int4*>(ob + C::kSsOff + (tl + 8 * tt + e) * 16);
      }
    }
    mbar_arrive(&empty[st]);  // this thread's reads of the stage are done
    if (++st == kS) { st = 0; ph ^= 1; }
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      if (2 * s + jb < NB) {
        // block 2s + jb is entry q of the four-block group
        const bool hi = (s & 1) != 0;
        const float dA = jb ? (hi ? sdA.w : sdA.y) : (hi ? sdA.z : sdA.x);
        const float dB = jb ? (hi ? sdB.w : sdB.y) : (hi ? sdB.z : sdB.x);
        const float2 dA2 = make_float2(dA, dA), dB2 = make_float2(dB, dB);
#pragma unroll
        for (int tt = 0; tt < kTT; ++tt) {
          acc[tt][0] = __ffma2_rn(make_float2(d[jb][tt][0], d[jb][tt][1]), dA2, acc[tt][0]);
          acc[tt][1] = __ffma2_rn(make_float2(d[jb][tt][2], d[jb][tt][3]), dB2, acc[tt][1]);
        }
        if constexpr (kQ4K) {
          // then the min term of the same sub-block: fma(-asum, dmin*m, acc)
          const float mA = jb ? (hi ? smA.w : smA.y) : (hi ? smA.z : smA.x);
          const float mB = jb ? (hi ? smB.w : smB.y) : (hi ? smB.z : smB.x);
          const float2 nmA2 = make_float2(-mA, -mA), nmB2 = make_float2(-mB, -mB);
#pragma unroll
          for (int tt = 0; tt < kTT; ++tt) {
            const int a0 = jb ? (hi ? ssv[tt][0].w : ssv[tt][0].y) : (hi ? ssv[tt][0].z : ssv[tt][0].x);
            const int a1 = jb ? (hi ? ssv[tt][1].w : ssv[tt][1].y) : (hi ? ssv[tt][1].z : ssv[tt][1].x);
            const float2 as = make_float2((float)a0, (float)a1);  // exact: |v| <= 4064
            acc[tt][0] = __ffma2_rn(as, nmA2, acc[tt][0]);
            acc[tt][1] = __ffma2_rn(as, nmB2, acc[tt][1]);
          }
        }
      }
    }
  }
  if (!ok) return;
  if (args.pdl) griddep_wait();  // the activation scales come from the quantize kernel
#pragma unroll
  for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = m0 + 8 * kTT * warp + 8 * tt + 2 * t + (e & 1);
      const int n = (e < 2) ? nA : nB;
      const float a = (e == 0) ? acc[tt][0].x : (e == 1) ? acc[tt][0].y
                    : (e == 2) ? acc[tt][1].x : acc[tt][1].y;
      if (m < M && n < N) {
        const float y = a * __ldg(args.sa + m);
        if (args.out_f32)
          reinterpret_cast<float*>(args.out)[(int64_t)m * args.ldo + n] = y;
        else
          reinterpret_cast<uint16_t*>(args.out)[(int64_t)m * args.ldo + n] = f32_to_bf16_rne(y);
      }
    }
  }
}

template <int TB, bool kQ4K, int kTT = 2>
static cudaError_t launch_skinny_t(const uint16_t* wq16, const uint16_t* q16, const SkinnyArgs& a,
                                   cudaStream_t st) {
  using C = SkinnyCfg<TB, kQ4K, kTT>;
  CUtensorMap ta, tb, td, tm, ts;
  if (!make_tmap(&ta, wq16, a.N, a.K, kSkRows) || !make_tmap(&tb, q16, a.M, a.K, TB))
    return cudaErrorNotSupported;
  // per-block operands as rows of 8-byte words, boxes of 2 words (four
  // blocks) x 16 weight rows or TB tokens; rows hold whole quads of blocks
  const int64_t nb = a.K / kBlk;
  if (!make_tmap_rows(&td, a.d32, a.N, a.ldd * 4, 2, kSkRows)) return cudaErrorNotSupported;
  memset(&tm, 0, sizeof(tm));
  memset(&ts, 0, sizeof(ts));
  if (kQ4K && (!make_tmap_rows(&tm, a.dm32, a.N, a.ldd * 4, 2, kSkRows) ||
               !make_tmap_rows(&ts, a.bsum, a.M, nb * 4, 2, TB)))
    return cudaErrorNotSupported;
  auto kern = skinny_gemm_kernel<TB, kQ4K, kTT>;
  static std::atomic<uint64_t> attr_set{0};
  {
    const cudaError_t e = smem_attr_once_per_device(kern, (int)C::kSmem, attr_set);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)ceil_div(a.N, kSkRows), (unsigned)ceil_div(a.M, TB));
  return launch_kernel(kern, grid, dim3(C::kThreads), C::kSmem, st, a.pdl != 0, ta, tb, td, tm, ts,
                       a);
}

// Weight rows [0, N) of the packed-layout views passed in (the caller offsets
// wq16, d32 and out to its first row), all M tokens, in tiles of tb (32, 64
// or 128) tokens.
cudaError_t launch_skinny_q8_0(const uint16_t* q16, const float* sa, int64_t M, int64_t K,
                               const uint16_t* wq16, const float* d32, int64_t ldd, int64_t N,
                               void* out, bool out_f32, int64_t ldo, int tb, uint32_t* err,
                               bool pdl, cudaStream_t st) {
  SkinnyArgs a{};
  a.pdl = pdl ? 1 : 0;
  a.d32 = d32;
  a.ldd = ldd;
  a.sa = sa;
  a.out = out;
  a.ldo = ldo;
  a.M = (int)M; a.N = (int)N; a.K = (int)K;
  a.out_f32 = out_f32 ? 1 : 0;
  a.err = err;
  if (tb == 32) return launch_skinny_t<32, false>(wq16, q16, a, st);
  if (tb == 64)
    return M <= 64 ? launch_skinny_t<64, false, 4>(wq16, q16, a, st)
                   : launch_skinny_t<64, false, 2>(wq16, q16, a, st);
  return launch_skinny_t<128, false>(wq16, q16, a, st);
}

// W4A8 (Q4_K): the same tiles over the fp16 copy of the 4-bit values, with the
// sub-block scales d*sc and dmin*m (rows of ldd floats) and the activation
// block sums [M][K/32]; each block's two FMAs in the order of the other W4A8
// kernels (isum term, then min term). 32 or 64 tokens.
cudaError_t launch_skinny_q4k(const uint16_t* q16, const float* sa, const int32_t* bsum,
                              int64_t M, int64_t K, const uint16_t* wq16, const float* ds32,
                              const float* dm32, int64_t ldd, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int tb, uint32_t* err, bool pdl, cudaStream_t st) {
  SkinnyArgs a{};
  a.pdl = pdl ? 1 : 0;
  a.d32 = ds32;
  a.dm32 = dm32;
  a.bsum = bsum;
  a.ldd = ldd;
  a.sa = sa;
  a.out = out;
  a.ldo = ldo;
  a.M = (int)M; a.N = (int)N; a.K = (int)K;
  a.out_f32 = out_f32 ? 1 : 0;
  a.err = err;
  if (tb == 32) return launch_skinny_t<32, true>(wq16, q16, a, st);
  return launch_skinny_t<64, true, 4>(wq16, q16, a, st);  // at most 64 tokens
}

}  // namespace qg
