// gemm_skinny.cu -- W8A8 GEMM tiles of 16 weight rows on legacy fp16 MMA.
//
// Operation: the W8A8 (Q8_0) product with exact int32 block sums and the
// fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit"; "How it works": int8 tensor
// cores with exact int32 sums) -- the same chain as the other kernels, so all
// give identical bits.
//
// Use: work that the tensor-memory kernel can only cut into narrow tiles --
// the weight rows left over after whole waves of 256-token tiles, and GEMMs
// whose weight-row tiles cannot fill the SMs. There each 32-block step of a
// narrow tile pays a fixed barrier round trip (~400 cycles). Here a CTA owns
// 16 weight rows x TB tokens, and every compute warp owns 16 tokens. Each
// warp sums a block exactly with four m16n8k16 fp16 MMAs and applies that
// block's FMAs at once, in registers: no accumulator hand-off at all.
//   * operands: the fp16 copies of the weights ([N][K], from the packed
//     buffer) and activations (q16 [M][K]) arrive by TMA, 64 K (two blocks)
//     per stage, 128-byte swizzle; fragments come out with ldmatrix;
//   * one producer warp (lane 0) runs the ring; the compute warps hand each
//     stage back per thread (no warp-wide operation on the path);
//   * weight scales: d[n][b] from the fp32 scale rows, a stage's two blocks
//     per 8-byte load, fetched three stages ahead through a short register
//     pipeline (one stage ahead left the loads' latency exposed).
#include <cuda.h>

#include <type_traits>

#include "qg_common.cuh"

namespace qg {

// from gemm_large.cu
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows);

#ifndef QG_SK_SCALE_AHEAD
#define QG_SK_SCALE_AHEAD 3  // trips whose scales are loaded ahead of their use
#endif
#ifndef QG_SK_STAGES_PER_TRIP
#define QG_SK_STAGES_PER_TRIP 1  // stages whose blocks a compute warp sums before their FMAs
#endif
constexpr int kSkRows = 16;  // weight rows per CTA (the MMA's M)
constexpr int kSkBK = 64;    // K per stage: two blocks, one 128-byte swizzle row

template <int TB>
struct SkinnyCfg {
  static_assert(TB % 16 == 0 && TB >= 16 && TB <= 256, "token tile");
  static constexpr int kWarps = TB / 16;  // compute warps, 16 tokens each
  static constexpr int kThreads = 32 * (kWarps + 1);
  static constexpr uint32_t kABytes = kSkRows * kSkBK * 2;  // 2 KB
  static constexpr uint32_t kBBytes = TB * kSkBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;  // multiple of 1024 (swizzle atoms)
  // resident CTAs per SM: three of 64 tokens (a shallower ring: 7 stages),
  // else two; 17408 -> 5120 at 33-64 tokens (320 CTAs) then runs as one wave
  static constexpr int kCtas = TB == 64 ? 3 : 2;
  static constexpr int kBudget = kCtas == 3 ? 70 * 1024 : 96 * 1024;
  static constexpr int kStages = kBudget / (int)kStageBytes > 8 ? 8 : kBudget / (int)kStageBytes;
  static constexpr size_t kSmem = kStages * kStageBytes + 2 * kStages * 8 + 1024;
  static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kStages >= 2, "ring depth");
};

struct SkinnyArgs {
  const float* d32;  // [N][ldd] fp32 weight scales (rows padded to whole quads)
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

template <int TB>
__global__ void __launch_bounds__(SkinnyCfg<TB>::kThreads, SkinnyCfg<TB>::kCtas)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const SkinnyArgs args) {
  using C = SkinnyCfg<TB>;
  constexpr int kW = C::kWarps;
  constexpr int kS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kS * C::kStageBytes);
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
      // tiles after it
      const int P = args.pdl ? min(min(NS, kS), 3) : 0;
      for (int s = 0; s < NS && ok; ++s) {
        ok = mbar_wait(&empty[st], ph ^ 1, args.err);
        if (!ok) break;
        // the compute warps read the slot through the generic proxy
        // (ldmatrix); the TMA loads below rewrite it through the async proxy.
        // Without this fence such a load could land before those reads
        // (measured: wrong sums for a warp in a few CTAs when three CTAs
        // shared an SM)
        fence_proxy_async_smem();
        uint8_t* a_s = sm + st * C::kStageBytes;
        mbar_arrive_expect_tx(&full[st], C::kStageBytes);  // whole boxes (zero-filled edges)
        tma_load_2d(a_s, &tmA, &full[st], s * kSkBK, n0);
        if (s >= P) tma_load_2d(a_s + C::kABytes, &tmB, &full[st], s * kSkBK, m0);
        if (s + 1 == P) {
          griddep_wait();
          for (int r = 0; r < P; ++r)
            tma_load_2d(sm + r * C::kStageBytes + C::kABytes, &tmB, &full[r], r * kSkBK, m0);
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
  const float* drA = args.d32 + (int64_t)(nA < N ? nA : 0) * args.ldd;
  const float* drB = args.d32 + (int64_t)(nB < N ? nB : 0) * args.ldd;
  // ldmatrix row addresses: lane l serves row l % 8 of matrix l / 8
  const int mi = lane >> 3, ri = lane & 7;
  const int a_row = ri + 8 * (mi & 1), a_k = 8 * (mi >> 1);      // A: rows 0-15, k 0-15
  const int b_row = 16 * warp + ri + 8 * (mi >> 1), b_k = 8 * (mi & 1);  // B: 16 tokens
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  float2 acc[2][2];  // [token tile][row nA / nB]: tokens 2t, 2t+1 of the tile
#pragma unroll
  for (int i = 0; i < 2; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

  // kU stages (2*kU blocks) per trip: their sums first, so the blocks' MMA
  // chains overlap, then their FMAs in block order. The trip's scales are
  // loaded one trip ahead (kU = 1: 8-byte loads, a stage's first block is
  // even; kU = 2: 16-byte loads, a pair's first block is a multiple of 4;
  // rows are padded to whole quads)
  constexpr int kU = QG_SK_STAGES_PER_TRIP;
  static_assert(kU == 1 || kU == 2, "stages per trip");
  using ScaleV = typename std::conditional<kU == 2, float4, float2>::type;
  auto load_scales = [&](const float* p) -> ScaleV {
    if constexpr (kU == 2) return ldg_f32x4_pinned(p);
    else return ldg_f32x2_pinned(p);
  };
  // scales of the next kP trips in flight (a shift register of loads)
  constexpr int kP = QG_SK_SCALE_AHEAD;
  ScaleV pA[kP], pB[kP];
#pragma unroll
  for (int p = 0; p < kP; ++p) {
    if (2 * kU * p < NB) {
      pA[p] = load_scales(drA + 2 * kU * p);
      pB[p] = load_scales(drB + 2 * kU * p);
    }
  }
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int s = 0; s < NS && ok; s += kU) {
    const ScaleV cA = pA[0], cB = pB[0];
#pragma unroll
    for (int p = 0; p + 1 < kP; ++p) {
      pA[p] = pA[p + 1];
      pB[p] = pB[p + 1];
    }
    if (2 * (s + kU * kP) < NB) {
      pA[kP - 1] = load_scales(drA + 2 * (s + kU * kP));
      pB[kP - 1] = load_scales(drB + 2 * (s + kU * kP));
    }
    const int nst = (s + kU <= NS) ? kU : NS - s;  // stages in this trip
    int sts[kU];
    uint32_t phs[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      sts[q] = st;
      phs[q] = ph;
      if (q < nst && ++st == kS) { st = 0; ph ^= 1; }
    }
#pragma unroll
    for (int q = 0; q < kU; ++q)
      if (q < nst && ok) ok = mbar_wait(&full[sts[q]], phs[q], args.err);
    if (!ok) break;
    // every block's sums first (a missing second block of a K tail reads the
    // zero-filled box and is never used; a missing stage is not read)
    float d[2 * kU][2][4];  // [block][token tile]: (nA, 2t), (nA, 2t+1), (nB, 2t), (nB, 2t+1)
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      if (q < nst) {
        const uint32_t a_s = smem_u32(sm + sts[q] * C::kStageBytes);
        const uint32_t b_s = a_s + C::kABytes;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            const int kc = jb * 32 + kh * 16;
            uint32_t af[4], bfr[4];
            ldsm_x4(a_s + sw128(a_row, kc + a_k), af);
            ldsm_x4(b_s + sw128(b_row, kc + b_k), bfr);
            // bfr: tile 0 (k 0-7, 8-15), tile 1 (k 0-7, 8-15); a fresh sum per block
            float(&dd)[2][4] = d[2 * q + jb];
            if (kh == 0) {
              mma_f16_16816(dd[0], af, bfr[0], bfr[1], zero4);
              mma_f16_16816(dd[1], af, bfr[2], bfr[3], zero4);
            } else {
              mma_f16_16816(dd[0], af, bfr[0], bfr[1], dd[0]);
              mma_f16_16816(dd[1], af, bfr[2], bfr[3], dd[1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kU; ++q)
      if (q < nst) mbar_arrive(&empty[sts[q]]);  // this thread's reads of the stage are done
#pragma unroll
    for (int jb = 0; jb < 2 * kU; ++jb) {
      if (2 * s + jb < NB) {
        const float* fa = reinterpret_cast<const float*>(&cA);
        const float* fb = reinterpret_cast<const float*>(&cB);
        const float dA = fa[jb], dB = fb[jb];
        const float2 dA2 = make_float2(dA, dA), dB2 = make_float2(dB, dB);
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          acc[tt][0] = __ffma2_rn(make_float2(d[jb][tt][0], d[jb][tt][1]), dA2, acc[tt][0]);
          acc[tt][1] = __ffma2_rn(make_float2(d[jb][tt][2], d[jb][tt][3]), dB2, acc[tt][1]);
        }
      }
    }
  }
  if (!ok) return;
  if (args.pdl) griddep_wait();  // the activation scales come from the quantize kernel
#pragma unroll
  for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = m0 + 16 * warp + 8 * tt + 2 * t + (e & 1);
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

template <int TB>
static cudaError_t launch_skinny_t(const uint16_t* wq16, const uint16_t* q16, const SkinnyArgs& a,
                                   cudaStream_t st) {
  using C = SkinnyCfg<TB>;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, wq16, a.N, a.K, kSkRows) || !make_tmap(&tb, q16, a.M, a.K, TB))
    return cudaErrorNotSupported;
  auto kern = skinny_gemm_kernel<TB>;
  static std::atomic<uint64_t> attr_set{0};
  {
    const cudaError_t e = smem_attr_once_per_device(kern, (int)C::kSmem, attr_set);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)ceil_div(a.N, kSkRows), (unsigned)ceil_div(a.M, TB));
  return launch_kernel(kern, grid, dim3(C::kThreads), C::kSmem, st, a.pdl != 0, ta, tb, a);
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
  if (tb == 32) return launch_skinny_t<32>(wq16, q16, a, st);
  if (tb == 64) return launch_skinny_t<64>(wq16, q16, a, st);
  return launch_skinny_t<128>(wq16, q16, a, st);
}

}  // namespace qg
