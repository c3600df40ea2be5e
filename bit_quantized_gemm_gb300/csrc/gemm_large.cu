// gemm_large.cu -- prefill (large-M) GEMMs on the 5th-generation tensor cores.
//
// Operation: the W8A8 (Q8_0) and W4A8 (Q4_K) products with exact int32 block
// sums and a fixed ascending-block fp32 epilogue (StartLux-Prism README, "Why
// StartLux-Prism": "Reproducible to the bit"; "How it works": int8 tensor
// cores with exact int32 sums; the pages' own Hopper kernels used warpgroup
// MMA with TMA, "Supported models and GPUs").
//
// sm_103a has no int8 kind for tcgen05.mma, so the exact integer product runs
// as kind::f16 on integer-valued fp16 operands: int8 values (|q| <= 127) and
// 4-bit values are exact in fp16, every product (<= 16129) is exact, and one
// 32-wide block sum (|isum| <= 516128 < 2^20) is accumulated from zero in the
// fp32 tensor accumulator, which holds it exactly. Each block gets its own
// accumulator, so the tensor-memory value IS (float)isum and the epilogue is
// one FMA per (row, token, block), in block order -- the same chain as the
// decode kernel, so both paths give identical bits.
//
// Tile: 128 weight rows (MMA M, tensor-memory lanes) x BM tokens (MMA N,
// tensor-memory columns; BM = 256 for W8A8, 128 for W4A8), K staged 64 at a
// time (two blocks) through a TMA ring with 128-byte swizzle (as deep as
// shared memory allows; 3 stages at BM = 256). Block b of
// a tile accumulates in buffer b % kTBufs (two 256-column buffers at BM = 256:
// all 512 columns), so the MMA of block b+1 overlaps the epilogue of block b.
// Warp roles (352 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (lane 0); for W4A8 the whole warp also converts
//               the activation block sums of each block into a float ring
//   warps 1, 2  MMA issuers (lane 0): warp 1 the even blocks of each tile,
//               warp 2 the odd ones -- two issuers, so that one's barrier
//               latencies overlap the other's work; warp 1 also allocates
//               tensor memory
//   warps 3..10 epilogue: warp w reads lanes 32*(w%4).. of tensor memory and
//               half (w-3)/4 of the token columns; each thread keeps its fp32
//               accumulators (one weight row x its tokens) in registers and
//               applies acc = fma(isum, d, acc) with packed f32x2 FMAs. Each
//               thread hands its part of a buffer back itself, as soon as its
//               loads are done (no warp-wide operation on this path).
//
// Waves: a GEMM whose 256-token tiles leave the last wave of SMs mostly idle
// runs as two launches -- the weight-row tiles that fill whole waves with
// 256-token tiles, then the remaining rows over all tokens, either as narrow
// tensor-memory tiles (32..128 tokens) or as the 16-row tiles of
// gemm_skinny.cu (legacy fp16 MMA), whichever a per-step cycle table
// predicts faster; small GEMMs may run as narrow or 16-row tiles alone.
// Every output element still gets its whole K chain from one thread, so the
// plan changes no bit.
#include <cuda.h>
#include <algorithm>
#include <cstring>

#include "qg_common.cuh"

namespace qg {

#ifndef QG_STAGES
#define QG_STAGES 0  // TMA ring depth; 0: as many as fit (3 at BM = 256 with output staging)
#endif
#ifndef QG_OUT_CHUNK
#define QG_OUT_CHUNK 128  // output columns per trip of the output loop (>= kColsPerThread: unrolled)
#endif
#ifndef QG_TMA_OUT
#define QG_TMA_OUT 1  // bf16 outputs staged in shared memory and stored by TMA
#endif
#ifndef QG_CTAS_PER_SM
#define QG_CTAS_PER_SM 1
#endif
#ifndef QG_EPI_WARPS
#define QG_EPI_WARPS 8
#endif
#ifndef QG_SKINNY
#define QG_SKINNY 0
#endif
#ifndef QG_FORCE_BM
#define QG_FORCE_BM 0  // tuning: nonzero runs every W8A8 GEMM as one launch of this width
#endif
#ifndef QG_BM_W4A8
#define QG_BM_W4A8 0  // W4A8 token-tile width above 64 tokens (0: chosen per shape)
#endif
#ifndef QG_EPI_BATCH
#define QG_EPI_BATCH 0  // loads per wait; 0: all chunks of a block up to 64 columns, else 1
#endif
#ifndef QG_CHUNK
#define QG_CHUNK 16  // tensor-memory columns per load (16 or 32)
#endif
#ifndef QG_W4_SCALAR_BM
#define QG_W4_SCALAR_BM 256  // W4A8 tiles at least this wide load scalar scales one block ahead
#endif
#ifndef QG_W4_SCALAR_AHEAD
#define QG_W4_SCALAR_AHEAD 1  // blocks ahead of their use that scalar W4A8 scales are loaded
#endif
#ifndef QG_W4_SKINNY
#define QG_W4_SKINNY 1  // W4A8 GEMMs of at most 64 tokens may run 16-row tiles
#endif
#ifndef QG_W4_BM32
#define QG_W4_BM32 1  // W4A8 GEMMs of at most 64 tokens may run 32-token tiles
#endif
#ifndef QG_PAIR_WAIT
#define QG_PAIR_WAIT 1  // W4A8 (stage mode): one accumulator wait per stage of two blocks
#endif
constexpr int kBN = 128;      // weight rows per tile (MMA M, tensor-memory lanes)
constexpr int kBK = 64;       // K per stage
constexpr int kFirstEpiWarp = 3;         // warp 0 producer, warps 1-2 MMA issuers
// Epilogue warps of a tile width (a multiple of 4: tensor-memory lane
// quarters); QG_EPI_WARPS applies to tiles of 128 tokens and more.
__host__ __device__ constexpr int epi_warps_for(int bm) { return bm >= 128 ? QG_EPI_WARPS : 8; }
__host__ __device__ constexpr int threads_for(int bm) { return 32 * (kFirstEpiWarp + epi_warps_for(bm)); }
constexpr uint32_t kStageABytes = kBN * kBK * 2;  // 16 KB
constexpr int kCtasPerSm = QG_CTAS_PER_SM;  // CTAs sharing an SM (and its tensor memory)
constexpr uint32_t kTmemCols = 512 / kCtasPerSm;
// blocks of activation sums in flight (W4A8); 256-token tiles keep 8, which
// leaves room for a third TMA stage
__host__ __device__ constexpr int asum_ring(int bm) { return bm >= 256 ? 8 : 16; }

// Tile width BM = tokens per tile (MMA N, tensor-memory columns). W8A8 runs
// 256 (one FMA per element per block) with narrower tiles for leftovers;
// W4A8 (two FMAs per element per block) 128 or 256, its 256-token tiles with
// scalar scale loads and four-block activation-sum rounds to stay in the
// registers of 11 warps.
template <int BM>
struct LargeCfg {
  static_assert(BM % 16 == 0 && BM >= 32 && BM <= 256 && kTmemCols % BM == 0, "tile width");
  static constexpr int kBM = BM;
  static constexpr int kEpiWarps = epi_warps_for(BM);
  static constexpr int kThreads = threads_for(BM);
  // per-block accumulators in this CTA's tensor memory (at most 8)
  static constexpr int kTBufs = kTmemCols / BM < 8 ? kTmemCols / BM : 8;
  static constexpr uint32_t kStageBBytes = BM * kBK * 2;
  static constexpr int kColsPerThread = BM / (kEpiWarps / 4);
  static_assert(kColsPerThread % 16 == 0, "whole 16-column tensor-memory loads per thread");
  static constexpr int kChunk = QG_CHUNK < kColsPerThread ? QG_CHUNK : kColsPerThread;
};

// TMA ring depth: as many stages as fit next to the output staging, the
// activation-sum ring and the barriers (narrow tiles have small stages and
// need many of them in flight: a stage's load takes ~1-2 us under load)
template <bool kQ4K, int BM>
__host__ __device__ constexpr int stages_for() {
  constexpr int kCols = LargeCfg<BM>::kColsPerThread;
  constexpr int kEpiWarps = LargeCfg<BM>::kEpiWarps;
  constexpr int kFixed = (QG_TMA_OUT ? (kEpiWarps / 4) * kCols * kBN * 2 : 16) +
                         (kQ4K ? asum_ring(BM) : 1) * BM * 4 +
                         kEpiWarps * kCols * 4 + 2048;  // + barriers and alignment slack
  constexpr int kPer = (int)kStageABytes + BM * kBK * 2;
  constexpr int n0 = (226 * 1024 - kFixed) / kPer;
  // Tiles with at least four accumulators alternate whole stages between the
  // two MMA issuers, each waiting only on its own stages' barriers. With an
  // even depth every ring slot belongs to one issuer, which then sees every
  // phase of it; with an odd depth a slot alternates between the issuers, so
  // each would see every other phase, and a parity wait could take a phase
  // two loads old for the one it needs.
  constexpr bool kAlternating = kTmemCols / BM >= 4;
  constexpr int n = kAlternating ? n0 & ~1 : n0;
  // (W4A8 keeps 4: a deeper ring measured ~25 % slower there)
  constexpr int cap = kQ4K ? 4 : 12;
  return QG_STAGES ? QG_STAGES : (n > cap ? cap : n);
}

template <bool kQ4K, int BM>
struct LargeSmem {
  static constexpr int kEpiWarps = LargeCfg<BM>::kEpiWarps;
  static constexpr int kStages = stages_for<kQ4K, BM>();
  static constexpr int kCols = LargeCfg<BM>::kColsPerThread;
  uint8_t a[kStages][kStageABytes];
  uint8_t b[kStages][LargeCfg<BM>::kStageBBytes];
  // bf16 output tile staged for the TMA store: per group of four epilogue
  // warps (a column slice of the tile), kCols token rows x 128 weight rows
  // (row-major, the store's box)
  uint16_t ostage[QG_TMA_OUT ? kEpiWarps / 4 : 1][QG_TMA_OUT ? kCols * kBN : 8];
  float asum[kQ4K ? asum_ring(BM) : 1][BM];
  float sa_stage[kEpiWarps][kCols];  // per epilogue warp: its tile's activation scales
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[LargeCfg<BM>::kTBufs], tempty[LargeCfg<BM>::kTBufs];
  uint64_t afull[asum_ring(BM)], aempty[asum_ring(BM)];
  uint64_t mdrain[2];    // per MMA issuer: completion of its MMAs after a wait gave up
  uint32_t tmem_base;
  uint32_t tmem_busy;    // nonzero: an issuer's MMAs did not complete; tensor memory stays allocated
};
template <bool kQ4K, int BM>
constexpr size_t large_smem_bytes() { return sizeof(LargeSmem<kQ4K, BM>) + 1024; }  // + alignment slack
static_assert(kStageABytes % 1024 == 0, "1024-B aligned stages");


struct LargeArgs {
  const float* d32;      // W8A8: [N][ldd] fp32 scales; W4A8: d*sc [N][ldd]
  const float* dm32;     // W4A8: dmin*m [N][ldd]
  const int32_t* bsum;   // W4A8: [M][B] activation block sums
  const float* sa;       // [M]
  void* out;
  int64_t ldo;
  int64_t ldd;
  int M, N, K;
  int out_f32;
  int tma_out;           // 1: bf16 outputs leave through the TMA store (tmO)
  int tile_group;        // token tiles per group of the persistent tile order
  int pdl;               // launched as a programmatic dependent of the quantize kernel
  int32_t* dbg;          // [M][N][B] isum export (debug) or null
  uint32_t* err;
};

__device__ __forceinline__ void tile_coords(int tile, int MT, int NT, int kGroup, int& mt,
                                            int& nt) {
  // groups of up to kGroup token tiles; inside a group the token tile varies
  // fastest so concurrently running CTAs share weight tiles in L2
  const int per_group = kGroup * NT;
  const int grp = tile / per_group;
  const int first = grp * kGroup;
  const int gm = min(kGroup, MT - first);
  const int idx = tile - grp * per_group;
  mt = first + idx % gm;
  nt = idx / gm;
}

template <bool kQ4K, bool kDebug, int BM>
__global__ void __launch_bounds__(threads_for(BM), kCtasPerSm)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const LargeArgs args) {
  using C = LargeCfg<BM>;
  constexpr int kEpiWarps = C::kEpiWarps;
  constexpr int kStages = stages_for<kQ4K, BM>();
  constexpr bool kStageMode = C::kTBufs % 4 == 0;
  static_assert(!kStageMode || kStages % 2 == 0, "alternating issuers need an even ring");
  constexpr int kBM = C::kBM;
  constexpr int kTBufs = C::kTBufs;
  constexpr uint32_t kStageBBytes = C::kStageBBytes;
  constexpr int kColsPerThread = C::kColsPerThread;
  constexpr int kAsumRing = asum_ring(BM);
  extern __shared__ uint8_t smem_raw[];
  LargeSmem<kQ4K, BM>& S = *reinterpret_cast<LargeSmem<kQ4K, BM>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = args.M, N = args.N, K = args.K;
  const int NB = K / kBlk;                  // blocks
  const int NS = (NB + 1) / 2;              // stages per tile
  const int MT = (M + kBM - 1) / kBM, NT = (N + kBN - 1) / kBN;
  const int tiles = MT * NT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kStageMode ? 1 : 2);  // commits of the issuers that use the stage
    }
    for (int i = 0; i < kTBufs; ++i) {
      mbar_init(&S.tfull[i], 1);
      mbar_init(&S.tempty[i], kEpiWarps * 32);  // every epilogue thread hands back its loads
    }
    for (int i = 0; i < kAsumRing; ++i) {
      mbar_init(&S.afull[i], 32);
      mbar_init(&S.aempty[i], kEpiWarps * 32);
    }
    mbar_init(&S.mdrain[0], 1);
    mbar_init(&S.mdrain[1], 1);
    S.tmem_busy = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int aslot = 0;
    uint32_t aphase = 0;
    bool ok = true;
    uint32_t loaded = 0, load_par = 0;  // per stage: a load was issued; parity of the last one
    // W4A8: activation block sums of kBsR blocks (a quad per 16-byte load)
    // for this lane's tokens; 256-token tiles take four blocks per round to
    // keep the two rounds in registers
    constexpr int kBsQ = kBM >= 256 ? 1 : 2, kBsR = 4 * kBsQ;
    int4 bs_cur[kQ4K ? kBM / 32 : 1][kBsQ], bs_nxt[kQ4K ? kBM / 32 : 1][kBsQ];
    auto load_bs = [&](int mt, int blk0, int4 (&dst)[kQ4K ? kBM / 32 : 1][kBsQ]) {
#pragma unroll
      for (int i = 0; i < kBM / 32; ++i) {
        const int m = mt * kBM + i * 32 + lane;
        const int4* p = reinterpret_cast<const int4*>(args.bsum + (int64_t)(m < M ? m : 0) * NB + blk0);
#pragma unroll
        for (int j = 0; j < kBsQ; ++j) dst[i][j] = m < M ? __ldg(p + j) : make_int4(0, 0, 0, 0);
      }
    };
    // As a programmatic dependent of the quantize kernel (W8A8): the weight
    // tiles of the first P stages are requested before the wait for its
    // grid, their activation tiles after it. W4A8 reads activation block
    // sums in this warp as well: it waits before anything.
    const int P = (args.pdl && !kQ4K) ? min(min(NS, kStages), 3) : 0;
    if (args.pdl && kQ4K) griddep_wait();
    bool first = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, first = false) {
      int mt, nt;
      tile_coords(tile, MT, NT, args.tile_group, mt, nt);
      for (int s = 0; s < NS && ok; ++s) {
        if (lane == 0) {
          ok = mbar_wait(&S.empty[stage], phase ^ 1, args.err);
          if (ok) {
            loaded |= 1u << stage;
            load_par = (load_par & ~(1u << stage)) | (phase << stage);
            mbar_arrive_expect_tx(&S.full[stage], kStageABytes + kStageBBytes);
            tma_load_2d(S.a[stage], &tmA, &S.full[stage], s * kBK, nt * kBN);
            if (!(first && s < P))
              tma_load_2d(S.b[stage], &tmB, &S.full[stage], s * kBK, mt * kBM);
            if (first && s + 1 == P) {
              // the first tile's first P stages are ring slots 0..P-1
              griddep_wait();
              for (int r = 0; r < P; ++r)
                tma_load_2d(S.b[r], &tmB, &S.full[r], r * kBK, mt * kBM);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
        if (kQ4K && ok) {
          for (int j = 0; j < 2; ++j) {
            const int blk = 2 * s + j;
            if (blk >= NB) break;
            // the tile's activation block sums come kBsR blocks per load
            // round (NB and the block index are multiples of 8), the next
            // round requested while this one is used, so each round's
            // latency is hidden behind its blocks
            if (blk % kBsR == 0) {
              if (blk == 0) load_bs(mt, 0, bs_cur);
              else {
#pragma unroll
                for (int i = 0; i < kBM / 32; ++i)
#pragma unroll
                  for (int j = 0; j < kBsQ; ++j) bs_cur[i][j] = bs_nxt[i][j];
              }
              if (blk + kBsR < NB) load_bs(mt, blk + kBsR, bs_nxt);
            }
            ok = mbar_wait(&S.aempty[aslot], aphase ^ 1, args.err);
            if (!ok) break;
            const int q = blk % kBsR;
#pragma unroll
            for (int i = 0; i < kBM / 32; ++i) {
              const int4 w = bs_cur[i][q >> 2];
              const int v = (q & 3) == 0 ? w.x : (q & 3) == 1 ? w.y : (q & 3) == 2 ? w.z : w.w;
              S.asum[aslot][i * 32 + lane] = (float)v;  // exact: |v| <= 4064
            }
            mbar_arrive(&S.afull[aslot]);
            if (++aslot == kAsumRing) { aslot = 0; aphase ^= 1; }
          }
        }
      }
    }
    // Tail: wait until the MMA has released every stage, so that no commit
    // arrival is still outstanding on this CTA's barriers when it exits.
    if (lane == 0 && ok) {
      for (int i = 0; i < kStages; ++i) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1, args.err)) break;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    // Every TMA load this thread issued has landed before the CTA exits, also
    // after a wait gave up (a bounded wait on each stage's last load; at
    // once when it was consumed).
    if (lane == 0) {
      for (int i = 0; i < kStages; ++i)
        if ((loaded >> i) & 1u) mbar_wait(&S.full[i], (load_par >> i) & 1u, args.err);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Block mode (two accumulators, wide tiles): issuer `par` handles block
    // 2s+par of every stage s, in buffer par. Stage mode (kTBufs a multiple
    // of 4, narrow tiles, whose MMAs are short): issuer `par` takes whole
    // stages -- the stages g = par, par+2, ... counted over all of this CTA's
    // tiles -- and block j of stage g goes to buffer (2g+j) % kTBufs, so each
    // issuer owns half the buffers and waits on a stage once for two blocks.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBN, kBM);
      static_assert(kTBufs >= 2 && kTBufs % 2 == 0, "accumulators split between two issuers");
      const int par = warp - 1;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tph = 0;  // bit b: phase of the next wait on tempty[b]
      bool ok = true;
      int gs = 0;        // stages issued so far over all tiles (stage mode)
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        for (int s = 0; s < NS && ok; ++s, ++gs) {
          if (kStageMode && (gs & 1) != par) {
            if (++stage == kStages) { stage = 0; phase ^= 1; }
            continue;
          }
          ok = mbar_wait(&S.full[stage], phase, args.err);
          if (!ok) break;
          const uint32_t a_addr = smem_u32(S.a[stage]);
          const uint32_t b_addr = smem_u32(S.b[stage]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (!kStageMode && j != par) continue;
            const int blk = 2 * s + j;
            if (blk >= NB) continue;
            const int tb = kStageMode ? (2 * gs + j) % kTBufs : blk % kTBufs;
            const uint32_t tpar = ((tph >> tb) & 1u) ^ 1u;
            ok = mbar_wait(&S.tempty[tb], tpar, args.err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(tb * kBM);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t koff = (uint32_t)((j * 32 + kk * 16) * 2);  // bytes within row
              mma_f16_ss(d_tmem, smem_desc_sw128(a_addr + koff), smem_desc_sw128(b_addr + koff),
                         idesc, kk);
            }
            mma_commit(&S.tfull[tb]);
            tph ^= 1u << tb;
          }
          if (!ok) break;
          mma_commit(&S.empty[stage]);  // arrives once this issuer's MMAs are done
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // a wait gave up: the MMAs this thread issued may still run; wait
        // (bounded) for all of them before tensor memory is freed. If even
        // that wait gives up, the tensor memory is left allocated.
        mma_commit(&S.mdrain[par]);
        if (!mbar_wait(&S.mdrain[par], 0, args.err)) atomicExch(&S.tmem_busy, 1u);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - kFirstEpiWarp) >> 2;
    uint32_t tph = 0;  // bit b: phase of the next wait on tfull[b]
    const bool ostore = args.tma_out && quarter == 0 && lane == 0;  // issues this half's stores
    // the activation scales come from the quantize kernel, and the output may
    // be what the kernel before it read
    if (args.pdl) griddep_wait();
    int aslot = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, MT, NT, args.tile_group, mt, nt);
      const int ti = (tile - (int)blockIdx.x) / (int)gridDim.x;  // this CTA's tile count so far
      const int n = nt * kBN + quarter * 32 + lane;
      const bool nvalid = n < N;
      const float* drow = args.d32 + (int64_t)(nvalid ? n : 0) * args.ldd;
      const float* mrow = kQ4K ? args.dm32 + (int64_t)(nvalid ? n : 0) * args.ldd : nullptr;
      float2 acc[kColsPerThread / 2];
#pragma unroll
      for (int i = 0; i < kColsPerThread / 2; ++i) acc[i] = make_float2(0.f, 0.f);
      // this tile's activation scales, copied to shared memory in the
      // background for the output phase (its previous reader, the last
      // tile's output phase, ended with a warp sync)
      const int mbase = mt * kBM + half * kColsPerThread;
      float* sw = S.sa_stage[warp - kFirstEpiWarp];
      if (!kDebug) {
#pragma unroll
        for (int j = 0; j < (kColsPerThread + 31) / 32; ++j) {
          const int c = 32 * j + lane, m = mbase + c;
          if (c < kColsPerThread) {
            if (m < M)
              cp_async_4(sw + c, args.sa + m);
            else
              sw[c] = 0.0f;
          }
        }
      }

      // Weight scales are prefetched; the loads are volatile so the compiler
      // keeps them where they are written. W8A8: one scalar load one block
      // ahead (quads of four blocks one to three quads ahead, or scalars two
      // blocks ahead, measured 3-55 % slower: the epilogue loop is tight on
      // registers). W4A8: four blocks per 16-byte load of d*sc and of dmin*m
      // (rows are 16-byte aligned: whole quads), one quad ahead of its use;
      // its 256-token tiles load both as scalars one block ahead (the quads
      // spill there).
      constexpr int kQA = (kQ4K && BM < QG_W4_SCALAR_BM) ? 1 : 0;
      constexpr int kQR = kQA > 0 ? kQA + 1 : 1;
      constexpr int kSA = kQ4K ? QG_W4_SCALAR_AHEAD : 1;  // scalar loads: blocks ahead
      float d_next[kSA], m_next[kSA];
      float4 dq[kQR], mq[kQR];
#pragma unroll
      for (int i = 0; i < kQR; ++i) {
        dq[i] = mq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kQA > 0 && nvalid && 4 * i < NB) {
          dq[i] = ldg_f32x4_pinned(drow + 4 * i);
          if (kQ4K) mq[i] = ldg_f32x4_pinned(mrow + 4 * i);
        }
      }
#pragma unroll
      for (int i = 0; i < kSA; ++i) {
        d_next[i] = m_next[i] = 0.0f;
        if (kQA == 0 && nvalid && i < NB) {
          d_next[i] = ldg_f32_pinned(drow + i);
          if (kQ4K) m_next[i] = ldg_f32_pinned(mrow + i);
        }
      }
      for (int blk = 0; blk < NB && ok; ++blk) {
        float dw, ndm = 0.0f;
        if (kQA > 0) {
          if ((blk & 3) == 0 && blk > 0) {
#pragma unroll
            for (int i = 0; i + 1 < kQR; ++i) {
              dq[i] = dq[i + 1];
              if (kQ4K) mq[i] = mq[i + 1];
            }
            const int nxt = blk + 4 * kQA;
            if (nxt < NB && nvalid) {
              dq[kQR - 1] = ldg_f32x4_pinned(drow + nxt);
              if (kQ4K) mq[kQR - 1] = ldg_f32x4_pinned(mrow + nxt);
            }
          }
          const int q = blk & 3;
          dw = q == 0 ? dq[0].x : q == 1 ? dq[0].y : q == 2 ? dq[0].z : dq[0].w;
          if (kQ4K) ndm = -(q == 0 ? mq[0].x : q == 1 ? mq[0].y : q == 2 ? mq[0].z : mq[0].w);
        } else {
          dw = d_next[0];
          if (kQ4K) ndm = -m_next[0];
#pragma unroll
          for (int i = 0; i + 1 < kSA; ++i) {
            d_next[i] = d_next[i + 1];
            if (kQ4K) m_next[i] = m_next[i + 1];
          }
          if (blk + kSA < NB && nvalid) {
            d_next[kSA - 1] = ldg_f32_pinned(drow + blk + kSA);
            if (kQ4K) m_next[kSA - 1] = ldg_f32_pinned(mrow + blk + kSA);
          }
        }
        const int tb = kStageMode ? (2 * (ti * NS + (blk >> 1)) + (blk & 1)) % kTBufs
                                  : blk % kTBufs;
        if (kStageMode && kQ4K && QG_PAIR_WAIT) {
          // one issuer commits both blocks of a stage, and the second commit
          // arrives only after all of that issuer's earlier MMAs: a wait on
          // the stage's second block covers the first (the first buffer's
          // own phase is counted as consumed; it completes no later). W4A8
          // only: M=4096 2.77 -> 2.70 ms; W8A8 narrow tiles measured 8-20 %
          // slower with it
          if ((blk & 1) == 0) {
            const bool pair = blk + 1 < NB;
            const int tw = pair ? (tb + 1) % kTBufs : tb;
            ok = mbar_wait(&S.tfull[tw], (tph >> tw) & 1u, args.err);
            tph ^= (1u << tb) | (pair ? (1u << tw) : 0u);
          }
          if (ok) ok = mbar_wait(&S.afull[aslot], aphase, args.err);
          if (!ok) break;
        } else {
          // `ok` is uniform across the warp without a vote: every lane runs the
          // same polling loop on the same barrier and sees the same answers (a
          // per-block warp vote or shuffle here costs about 9 % of the time)
          ok = mbar_wait(&S.tfull[tb], (tph >> tb) & 1u, args.err);
          if (kQ4K && ok) ok = mbar_wait(&S.afull[aslot], aphase, args.err);
          if (!ok) break;
          tph ^= 1u << tb;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)(tb * kBM + half * kColsPerThread);
        const float2 dw2 = make_float2(dw, dw);
        const float2 ndm2 = make_float2(ndm, ndm);
        constexpr int kChunk = C::kChunk;  // columns per tensor-memory load
        constexpr int kNch = kColsPerThread / kChunk;
        // kBatch loads are issued before one wait, so the tensor-memory load
        // latency is paid once per batch instead of once per chunk
        constexpr int kBatchCfg = QG_EPI_BATCH ? QG_EPI_BATCH : (kColsPerThread <= 64 ? kNch : 1);
        constexpr int kBatch = kBatchCfg > kNch ? kNch : kBatchCfg;
        static_assert(kNch % kBatch == 0, "batch must divide the chunks");
#pragma unroll
        for (int c0 = 0; c0 < kNch; c0 += kBatch) {
          uint32_t v[kBatch][kChunk];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if constexpr (kChunk == 32)
              tmem_ld32(taddr + (c0 + b) * kChunk, v[b]);
            else
              tmem_ld16(taddr + (c0 + b) * kChunk, v[b]);
          }
          tmem_wait_ld();
          // pin the loaded registers after the wait: no use may move above it
#pragma unroll
          for (int b = 0; b < kBatch; ++b)
#pragma unroll
            for (int i = 0; i < kChunk; ++i) asm volatile("" : "+r"(v[b][i]));
          if (c0 + kBatch == kNch) {
            // all of this thread's columns of the block are in registers:
            // each thread hands its part of the buffer back (no warp sync)
            tc_fence_before();
            mbar_arrive(&S.tempty[tb]);
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int ch = c0 + b;
            if (kDebug) {
              const int m0 = mt * kBM + half * kColsPerThread + ch * kChunk;
#pragma unroll
              for (int i = 0; i < kChunk; ++i) {
                const int m = m0 + i;
                if (m < M && nvalid)
                  args.dbg[((int64_t)m * N + n) * NB + blk] =
                      __float2int_rn(__uint_as_float(v[b][i]));
              }
            }
#pragma unroll
            for (int i = 0; i < kChunk / 2; ++i) {
              const float2 x =
                  make_float2(__uint_as_float(v[b][2 * i]), __uint_as_float(v[b][2 * i + 1]));
              float2& a2 = acc[ch * (kChunk / 2) + i];
              a2 = __ffma2_rn(x, dw2, a2);
              if (kQ4K) {
                const float2 as = *reinterpret_cast<const float2*>(
                    &S.asum[aslot][half * kColsPerThread + ch * kChunk + 2 * i]);
                a2 = __ffma2_rn(as, ndm2, a2);
              }
            }
          }
        }
        if (kQ4K) {
          mbar_arrive(&S.aempty[aslot]);  // this thread's reads of the slot are done
          if (++aslot == kAsumRing) { aslot = 0; aphase ^= 1; }
        }
      }
      if (kDebug) continue;
      if (args.tma_out) {
        // the store issued one tile ago must have read this half's staging
        // buffer; the four warps of the half also agree on going on (a wait
        // that gave up in one of them stops all four, none is left at a barrier)
        if (ostore) bulk_wait_read_all();
        ok = bar_and(1 + half, 128, ok);
      }
      if (!ok) break;
      // final scale by the activation scale. This code runs once per tile,
      // cold in the instruction cache, so it is kept short: packed f32x2
      // multiplies and bf16x2 conversions, scales read through restrict
      // pointers (without them every scale load waited behind the previous
      // output's store). A rolled variant (kCh < kColsPerThread: trips of kCh
      // columns, accumulators slid down after each) measured slower.
      cp_async_wait_all();
      __syncwarp();
      constexpr int kCh = kColsPerThread < QG_OUT_CHUNK ? kColsPerThread : QG_OUT_CHUNK;
      const float* __restrict__ swr = sw;
      if (args.tma_out) {
        // bf16 outputs into this half's staging tile, then one thread stores
        // it with TMA (rows >= M and columns >= N are clipped); the store
        // drains while the next tile computes
        __nv_bfloat16* __restrict__ ob =
            reinterpret_cast<__nv_bfloat16*>(S.ostage[QG_TMA_OUT ? half : 0]) + quarter * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < kColsPerThread; c0 += kCh) {
#pragma unroll
          for (int j = 0; j < kCh; j += 2) {
            const float4 q = *reinterpret_cast<const float4*>(swr + c0 + (j & ~3));
            const float2 y = __fmul2_rn(acc[j / 2], (j & 2) ? make_float2(q.z, q.w) : make_float2(q.x, q.y));
            const __nv_bfloat162 h = __floats2bfloat162_rn(y.x, y.y);  // both RNE
            ob[(c0 + j) * kBN] = h.x;
            ob[(c0 + j + 1) * kBN] = h.y;
          }
#pragma unroll
          for (int i = 0; i < (kColsPerThread - kCh) / 2; ++i) acc[i] = acc[i + kCh / 2];
        }
        fence_proxy_async_smem();
        named_barrier(1 + half, 128);
        if (ostore && mbase < M) {  // no store of a box wholly past M
          tma_store_2d(&tmO, S.ostage[QG_TMA_OUT ? half : 0], nt * kBN, mbase);
          bulk_commit_group();
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < kColsPerThread; c0 += kCh) {
#pragma unroll
          for (int j = 0; j < kCh; j += 2) {
            const float4 q = *reinterpret_cast<const float4*>(swr + c0 + (j & ~3));
            const float2 y = __fmul2_rn(acc[j / 2], (j & 2) ? make_float2(q.z, q.w) : make_float2(q.x, q.y));
            const int m = mbase + c0 + j;
            if (nvalid && m < M) {
              if (args.out_f32)
                reinterpret_cast<float*>(args.out)[(int64_t)m * args.ldo + n] = y.x;
              else
                reinterpret_cast<uint16_t*>(args.out)[(int64_t)m * args.ldo + n] =
                    f32_to_bf16_rne(y.x);
            }
            if (nvalid && m + 1 < M) {
              if (args.out_f32)
                reinterpret_cast<float*>(args.out)[(int64_t)(m + 1) * args.ldo + n] = y.y;
              else
                reinterpret_cast<uint16_t*>(args.out)[(int64_t)(m + 1) * args.ldo + n] =
                    f32_to_bf16_rne(y.y);
            }
          }
#pragma unroll
          for (int i = 0; i < (kColsPerThread - kCh) / 2; ++i) acc[i] = acc[i + kCh / 2];
        }
      }
      __syncwarp();  // sw is rewritten at the next tile
    }
    cp_async_wait_all();          // no copy into shared memory outlives the loop
    if (ostore) bulk_wait_all();  // this CTA's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && S.tmem_busy == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// fp16 matrix [rows][K] row-major, box = 64 (K) x box_rows, 128-byte swizzle
// (also used by gemm_skinny.cu)
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                      uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// rows of `row_bytes` bytes (a multiple of 16), read as 8-byte words:
// box = box_words x box_rows, no swizzle, so the box lands row after row at a
// pitch of 8 * box_words bytes; words past a row's end read as zero (used by
// gemm_small.cu for the decode kernels' activation rows and block sums)
bool make_tmap_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                    uint32_t box_words, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15) || row_bytes % 16) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_words, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output [M][ldo] as the TMA store's destination, box = 128 weight rows
// x `rows` tokens; false when the base or the row pitch is not 16-byte
// aligned (the kernel then stores element by element)
static bool make_out_tmap(CUtensorMap* map, void* base, int64_t M, int64_t N, int64_t ldo,
                          uint32_t rows) {
  if (!base || (reinterpret_cast<uintptr_t>(base) & 15) || (ldo * 2) % 16) return false;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)(ldo * 2)};
  cuuint32_t box[2] = {(cuuint32_t)kBN, rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kQ4K, bool kDebug, int BM>
static cudaError_t launch_prefill_t(const CUtensorMap& ta, const void* q16, const LargeArgs& a,
                                   cudaStream_t st) {
  constexpr size_t kSmem = large_smem_bytes<kQ4K, BM>();
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  CUtensorMap tb, to;
  if (!make_tmap(&tb, q16, a.M, a.K, BM)) return cudaErrorNotSupported;
  memset(&to, 0, sizeof(to));
  LargeArgs args = a;
  args.tma_out = (QG_TMA_OUT && !kDebug && !a.out_f32 &&
                  make_out_tmap(&to, a.out, a.M, a.N, a.ldo, LargeCfg<BM>::kColsPerThread))
                     ? 1 : 0;
  // tile order: groups of 2 token tiles when a GEMM has at most 8 of them
  // (4B-class prefill shapes: 2-3 % faster than 8), else of 16 (27B-class:
  // ~0.5 % faster than 8); measured on GB300
  args.tile_group = ceil_div(a.M, BM) <= 8 ? 2 : 16;
  auto kern = prefill_gemm_kernel<kQ4K, kDebug, BM>;
  static std::atomic<uint64_t> attr_set{0};
  {
    const cudaError_t e = smem_attr_once_per_device(kern, (int)kSmem, attr_set);
    if (e != cudaSuccess) return e;
  }
  const int tiles = (int)(ceil_div(a.M, BM) * ceil_div(a.N, kBN));
  const int slots = num_sms() * kCtasPerSm;
  const int grid = tiles < slots ? tiles : slots;
  return launch_kernel(kern, dim3(grid), dim3(LargeCfg<BM>::kThreads), kSmem, st, a.pdl != 0, ta,
                       tb, to, args);
}

// Cycles of one 32-block step of one tile (measured on GB300 with forced
// choices): tensor-memory tiles of 128 weight rows x BM tokens, whose fixed
// per-step barrier round trip does not shrink with BM; and 16-row tiles of
// gemm_skinny.cu (two CTAs per SM), whose steps are cheap but whose tiles are
// 8x smaller. Narrow work goes where the SMs fill best.
static double tc_step_cycles(int bm) {
  switch (bm) {
    case 256: return 800.0;
    case 128: return 560.0;
    case 64: return 450.0;
    default: return 420.0;  // 32
  }
}
static double skinny_step_cycles(int tb, int64_t per_sm) {
  return tb == 32 ? 135.0 : (tb == 64 ? (per_sm > 2 ? 332.0 : 260.0) : 300.0);
}
// Token-tile width of the 16-row tiles (64-token tiles three CTAs per SM,
// the others two): the one of the smallest estimated time, waves x step cost
// (64-token steps cost more when three CTAs share an SM).
static double skinny_time(int64_t M, int64_t rows, int sms, int tb) {
  const int64_t ctas = ceil_div(rows, (int64_t)16) * ceil_div(M, (int64_t)tb);
  const int64_t slots = (tb == 64 ? 3 : 2) * (int64_t)sms;
  const int64_t per_sm = std::min<int64_t>(ceil_div(ctas, (int64_t)sms), tb == 64 ? 3 : 2);
  return (double)ceil_div(ctas, slots) * skinny_step_cycles(tb, per_sm);
}
static int skinny_tb(int64_t M, int64_t rows, int sms) {
  int best = 32;
  for (int tb : {64, 128})
    if (M > tb / 2 && skinny_time(M, rows, sms, tb) < skinny_time(M, rows, sms, best)) best = tb;
  return best;
}

// Wave plan of a W8A8 prefill GEMM: the weight-row tiles [0, nt_wide) run as
// 256-token tensor-memory tiles; the remaining rows (all tokens) run in a
// second launch, as bm_tail-token tensor-memory tiles or, with bm_tail = 0,
// as 16-row tiles of gemm_skinny.cu. nt_wide = NT: one launch.
struct PrefillPlan {
  int nt_wide;
  int bm_tail;
};
static PrefillPlan plan_prefill_w8a8(int64_t M, int64_t N, int sms) {
  const int64_t NT = ceil_div(N, kBN), MT = ceil_div(M, 256);
  auto waves = [&](int64_t tiles, int per_sm) {
    return (double)ceil_div(tiles, (int64_t)sms * per_sm);
  };
  auto rest = [&](int64_t nw, int& bm_best) {  // best time of rows [nw*128, N) over all tokens
    double best = 1e30;
    for (int bm : {128, 64, 32}) {
      const double t = waves(ceil_div(M, (int64_t)bm) * (NT - nw), 1) * tc_step_cycles(bm);
      if (t < best) { best = t; bm_best = bm; }
    }
    const int64_t rows = N - nw * kBN;
    const double ts = skinny_time(M, rows, sms, skinny_tb(M, rows, sms));
    if (ts * 1.1 < best) { best = ts; bm_best = 0; }  // the table is rougher for 16-row tiles
    return best;
  };
  PrefillPlan best{(int)NT, 256};
  double best_t = waves(MT * NT, 1) * tc_step_cycles(256);
  const int64_t nt_wide = (sms * (MT * NT / sms)) / MT;  // weight-row tiles that fill whole waves
  for (int64_t nw = nt_wide; nw >= 0 && nw >= nt_wide - 1; --nw) {
    if (nw >= NT) continue;
    int bm = 0;
    const double t = (nw ? waves(MT * nw, 1) * tc_step_cycles(256) : 0.0) + rest(nw, bm);
    if (t < best_t * 0.97) { best_t = t; best = PrefillPlan{(int)nw, bm}; }
  }
  return best;
}

// The plan a launch carries out: the wave plan, or the one the tuning
// switches of this build force (QG_FORCE_BM: every W8A8 GEMM as one launch of
// that width; QG_SKINNY 1: the narrow part as 16-row tiles, 2: the whole GEMM
// as 16-row tiles). Launch, launch count and the host query all use it.
static PrefillPlan plan_as_built(int64_t M, int64_t N, int sms) {
  if (QG_SKINNY == 2) return PrefillPlan{0, 0};
  PrefillPlan p = QG_FORCE_BM ? PrefillPlan{0, QG_FORCE_BM} : plan_prefill_w8a8(M, N, sms);
  if (QG_SKINNY == 1 && (int64_t)p.nt_wide * kBN < N) p.bm_tail = 0;
  return p;
}

// gemm_skinny.cu: 16-weight-row tiles on legacy fp16 MMA
cudaError_t launch_skinny_q4k(const uint16_t* q16, const float* sa, const int32_t* bsum,
                              int64_t M, int64_t K, const uint16_t* wq16, const float* ds32,
                              const float* dm32, int64_t ldd, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int tb, uint32_t* err, bool pdl, cudaStream_t st);
cudaError_t launch_skinny_q8_0(const uint16_t* q16, const float* sa, int64_t M, int64_t K,
                               const uint16_t* wq16, const float* d32, int64_t ldd, int64_t N,
                               void* out, bool out_f32, int64_t ldo, int tb, uint32_t* err,
                               bool pdl, cudaStream_t st);

// The plan for M x N on `sms` SMs, as launch_prefill_q8_0 carries it out
// (host only): the weight rows of the 256-token launch, then the remaining
// rows' kind (0 none, 1 tensor-memory tiles, 2 16-row tiles) and token width.
void prefill_plan_q8_0(int64_t M, int64_t N, int sms, int64_t* rows_wide, int* narrow_kind,
                       int* narrow_tokens) {
  const PrefillPlan p = plan_as_built(M, N, sms);
  const int64_t n0 = (int64_t)p.nt_wide * kBN;
  *rows_wide = n0 < N ? n0 : N;
  *narrow_kind = 0;
  *narrow_tokens = 0;
  if (n0 >= N) return;
  if (p.bm_tail == 0) {
    *narrow_kind = 2;
    *narrow_tokens = skinny_tb(M, N - n0, sms);
  } else {
    *narrow_kind = 1;
    *narrow_tokens = p.bm_tail;
  }
}

int prefill_launches_q8_0(int64_t M, int64_t N) {
  const PrefillPlan p = plan_as_built(M, N, num_sms());
  return (p.nt_wide > 0 && (int64_t)p.nt_wide * kBN < N) ? 2 : 1;
}

// returns cudaErrorNotSupported when the tensor-map encoder is unavailable;
// pdl: the first launch is a programmatic dependent of the quantize kernel
// before it on the stream (a second launch follows the first in stream order)
cudaError_t launch_prefill_q8_0(const uint16_t* q16, const float* sa, int64_t M, int64_t K,
                                const void* packed, int64_t N, void* out, bool out_f32,
                                int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                                cudaStream_t st) {
  const Q8Layout L(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  LargeArgs a{};
  a.d32 = reinterpret_cast<const float*>(base + L.off_d32);
  a.ldd = L.B4;
  a.sa = sa;
  a.out = out;
  a.ldo = ldo;
  a.M = (int)M; a.N = (int)N; a.K = (int)K;
  a.out_f32 = out_f32 ? 1 : 0;
  a.dbg = dbg;
  a.err = err;
  const uint8_t* wq16 = base + L.off_q16;  // fp16 weights [N][K]
  CUtensorMap ta;
  if (dbg) {  // exported block sums: one launch of 256-token tiles
    if (!make_tmap(&ta, wq16, N, K, kBN)) return cudaErrorNotSupported;
    return launch_prefill_t<false, true, 256>(ta, q16, a, st);
  }
  const PrefillPlan p = plan_as_built(M, N, num_sms());
  const int64_t n0 = (int64_t)p.nt_wide * kBN;  // first weight row of the narrow part
  if (n0 > 0) {
    LargeArgs aw = a;
    aw.N = (int)(n0 < N ? n0 : N);
    aw.pdl = pdl ? 1 : 0;
    if (!make_tmap(&ta, wq16, aw.N, K, kBN)) return cudaErrorNotSupported;
    const cudaError_t e = launch_prefill_t<false, false, 256>(ta, q16, aw, st);
    if (e != cudaSuccess || n0 >= N) return e;
  }
  // weight rows [n0, N) over all tokens, as narrow tiles
  LargeArgs an = a;
  an.N = (int)(N - n0);
  an.pdl = (pdl && n0 == 0) ? 1 : 0;
  an.d32 = a.d32 + n0 * a.ldd;
  an.out = out_f32 ? (void*)(reinterpret_cast<float*>(out) + n0)
                   : (void*)(reinterpret_cast<uint16_t*>(out) + n0);
  if (p.bm_tail == 0)  // 16-row tiles (legacy fp16 MMA)
    return launch_skinny_q8_0(q16, sa, M, K, reinterpret_cast<const uint16_t*>(wq16 + n0 * K * 2),
                              an.d32, an.ldd, an.N, an.out, out_f32, ldo,
                              skinny_tb(M, an.N, num_sms()), err, an.pdl != 0, st);
  if (!make_tmap(&ta, wq16 + n0 * K * 2, an.N, K, kBN)) return cudaErrorNotSupported;
  switch (p.bm_tail) {
    case 128: return launch_prefill_t<false, false, 128>(ta, q16, an, st);
    case 64: return launch_prefill_t<false, false, 64>(ta, q16, an, st);
    case 32: return launch_prefill_t<false, false, 32>(ta, q16, an, st);
    default: return launch_prefill_t<false, false, 256>(ta, q16, an, st);
  }
}

// Tiles of the W4A8 GEMM for M x N on `sms` SMs: kind 1 = tensor-memory tiles
// of 128 weight rows, kind 2 = 16-row tiles of gemm_skinny.cu; and the token
// width. A GEMM of at most 64 tokens whose 128-row tiles cannot fill half the
// SMs runs as 16-row tiles of 32 or 64 tokens (each tile walks all of K
// alone, so tile count sets the pace: 17408 -> 5120 at 64 tokens, 40 row
// tiles, 215 us as 32-token tensor-memory tiles). Other GEMMs of at most 64
// tokens: 64-token tensor-memory tiles (32 up to 32 tokens). Above, 128- or
// 256-token tiles, whichever needs fewer whole waves of persistent CTAs, a
// wave of 256-token tiles counted as 1.27 of 128-token ones (measured on
// GB300: 1.22 to 1.29 per wave over 1024-4096 tokens, both shapes of a
// 27B-class MLP; the wider tile halves the epilogue's fixed cost per element)
int prefill_tile_q4k(int64_t M, int64_t N, int sms, int* kind) {
  const int64_t NT = ceil_div(N, (int64_t)kBN);
  *kind = 1;
  if (M <= 64) {
    if (QG_W4_SKINNY && 2 * NT <= sms) {
      *kind = 2;
      return M <= 32 ? 32 : 64;
    }
    return (QG_W4_BM32 && (M <= 32 || 2 * NT <= sms)) ? 32 : 64;
  }
  if (QG_BM_W4A8) return QG_BM_W4A8;
  const int64_t w128 = ceil_div(ceil_div(M, (int64_t)128) * NT, (int64_t)sms);
  const int64_t w256 = ceil_div(ceil_div(M, (int64_t)256) * NT, (int64_t)sms);
  return 127 * w256 < 100 * w128 ? 256 : 128;
}

cudaError_t launch_prefill_q4k(const uint16_t* q16, const float* sa, const int32_t* bsum,
                               int64_t M, int64_t K, const void* packed, int64_t N, void* out,
                               bool out_f32, int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                               cudaStream_t st) {
  const Q4kLayout L(N, K);
  const auto* base = reinterpret_cast<const uint8_t*>(packed);
  CUtensorMap ta;
  if (!make_tmap(&ta, base + L.off_q16, N, K, kBN)) return cudaErrorNotSupported;
  LargeArgs a{};
  a.d32 = reinterpret_cast<const float*>(base + L.off_ds32);
  a.dm32 = reinterpret_cast<const float*>(base + L.off_dm32);
  a.ldd = L.B;
  a.bsum = bsum;
  a.sa = sa;
  a.out = out;
  a.ldo = ldo;
  a.M = (int)M; a.N = (int)N; a.K = (int)K;
  a.out_f32 = out_f32 ? 1 : 0;
  a.dbg = dbg;
  a.err = err;
  a.pdl = (pdl && !dbg) ? 1 : 0;
  if (dbg) return launch_prefill_t<true, true, 128>(ta, q16, a, st);
  int kind = 1;
  const int tb = prefill_tile_q4k(M, N, num_sms(), &kind);
  if (kind == 2)
    return launch_skinny_q4k(q16, sa, bsum, M, K, reinterpret_cast<const uint16_t*>(base + L.off_q16),
                             a.d32, a.dm32, a.ldd, N, out, out_f32, ldo, tb, err, a.pdl != 0, st);
  switch (tb) {
    case 32: return launch_prefill_t<true, false, 32>(ta, q16, a, st);
    case 64: return launch_prefill_t<true, false, 64>(ta, q16, a, st);
    case 256: return launch_prefill_t<true, false, 256>(ta, q16, a, st);
    default: return launch_prefill_t<true, false, 128>(ta, q16, a, st);
  }
}

}  // namespace qg
