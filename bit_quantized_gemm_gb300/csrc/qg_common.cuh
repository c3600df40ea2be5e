// qg_common.cuh -- shared device helpers for the quantized linear layer
// kernels: the packed-weight layout, bounded mbarrier waits, TMA, tcgen05
// (tensor memory + 5th-generation MMA) and legacy fp16 MMA wrappers.
//
// Everything here is hand-written inline PTX for sm_103a.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qgemm.h"

namespace qg {

// ---------------------------------------------------------------------------
// Sizes fixed by the formats (StartLux-Prism README, "Why StartLux-Prism":
// Q8_0 blocks of 32 int8 weights with one fp16 scale; Q4_K super-blocks of
// 256 4-bit weights in 8 sub-blocks of 32).
// ---------------------------------------------------------------------------
constexpr int kBlk = 32;          // K per block / sub-block
constexpr int kQ8Bytes = 34;      // {fp16 d; int8 q[32]}
constexpr int kQ4kWeights = 256;  // weights per super-block
constexpr int kQ4kBytes = 144;    // super-block bytes
constexpr int kMaxK = 65536;

// Error word codes (device-side, read by qg_check_device_error).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrRange = 2u;  // a packed value outside its format's range

__host__ __device__ constexpr int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Packed weight layout (opaque to callers; sized by qg_*_packed_bytes).
//
// Q8_0, for N rows, K columns, B = K/32 blocks, G = ceil(N/16) row groups:
//  stream  G*B*512 B   weights of group g, block b as 32 chunks of 16
//                       signed bytes: chunk 16h + (r ^ 4h) holds q[16g+r]
//                       [32b+16h .. +15] (a dot-product lane reads its row as
//                       chunks (0, r), (1, r); an MMA lane reads 8 bytes of
//                       rows r and r+8, free of bank conflicts).
//  dsc     G*(B4/4)*128 B  fp16 scales for the decode kernel: for group g,
//                       block quad p, row r (0..7): 16 bytes =
//                       d[16g+r][4p .. 4p+3], d[16g+r+8][4p .. 4p+3].
//  q16     N*K*2 B     the same int8 values as fp16, row-major [N][K]
//                       (operand A of the prefill tensor-core kernel).
//  d32     N*B4*4 B    scales as fp32, [N][B4] (B4 = B rounded up to 4).
// Q4_K, with J = K/256 super-blocks per row:
//  stream  G*B*256 B   nibbles of group g, block b, row r in 16 bytes,
//                       [G][B][16][16 B]: word x holds k = 8x..8x+3 in the
//                       low nibbles of its bytes, 8x+4..8x+7 in the high ones.
//  shdr    G*J*256 B   per row and super-block, [G][J][16 rows][16 B]: d,
//                       dmin (fp16), then eight 12-bit units sc_i | m_i << 6
//                       at bits [12i, 12i+12) of a 96-bit little-endian string.
//  q16     N*K*2 B     q (0..15) as fp16, row-major [N][K].
//  ds32    N*B*4 B     d*sc_b as fp32 (exact), [N][B].
//  dm32    N*B*4 B     dmin*m_b as fp32 (exact), [N][B].
// ---------------------------------------------------------------------------
struct Q8Layout {
  int64_t N, K, B, B4, G;
  int64_t off_stream, off_dsc, off_q16, off_d32, total;
  __host__ __device__ Q8Layout(int64_t n, int64_t k) : N(n), K(k) {
    B = K / kBlk;
    B4 = align_up(B, 4);
    G = ceil_div(N, 16);
    off_stream = 0;
    off_dsc = align_up(off_stream + G * B * 512, 256);
    off_q16 = align_up(off_dsc + G * (B4 / 4) * 128, 256);
    off_d32 = align_up(off_q16 + N * K * 2, 256);
    total = align_up(off_d32 + N * B4 * 4, 256);
  }
};

struct Q4kLayout {
  int64_t N, K, B, J, G;
  int64_t off_stream, off_shdr, off_q16, off_ds32, off_dm32, total;
  __host__ __device__ Q4kLayout(int64_t n, int64_t k) : N(n), K(k) {
    B = K / kBlk;
    J = K / kQ4kWeights;
    G = ceil_div(N, 16);
    off_stream = 0;
    off_shdr = align_up(off_stream + G * B * 256, 256);
    off_q16 = align_up(off_shdr + G * J * 256, 256);
    off_ds32 = align_up(off_q16 + N * K * 2, 256);
    off_dm32 = align_up(off_ds32 + N * B * 4, 256);
    total = align_up(off_dm32 + N * B * 4, 256);
  }
};

// SM count of the current device (cached per device)
inline int num_sms() {
  static std::atomic<int> cached[64] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// cudaFuncAttributeMaxDynamicSharedMemorySize for `kern`, set once per device
// (the attribute belongs to the function on the current device). `done`
// holds one bit per device 0..63; devices past 63 set it on every call.
template <typename Kern>
inline cudaError_t smem_attr_once_per_device(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launch `kern` on `st`; with `pdl`, as a programmatic dependent of the
// kernel before it on the stream: its CTAs may start while that kernel runs,
// and every read of that kernel's outputs (and every write of its inputs)
// in `kern` must follow griddep_wait().
template <class Kern, class... Args>
inline cudaError_t launch_kernel(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 bool pdl, const Args&... args) {
  if (!pdl) {
    kern<<<grid, block, smem, st>>>(args...);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Kernels that wait on barriers receive the address of the library's device
// error word (one per device) and OR a code into it when a wait gives up.
__device__ __forceinline__ void set_error(uint32_t* err, uint32_t code) {
  if (err) atomicOr(err, code);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and records a timeout) after `limit` polls.
// Each try_wait may suspend the thread for a short hardware-defined time
// while the phase is incomplete, so the default limit amounts to seconds,
// far above any legitimate wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          uint32_t limit = (1u << 24)) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  set_error(err, kErrTimeout);
  return false;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) -- 2D tiled load into shared memory, completion
// signalled on an mbarrier as transaction bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// TMA store of a 2D box from shared memory (bulk async-group completion)
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until every committed bulk store has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until every committed bulk store has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the TMA unit
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// named barrier among `count` threads (id 1..15; id 0 is __syncthreads)
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 1-D bulk copy global -> shared, completing on `bar` as transaction bytes
// (addresses 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// asynchronous 4-byte global -> shared copy (completes at cp_async_wait_all)
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// barrier among `count` threads that also returns the AND of their `v`
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (taddr.lane + i), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same wait, with the destination registers of the outstanding loads as
// operands, so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
        "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
        "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
        "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
        "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
      :
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Bits: [0,14) start>>4, [16,30) leading offset>>4 (unused for swizzled
// K-major), [32,46) stride offset>>4 (1024 B), [46,48) version 1,
// [61,64) layout 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major,
// M = m, N = n.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4)                       // D format: f32
         | (0u << 7) | (0u << 10)        // A, B format: f16
         | ((uint32_t)(n >> 3) << 17)    // N >> 3
         | ((uint32_t)(m >> 4) << 24);   // M >> 4
}

// ---------------------------------------------------------------------------
// Warp-level fp16 MMA, fp32 accumulate: m16n8k16 (d = a*b + c). On integer-
// valued operands with |sum| < 2^24 the fp32 accumulation is exact.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// Legacy int8 tensor-core MMA, m16n8k32, exact int32 sums from zero: A
// (16 x 32) as signed (kUA = false) or unsigned bytes, B (32 x 8) signed.
// Fragments: a0/a2 row g, a1/a3 row g+8 (g = lane / 4), k 4t..4t+3 for
// a0/a1 and 16 + 4t.. for a2/a3 (t = lane % 4); b0 k 4t.., b1 k 16 + 4t..,
// column g; d as for m16n8k16.
template <bool kUA>
__device__ __forceinline__ void mma_i8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  if (kUA)
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// Four biased bytes (q + 128) -> two fp16 pairs holding q exactly:
// the bytes become the low mantissa bits of 1024 + (q + 128), then 1152 is
// subtracted (all values are integers below 2048, exact in fp16).
__device__ __forceinline__ void biased_u8x4_to_f16x4(uint32_t u, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// Read-only 4-byte global load as volatile asm: it stays where it is written
// in program order (a prefetch the compiler may not sink to its use).
__device__ __forceinline__ float ldg_f32_pinned(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// 8-byte read-only load, volatile like ldg_f32_pinned (p 8-byte aligned)
__device__ __forceinline__ float2 ldg_f32x2_pinned(const float* p) {
  float2 v;
  asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}

// 16-byte read-only load, volatile like ldg_f32_pinned (p 16-byte aligned)
__device__ __forceinline__ float4 ldg_f32x4_pinned(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on its stream still
// runs; griddep_wait() returns once that kernel has completed and its memory
// writes are visible (immediately when the launch was an ordinary one).
// griddep_launch_dependents() lets the next such kernel start early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Per-token activation quantization arithmetic (the quantize kernels).
// ---------------------------------------------------------------------------
// s = absmax / 127, one correctly rounded division
__device__ __forceinline__ float act_scale(float amax) { return __fdiv_rn(amax, 127.0f); }

// The reciprocal qround multiplies by: 1/s rounded once when s is normal (then
// finite and exact to 2^-24), else 0, which makes qround divide exactly.
__device__ __forceinline__ float act_scale_rcp(float s) {
  if (!(s >= 1.17549435e-38f)) return 0.0f;
  const float inv = __frcp_rn(s);
  return isinf(inv) ? 0.0f : inv;
}

// rint(x / s) with the IEEE-rounded quotient, returned as a float.
// r = x * rcp_rn(s) differs from the exact quotient by at most 2^-16 for
// |x/s| <= 128 (two roundings of relative size 2^-24 each), and the rounded
// quotient by at most 2^-16 + 2^-17 < 2^-15. rint() of the two can only
// differ when a half-integer lies within 2^-15 of r; those rare elements take
// the exact division.
// inv = 0 selects the exact division for every element (used when s is
// subnormal, where the reciprocal loses precision or overflows).
__device__ __forceinline__ float qround(float x, float s, float inv) {
  const float r = x * inv;
  const float q0 = rintf(r);
  if (__builtin_expect(inv == 0.0f || fabsf(r - q0) >= 0.5f - 3.0517578125e-05f, 0))
    return rintf(__fdiv_rn(x, s));
  return q0;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

}  // namespace qg
