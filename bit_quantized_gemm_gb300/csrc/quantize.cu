// quantize.cu -- per-token int8 activation quantization.
//
// Operation (StartLux-Prism README, "Supported models and GPUs": Q8_0 runs as
// int8 W8A8; "How it works": int8 tensor cores with exact int32 sums): for
// each row m, s = absmax/127 (correctly rounded fp32 division) and
// q = clamp(rint(x/s), -127, 127) with the IEEE-rounded quotient and
// ties-to-even; an all-zero row gives s = 0, q = 0. Optional outputs: the
// per-32-block sums of q (the W4A8 min term needs them) and an fp16 copy of q
// (the prefill tensor-core operand).
//
// One CTA per row, 16-byte vector loads of 8 values. The row is held in
// registers between the absmax pass and the quantize pass when it fits
// (K <= kThreads*8*kRegChunks), else re-read (second read hits L2); threads
// and register chunks are chosen from K so that several rows per SM are in
// flight (many rows, or long ones, are re-read: see launch_q_k). HBM-bound:
// per element 2 (bf16) or 4 (fp32) bytes read, 1 (+2 with q16) written.
#include "qg_common.cuh"

namespace qg {


template <bool kBf16>
__device__ __forceinline__ void load_chunk(const void* row, int64_t c, float (&v)[8]) {
  if (kBf16) {
    int4 raw = *reinterpret_cast<const int4*>(reinterpret_cast<const uint16_t*>(row) + c * 8);
    const uint32_t w[4] = {(uint32_t)raw.x, (uint32_t)raw.y, (uint32_t)raw.z, (uint32_t)raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(row) + c * 8);
    float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// kStatic: the scale is given (s_in[m * s_stride], e.g. calibrated once) and
// not computed; values beyond it saturate at +-127.
template <bool kBf16, int kQThreads, int kRegChunks, bool kStatic>
__global__ void __launch_bounds__(kQThreads) quantize_act_kernel(
    const void* __restrict__ x, int64_t ldx, int K, int8_t* __restrict__ q,
    float* __restrict__ scale, int32_t* __restrict__ bsum, __half* __restrict__ q16,
    const float* __restrict__ s_in, int64_t s_stride) {
  // a GEMM launched after this kernel with programmatic stream serialization
  // may start now (its weight streaming overlaps this kernel; it waits for
  // this grid's completion before it reads the activations)
  griddep_launch_dependents();
  const int64_t m = blockIdx.x;
  const int tid = threadIdx.x;
  const int nchunks = K / 8;
  const char* row = reinterpret_cast<const char*>(x) + m * ldx * (kBf16 ? 2 : 4);

  float v[kRegChunks][8];
  float amax = 0.0f;
  if (kStatic) amax = 1.0f;  // no absmax pass: only the given scale matters
  const bool in_regs = nchunks <= kRegChunks * kQThreads;
#pragma unroll
  for (int i = 0; i < kRegChunks; ++i) {
    const int c = tid + i * kQThreads;
    if (c < nchunks) {
      load_chunk<kBf16>(row, c, v[i]);
      if (!kStatic) {
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
    }
  }
  if (!in_regs && !kStatic) {
    for (int c = tid + kRegChunks * kQThreads; c < nchunks; c += kQThreads) {
      float t[8];
      load_chunk<kBf16>(row, c, t);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(t[j]));
    }
  }
  float s;
  if (kStatic) {
    s = s_in[m * s_stride];
  } else {
    // block-wide max
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float red[kQThreads / 32];
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    s = act_scale(amax);
  }
  const bool zero_row = kStatic ? (s == 0.0f) : (amax == 0.0f);
  const float inv = zero_row ? 0.0f : act_scale_rcp(s);
  if (!kStatic && tid == 0) scale[m] = s;

  int8_t* qrow = q ? q + m * (int64_t)K : nullptr;
  __half* hrow = q16 ? q16 + m * (int64_t)K : nullptr;
  int32_t* brow = bsum ? bsum + m * (int64_t)(K / kBlk) : nullptr;

  // All lanes of a warp run every trip of the loops below (invalid chunks
  // compute on zeros and store nothing), so the block-sum shuffles always
  // see the full warp.
  auto emit = [&](int c, bool valid, const float (&t)[8]) {
    float qf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float v = (valid && !zero_row) ? qround(t[j], s, inv) : 0.0f;
      qf[j] = fminf(127.0f, fmaxf(-127.0f, v));
    }
    if (valid) {
      if (qrow) {
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t b0 = (uint32_t)__float2int_rz(qf[4 * h + 0]);
          const uint32_t b1 = (uint32_t)__float2int_rz(qf[4 * h + 1]);
          const uint32_t b2 = (uint32_t)__float2int_rz(qf[4 * h + 2]);
          const uint32_t b3 = (uint32_t)__float2int_rz(qf[4 * h + 3]);
          uint32_t lo, hi;
          asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(lo) : "r"(b0), "r"(b1));  // b0.x, b1.x
          asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(hi) : "r"(b2), "r"(b3));
          asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w[h]) : "r"(lo), "r"(hi));
        }
        *reinterpret_cast<uint2*>(qrow + (int64_t)c * 8) = make_uint2(w[0], w[1]);
      }
      if (hrow) {
        __half2 h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(qf[2 * j], qf[2 * j + 1]);  // exact
        *reinterpret_cast<uint4*>(hrow + (int64_t)c * 8) = *reinterpret_cast<uint4*>(h);
      }
    }
    if (brow) {
      // chunks 4j..4j+3 form block j; their owners are 4 consecutive lanes,
      // all valid or all invalid (the chunk count is a multiple of 4)
      float part = 0.0f;  // exact: |sum| <= 32 * 127
#pragma unroll
      for (int j = 0; j < 8; ++j) part += qf[j];
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      if (valid && (c & 3) == 0) brow[c >> 2] = (int32_t)part;
    }
  };

#pragma unroll
  for (int i = 0; i < kRegChunks; ++i) {
    const int c = tid + i * kQThreads;
    const bool valid = c < nchunks;
    if (in_regs) {
      emit(c, valid, v[i]);
    } else {
      float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (valid) load_chunk<kBf16>(row, c, t);
      emit(c, valid, t);
    }
  }
  if (!in_regs) {
    for (int base = kRegChunks * kQThreads; base < nchunks; base += kQThreads) {
      const int c = base + tid;
      const bool valid = c < nchunks;
      float t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (valid) load_chunk<kBf16>(row, c, t);
      emit(c, valid, t);
    }
  }
}

struct QArgs {
  const void* x;
  int64_t M, K, ldx;
  int8_t* q;
  float* scale;
  int32_t* bsum;
  uint16_t* q16;
  const float* s_in;
  int64_t s_stride;
};

template <bool kBf16, int kT, int kRC, bool kStatic>
static void launch_q(const QArgs& a, cudaStream_t st) {
  quantize_act_kernel<kBf16, kT, kRC, kStatic><<<(unsigned)a.M, kT, 0, st>>>(
      a.x, a.ldx, (int)a.K, a.q, a.scale, a.bsum, reinterpret_cast<__half*>(a.q16), a.s_in,
      a.s_stride);
}

template <bool kBf16, bool kStatic>
static void launch_q_k(const QArgs& a, cudaStream_t st) {
  // Two regimes, measured on GB300 (bf16 rows, us):
  // * many rows (M >= 1024, throughput): a thread holds one 8-value chunk and
  //   re-reads the rest of the row for the quantize pass (from L2), so that
  //   many rows are in flight per SM: 8192 x 5120 47.8 (row held: 51.8),
  //   8192 x 17408 144 (held: 236), 2048 x 9728 31.3 (33.4); rows up to 3072
  //   stay held (2048 x 2560: 15.0 both ways);
  // * few rows (decode sizes, latency): the row is held in registers between
  //   its two passes with threads x chunks x 8 >= K (64 x 5120: 8.8 against
  //   10.9 re-read), and rows longer than 10240 take the 256-thread re-read
  //   configuration (8 x 17408: 15.0 either way).
  const int64_t K = a.K;
  if (K > 256 * 5 * 8 || (a.M >= 1024 && K > 256 * 3 * 8)) {
    launch_q<kBf16, 256, 1, kStatic>(a, st);
  } else if (a.M >= 1024 && K > 128 * 3 * 8) {
    launch_q<kBf16, 128, 1, kStatic>(a, st);
  } else if (K <= 128 * 3 * 8) {
    launch_q<kBf16, 128, 3, kStatic>(a, st);
  } else if (K <= 128 * 5 * 8) {
    launch_q<kBf16, 128, 5, kStatic>(a, st);
  } else {
    launch_q<kBf16, 256, 5, kStatic>(a, st);
  }
}

cudaError_t launch_quantize_act(const void* x, bool bf16, int64_t M, int64_t K, int64_t ldx,
                                int8_t* q, float* scale, int32_t* bsum, uint16_t* q16,
                                cudaStream_t st) {
  const QArgs a{x, M, K, ldx, q, scale, bsum, q16, nullptr, 0};
  if (bf16)
    launch_q_k<true, false>(a, st);
  else
    launch_q_k<false, false>(a, st);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act_static(const void* x, bool bf16, int64_t M, int64_t K,
                                       int64_t ldx, const float* s_in, int64_t s_stride,
                                       int8_t* q, int32_t* bsum, uint16_t* q16,
                                       cudaStream_t st) {
  const QArgs a{x, M, K, ldx, q, nullptr, bsum, q16, s_in, s_stride};
  if (bf16)
    launch_q_k<true, true>(a, st);
  else
    launch_q_k<false, true>(a, st);
  return cudaGetLastError();
}

}  // namespace qg
