// api.cu -- the library's extern "C" entry points (declared in
// include/qgemm.h): host-side argument validation, kernel selection and
// launch. No call allocates memory or synchronizes (qg_check_device_error
// aside, which exists to synchronize).
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "qg_common.cuh"

namespace qg {
cudaError_t launch_quantize_act(const void* x, bool bf16, int64_t M, int64_t K, int64_t ldx,
                                int8_t* q, float* scale, int32_t* bsum, uint16_t* q16,
                                cudaStream_t st);
cudaError_t launch_quantize_act_static(const void* x, bool bf16, int64_t M, int64_t K,
                                       int64_t ldx, const float* s_in, int64_t s_stride,
                                       int8_t* q, int32_t* bsum, uint16_t* q16,
                                       cudaStream_t st);
cudaError_t launch_pack_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                             cudaStream_t st);
cudaError_t launch_pack_q4k(const void* sblocks, int64_t N, int64_t K, void* packed,
                            cudaStream_t st);
cudaError_t launch_pack_mxfp4_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                                   uint32_t* err, cudaStream_t st);
// pdl: launch with programmatic stream serialization (the kernel may start
// while the previous kernel on the stream, the quantize kernel, still runs)
cudaError_t launch_decode_q8_0(const int8_t* qa, const float* sa, int64_t M, int64_t K,
                               const void* packed, int64_t N, void* out, bool out_f32,
                               int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                               cudaStream_t st);
cudaError_t launch_decode_q4k(const int8_t* qa, const float* sa, const int32_t* asum, int64_t M,
                              int64_t K, const void* packed, int64_t N, void* out, bool out_f32,
                              int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                              cudaStream_t st);
cudaError_t launch_prefill_q8_0(const uint16_t* q16, const float* sa, int64_t M, int64_t K,
                                const void* packed, int64_t N, void* out, bool out_f32,
                                int64_t ldo, int32_t* dbg, uint32_t* err, bool pdl,
                                cudaStream_t st);
int prefill_launches_q8_0(int64_t M, int64_t N);
int prefill_tile_q4k(int64_t M, int64_t N, int sms, int* kind);
void prefill_plan_q8_0(int64_t M, int64_t N, int sms, int64_t* rows_wide, int* narrow_kind,
                       int* narrow_tokens);

cudaError_t launch_prefill_q4k(const uint16_t* q16, const float* sa, const int32_t* bsum,
                               int64_t M, int64_t K, const void* packed, int64_t N, void* out,
                               bool out_f32, int64_t ldo, int32_t* dbg, uint32_t* err,
                               bool pdl, cudaStream_t st);
}  // namespace qg

using namespace qg;

// One error word per device that loads the library (module-scope device
// memory, not allocated by any call).
static __device__ uint32_t g_error_word_dev;

// Scratch of qg_linear_w8a8_q8_0_noalloc: module-scope device memory, one
// copy on every device that loads the library, never allocated by a call.
// In host code its name is only a stand-in: the device address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_linear_scratch[QG_LINEAR_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kVersion = 10000;        // 1.0.0
constexpr int64_t kSmallMMax = 16;     // AUTO: decode kernel for M <= 16
constexpr int64_t kDecodeRows = 16;    // rows per decode launch
constexpr int64_t kMaxN = int64_t(1) << 24;
constexpr int64_t kMaxM = int64_t(1) << 24;

thread_local char t_last_error[256] = "";

qg_status fail(qg_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qg_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return QG_OK;
  if (e == cudaErrorNotSupported)
    return fail(QG_EUNSUPPORTED, "%s: tensor-map encoder unavailable in this driver", what);
  return fail(QG_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// address of the device error word on the current device (cached per device)
uint32_t* error_word() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word_dev) != cudaSuccess) return nullptr;
    ptrs[dev] = reinterpret_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

qg_status check_k(int64_t K, int64_t mult) {
  if (K < mult || K % mult != 0 || K > kMaxK)
    return fail(QG_EINVAL, "K=%lld must be a positive multiple of %lld, at most %d",
                (long long)K, (long long)mult, kMaxK);
  return QG_OK;
}

qg_status check_gemm_common(const int8_t* q, const uint16_t* q16, const float* scale, int64_t M,
                            int64_t K, const void* w, int64_t N, void* out, qg_dtype odt,
                            int64_t ldo, qg_path path, int64_t kmult, bool* large) {
  if (!scale || !w || !out) return fail(QG_EINVAL, "null pointer argument");
  if (M < 1 || M > kMaxM) return fail(QG_EINVAL, "M=%lld out of range [1, 2^24]", (long long)M);
  if (N < 1 || N > kMaxN) return fail(QG_EINVAL, "N=%lld out of range [1, 2^24]", (long long)N);
  qg_status s = check_k(K, kmult);
  if (s != QG_OK) return s;
  if (odt != QG_BF16 && odt != QG_F32) return fail(QG_EINVAL, "out_dtype must be QG_BF16 or QG_F32");
  if (ldo < N) return fail(QG_EINVAL, "ldo=%lld < N=%lld", (long long)ldo, (long long)N);
  if ((q && !aligned(q, 16)) || !aligned(out, 16) || !aligned(w, 256) || !aligned(scale, 4))
    return fail(QG_EALIGN, "q and out need 16-byte, w_packed 256-byte, scale 4-byte alignment");
  if (q16 && !aligned(q16, 16)) return fail(QG_EALIGN, "q16 needs 16-byte alignment");
  if (path != QG_PATH_AUTO && path != QG_PATH_SMALL && path != QG_PATH_LARGE)
    return fail(QG_EINVAL, "unknown path %d", (int)path);
  *large = (path == QG_PATH_LARGE) || (path == QG_PATH_AUTO && M > kSmallMMax);
  if (!*large && !q)
    return fail(QG_EINVAL,
                "the decode kernel (M <= %lld or QG_PATH_SMALL) reads q, the int8 activations",
                (long long)kSmallMMax);
  if (*large && !q16)
    return fail(QG_EINVAL,
                "the prefill kernel (M > %lld or QG_PATH_LARGE) needs q16, the fp16 copy of q "
                "written by qg_quantize_act",
                (long long)kSmallMMax);
  return QG_OK;
}

template <typename F>
qg_status decode_chunks(int64_t M, int64_t K, int64_t N, int64_t ldo, size_t out_esize,
                        void* out, int32_t* dbg, F&& launch) {
  // the decode kernel takes up to 16 rows per launch; rows are independent
  for (int64_t m0 = 0; m0 < M; m0 += kDecodeRows) {
    const int64_t mc = (M - m0) < kDecodeRows ? (M - m0) : kDecodeRows;
    void* o = out ? reinterpret_cast<char*>(out) + m0 * ldo * out_esize : nullptr;
    int32_t* d = dbg ? dbg + m0 * N * (K / kBlk) : nullptr;
    qg_status s = from_cuda(launch(m0, mc, o, d), "decode GEMM launch");
    if (s != QG_OK) return s;
  }
  return QG_OK;
}

// Workspace of qg_linear_*, each part 256-byte aligned:
// the row scales [M] (unless the caller passes scale_out), then the int8
// activations [M][K] (decode kernel, M <= kSmallMMax) or their fp16 copy
// [M][K] (prefill kernel), then for W4A8 the block sums [M][K/32].
struct LinearWs {
  int64_t off_scale, off_act, off_bsum, total;
  LinearWs(bool q4k, int64_t M, int64_t K) {
    off_scale = 0;
    off_act = align_up(M * 4, 256);
    const int64_t act = M <= kSmallMMax ? M * K : M * K * 2;
    off_bsum = align_up(off_act + act, 256);
    total = align_up(off_bsum + (q4k ? M * (K / kBlk) * 4 : 0), 256);
  }
};

qg_status linear(bool q4k, const void* x, qg_dtype xdt, int64_t M, int64_t K, int64_t ldx,
                 const void* w, int64_t N, void* out, qg_dtype odt, int64_t ldo, float* scale_out,
                 void* ws, size_t ws_bytes, void* stream) {
  if (!x || !w || !out) return fail(QG_EINVAL, "null pointer argument");
  if (xdt != QG_BF16 && xdt != QG_F32) return fail(QG_EINVAL, "x_dtype must be QG_BF16 or QG_F32");
  if (odt != QG_BF16 && odt != QG_F32) return fail(QG_EINVAL, "out_dtype must be QG_BF16 or QG_F32");
  if (M < 1 || M > kMaxM) return fail(QG_EINVAL, "M=%lld out of range [1, 2^24]", (long long)M);
  if (N < 1 || N > kMaxN) return fail(QG_EINVAL, "N=%lld out of range [1, 2^24]", (long long)N);
  qg_status s = check_k(K, q4k ? kQ4kWeights : kBlk);
  if (s != QG_OK) return s;
  const int64_t es = xdt == QG_BF16 ? 2 : 4;
  if (ldx < K) return fail(QG_EINVAL, "ldx=%lld < K=%lld", (long long)ldx, (long long)K);
  if (ldo < N) return fail(QG_EINVAL, "ldo=%lld < N=%lld", (long long)ldo, (long long)N);
  if (!aligned(x, 16) || (ldx * es) % 16 != 0)
    return fail(QG_EALIGN, "x needs 16-byte alignment and a row stride that is a multiple of 16 bytes");
  if (!aligned(out, 16) || !aligned(w, 256) || (scale_out && !aligned(scale_out, 4)))
    return fail(QG_EALIGN, "out needs 16-byte, w_packed 256-byte, scale_out 4-byte alignment");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool f32 = odt == QG_F32;
  const LinearWs L(q4k, M, K);
  if (!ws || ws_bytes < (size_t)L.total)
    return fail(QG_EINVAL, "workspace of %lld bytes needed for M=%lld (qg_linear_workspace_bytes)",
                (long long)L.total, (long long)M);
  if (!aligned(ws, 256)) return fail(QG_EALIGN, "workspace needs 256-byte alignment");
  char* base = reinterpret_cast<char*>(ws);
  float* scale = scale_out ? scale_out : reinterpret_cast<float*>(base + L.off_scale);
  const bool small = M <= kSmallMMax;
  int8_t* q = small ? reinterpret_cast<int8_t*>(base + L.off_act) : nullptr;
  uint16_t* q16 = small ? nullptr : reinterpret_cast<uint16_t*>(base + L.off_act);
  int32_t* bsum = q4k ? reinterpret_cast<int32_t*>(base + L.off_bsum) : nullptr;
  bool large = false;
  s = check_gemm_common(q, q16, scale, M, K, w, N, out, odt, ldo, QG_PATH_AUTO,
                        q4k ? kQ4kWeights : kBlk, &large);
  if (s != QG_OK) return s;
  s = from_cuda(launch_quantize_act(x, xdt == QG_BF16, M, K, ldx, q, scale, bsum, q16, st),
                "quantize launch");
  if (s != QG_OK) return s;
  // The GEMM's first launch (decode or prefill kernel) is a programmatic dependent of the
  // quantize kernel: its CTAs start, and request their first weight stages,
  // while the activations are quantized
  if (large)
    return from_cuda(q4k ? launch_prefill_q4k(q16, scale, bsum, M, K, w, N, out, f32, ldo, nullptr,
                                              error_word(), true, st)
                         : launch_prefill_q8_0(q16, scale, M, K, w, N, out, f32, ldo, nullptr,
                                               error_word(), true, st),
                     "prefill GEMM launch");
  return from_cuda(q4k ? launch_decode_q4k(q, scale, bsum, M, K, w, N, out, f32, ldo, nullptr,
                                           error_word(), true, st)
                       : launch_decode_q8_0(q, scale, M, K, w, N, out, f32, ldo, nullptr,
                                            error_word(), true, st),
                   "decode GEMM launch");
}

// Device address of g_linear_scratch on the current device, looked up once
// per device (with that device current) and cached; nullptr if the lookup
// fails.
void* linear_scratch() {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_linear_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" {

const char* qg_status_string(qg_status s) {
  switch (s) {
    case QG_OK: return "QG_OK";
    case QG_EINVAL: return "QG_EINVAL: invalid argument";
    case QG_EALIGN: return "QG_EALIGN: misaligned pointer or stride";
    case QG_EUNSUPPORTED: return "QG_EUNSUPPORTED: not supported";
    case QG_ECUDA: return "QG_ECUDA: CUDA error";
    case QG_ETIMEOUT: return "QG_ETIMEOUT: a device-side wait gave up";
  }
  return "unknown qg_status";
}

const char* qg_last_error(void) { return t_last_error; }
int qg_version(void) { return kVersion; }
int64_t qg_small_m_max(void) { return kSmallMMax; }

int qg_gemm_launch_count(int weights_kind, int64_t M, int64_t K, int64_t N, qg_path path) {
  if (weights_kind != 0 && weights_kind != 1) return 0;
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN) return 0;
  if (check_k(K, weights_kind ? kQ4kWeights : kBlk) != QG_OK) return 0;
  if (path != QG_PATH_AUTO && path != QG_PATH_SMALL && path != QG_PATH_LARGE) return 0;
  const bool large = (path == QG_PATH_LARGE) || (path == QG_PATH_AUTO && M > kSmallMMax);
  if (!large) return (int)ceil_div(M, kDecodeRows);
  return weights_kind ? 1 : prefill_launches_q8_0(M, N);
}

qg_status qg_debug_prefill_plan_q8_0(int64_t M, int64_t N, int sms, int64_t* rows_wide,
                                     int* narrow_kind, int* narrow_tokens) {
  if (!rows_wide || !narrow_kind || !narrow_tokens) return fail(QG_EINVAL, "null pointer argument");
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN)
    return fail(QG_EINVAL, "M, N out of range [1, 2^24]");
  if (sms < 1 || sms > 4096) return fail(QG_EINVAL, "sms=%d out of range [1, 4096]", sms);
  prefill_plan_q8_0(M, N, sms, rows_wide, narrow_kind, narrow_tokens);
  return QG_OK;
}

qg_status qg_debug_prefill_tile_q4k(int64_t M, int64_t N, int sms, int* kind, int* tokens) {
  if (!kind || !tokens) return fail(QG_EINVAL, "null pointer argument");
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN)
    return fail(QG_EINVAL, "M, N out of range [1, 2^24]");
  if (sms < 1 || sms > 4096) return fail(QG_EINVAL, "sms=%d out of range [1, 4096]", sms);
  *tokens = prefill_tile_q4k(M, N, sms, kind);
  return QG_OK;
}

qg_status qg_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(QG_ECUDA, "stream synchronize: %s", cudaGetErrorString(e));
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_error_word_dev, sizeof(v));
  if (e != cudaSuccess) return fail(QG_ECUDA, "read error word: %s", cudaGetErrorString(e));
  if (v) {
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_error_word_dev, &zero, sizeof(zero));
    if (v & kErrTimeout)
      return fail(QG_ETIMEOUT, "device error word 0x%x: a bounded barrier wait gave up", v);
    return fail(QG_ERANGE,
                "device error word 0x%x: a packed MXFP4 block scale is outside fp16's range "
                "(the decode kernels' scales)", v);
  }
  return QG_OK;
}

qg_status qg_quantize_act(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                          int8_t* q, float* scale, int32_t* block_sums, uint16_t* q16,
                          void* stream) {
  if (!x || !scale) return fail(QG_EINVAL, "null pointer argument");
  if (!q && !q16) return fail(QG_EINVAL, "q and q16 are both NULL: no activations to write");
  if (x_dtype != QG_BF16 && x_dtype != QG_F32) return fail(QG_EINVAL, "x_dtype must be QG_BF16 or QG_F32");
  if (M < 1 || M > kMaxM) return fail(QG_EINVAL, "M=%lld out of range [1, 2^24]", (long long)M);
  qg_status s = check_k(K, kBlk);
  if (s != QG_OK) return s;
  const int64_t es = x_dtype == QG_BF16 ? 2 : 4;
  if (ldx < K) return fail(QG_EINVAL, "ldx=%lld < K=%lld", (long long)ldx, (long long)K);
  if (!aligned(x, 16) || (ldx * es) % 16 != 0)
    return fail(QG_EALIGN, "x needs 16-byte alignment and a row stride that is a multiple of 16 bytes");
  if ((q && !aligned(q, 16)) || !aligned(scale, 4) || (block_sums && !aligned(block_sums, 4)) ||
      (q16 && !aligned(q16, 16)))
    return fail(QG_EALIGN, "q and q16 need 16-byte, scale and block_sums 4-byte alignment");
  return from_cuda(launch_quantize_act(x, x_dtype == QG_BF16, M, K, ldx, q, scale, block_sums, q16,
                                       reinterpret_cast<cudaStream_t>(stream)),
                   "quantize launch");
}

qg_status qg_quantize_act_static(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                                 int64_t ldx, const float* scale, int64_t scale_stride, int8_t* q,
                                 int32_t* block_sums, uint16_t* q16, void* stream) {
  if (!x || !scale) return fail(QG_EINVAL, "null pointer argument");
  if (!q && !q16) return fail(QG_EINVAL, "q and q16 are both NULL: no activations to write");
  if (x_dtype != QG_BF16 && x_dtype != QG_F32) return fail(QG_EINVAL, "x_dtype must be QG_BF16 or QG_F32");
  if (M < 1 || M > kMaxM) return fail(QG_EINVAL, "M=%lld out of range [1, 2^24]", (long long)M);
  if (scale_stride != 0 && scale_stride != 1) return fail(QG_EINVAL, "scale_stride must be 0 or 1");
  qg_status s = check_k(K, kBlk);
  if (s != QG_OK) return s;
  const int64_t es = x_dtype == QG_BF16 ? 2 : 4;
  if (ldx < K) return fail(QG_EINVAL, "ldx=%lld < K=%lld", (long long)ldx, (long long)K);
  if (!aligned(x, 16) || (ldx * es) % 16 != 0)
    return fail(QG_EALIGN, "x needs 16-byte alignment and a row stride that is a multiple of 16 bytes");
  if ((q && !aligned(q, 16)) || !aligned(scale, 4) || (block_sums && !aligned(block_sums, 16)) ||
      (q16 && !aligned(q16, 16)))
    return fail(QG_EALIGN, "q and q16 need 16-byte, block_sums 16-byte, scale 4-byte alignment");
  return from_cuda(launch_quantize_act_static(x, x_dtype == QG_BF16, M, K, ldx, scale,
                                              scale_stride, q, block_sums, q16,
                                              reinterpret_cast<cudaStream_t>(stream)),
                   "quantize launch");
}

size_t qg_q8_0_packed_bytes(int64_t N, int64_t K) {
  if (N < 1 || N > kMaxN || K < kBlk || K % kBlk || K > kMaxK) return 0;
  return (size_t)Q8Layout(N, K).total;
}

size_t qg_q4k_packed_bytes(int64_t N, int64_t K) {
  if (N < 1 || N > kMaxN || K < kQ4kWeights || K % kQ4kWeights || K > kMaxK) return 0;
  return (size_t)Q4kLayout(N, K).total;
}

qg_status qg_pack_q8_0(const void* blocks, int64_t N, int64_t K, void* packed, void* stream) {
  if (!blocks || !packed) return fail(QG_EINVAL, "null pointer argument");
  if (N < 1 || N > kMaxN) return fail(QG_EINVAL, "N=%lld out of range [1, 2^24]", (long long)N);
  qg_status s = check_k(K, kBlk);
  if (s != QG_OK) return s;
  if (!aligned(packed, 256)) return fail(QG_EALIGN, "packed needs 256-byte alignment");
  return from_cuda(launch_pack_q8_0(blocks, N, K, packed, reinterpret_cast<cudaStream_t>(stream)),
                   "pack launch");
}

qg_status qg_pack_q4k(const void* sblocks, int64_t N, int64_t K, void* packed, void* stream) {
  if (!sblocks || !packed) return fail(QG_EINVAL, "null pointer argument");
  if (N < 1 || N > kMaxN) return fail(QG_EINVAL, "N=%lld out of range [1, 2^24]", (long long)N);
  qg_status s = check_k(K, kQ4kWeights);
  if (s != QG_OK) return s;
  if (!aligned(packed, 256)) return fail(QG_EALIGN, "packed needs 256-byte alignment");
  return from_cuda(launch_pack_q4k(sblocks, N, K, packed, reinterpret_cast<cudaStream_t>(stream)),
                   "pack launch");
}

static qg_status gemm_q8_0(const int8_t* q, const uint16_t* q16, const float* scale, int64_t M,
                           int64_t K, const void* w, int64_t N, void* out, qg_dtype odt,
                           int64_t ldo, qg_path path, int32_t* dbg, void* stream) {
  bool large = false;
  qg_status s = check_gemm_common(q, q16, scale, M, K, w, N, dbg ? reinterpret_cast<void*>(dbg) : out,
                                  odt, dbg ? N : ldo, path, kBlk, &large);
  if (s != QG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool f32 = odt == QG_F32;
  if (large)
    return from_cuda(launch_prefill_q8_0(q16, scale, M, K, w, N, out, f32, ldo, dbg, error_word(), false, st),
                     "prefill GEMM launch");
  return decode_chunks(M, K, N, ldo, f32 ? 4 : 2, out, dbg,
                       [&](int64_t m0, int64_t mc, void* o, int32_t* d) {
                         return launch_decode_q8_0(q + m0 * K, scale + m0, mc, K, w, N, o, f32,
                                                   ldo, d, error_word(), false, st);
                       });
}

static qg_status gemm_q4k(const int8_t* q, const uint16_t* q16, const float* scale,
                          const int32_t* bsum, int64_t M, int64_t K, const void* w, int64_t N,
                          void* out, qg_dtype odt, int64_t ldo, qg_path path, int32_t* dbg,
                          void* stream) {
  if (!bsum) return fail(QG_EINVAL, "block_sums is required for W4A8");
  if (!aligned(bsum, 16)) return fail(QG_EALIGN, "block_sums needs 16-byte alignment");
  bool large = false;
  qg_status s = check_gemm_common(q, q16, scale, M, K, w, N, dbg ? reinterpret_cast<void*>(dbg) : out,
                                  odt, dbg ? N : ldo, path, kQ4kWeights, &large);
  if (s != QG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool f32 = odt == QG_F32;
  if (large)
    return from_cuda(
        launch_prefill_q4k(q16, scale, bsum, M, K, w, N, out, f32, ldo, dbg, error_word(), false, st),
        "prefill GEMM launch");
  const int64_t B = K / kBlk;
  return decode_chunks(M, K, N, ldo, f32 ? 4 : 2, out, dbg,
                       [&](int64_t m0, int64_t mc, void* o, int32_t* d) {
                         return launch_decode_q4k(q + m0 * K, scale + m0, bsum + m0 * B, mc, K, w,
                                                  N, o, f32, ldo, d, error_word(), false, st);
                       });
}

qg_status qg_gemm_w8a8_q8_0_ex(const int8_t* q, const uint16_t* q16, const float* scale,
                               int64_t M, int64_t K, const void* w_packed, int64_t N, void* out,
                               qg_dtype out_dtype, int64_t ldo, qg_path path, void* stream) {
  return gemm_q8_0(q, q16, scale, M, K, w_packed, N, out, out_dtype, ldo, path, nullptr, stream);
}

qg_status qg_gemm_w8a8_q8_0(const int8_t* q, const uint16_t* q16, const float* scale, int64_t M,
                            int64_t K, const void* w_packed, int64_t N, void* out,
                            qg_dtype out_dtype, int64_t ldo, void* stream) {
  return gemm_q8_0(q, q16, scale, M, K, w_packed, N, out, out_dtype, ldo, QG_PATH_AUTO, nullptr,
                   stream);
}

qg_status qg_gemm_w4a8_q4k_ex(const int8_t* q, const uint16_t* q16, const float* scale,
                              const int32_t* block_sums, int64_t M, int64_t K,
                              const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                              int64_t ldo, qg_path path, void* stream) {
  return gemm_q4k(q, q16, scale, block_sums, M, K, w_packed, N, out, out_dtype, ldo, path, nullptr,
                  stream);
}

qg_status qg_gemm_w4a8_q4k(const int8_t* q, const uint16_t* q16, const float* scale,
                           const int32_t* block_sums, int64_t M, int64_t K, const void* w_packed,
                           int64_t N, void* out, qg_dtype out_dtype, int64_t ldo, void* stream) {
  return gemm_q4k(q, q16, scale, block_sums, M, K, w_packed, N, out, out_dtype, ldo, QG_PATH_AUTO,
                  nullptr, stream);
}

size_t qg_linear_workspace_bytes(int weights_kind, int64_t M, int64_t K) {
  if (weights_kind != 0 && weights_kind != 1) return 0;
  if (M < 1 || M > kMaxM || check_k(K, weights_kind ? kQ4kWeights : kBlk) != QG_OK) return 0;
  return (size_t)LinearWs(weights_kind == 1, M, K).total;
}

qg_status qg_linear_w8a8_q8_0(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                              const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                              int64_t ldo, float* scale_out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return linear(false, x, x_dtype, M, K, ldx, w_packed, N, out, out_dtype, ldo, scale_out,
                workspace, workspace_bytes, stream);
}

qg_status qg_linear_w4a8_q4k(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                             const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                             int64_t ldo, float* scale_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return linear(true, x, x_dtype, M, K, ldx, w_packed, N, out, out_dtype, ldo, scale_out,
                workspace, workspace_bytes, stream);
}

size_t qg_mxfp4_packed_bytes(int64_t N, int64_t K) { return qg_q8_0_packed_bytes(N, K); }

qg_status qg_pack_mxfp4_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                             void* stream) {
  if (!blocks || !packed) return fail(QG_EINVAL, "null pointer argument");
  if (N < 1 || N > kMaxN) return fail(QG_EINVAL, "N=%lld out of range [1, 2^24]", (long long)N);
  qg_status s = check_k(K, kBlk);
  if (s != QG_OK) return s;
  if (!aligned(packed, 256)) return fail(QG_EALIGN, "packed needs 256-byte alignment");
  return from_cuda(launch_pack_mxfp4_q8_0(blocks, N, K, packed, error_word(),
                                          reinterpret_cast<cudaStream_t>(stream)),
                   "pack launch");
}

// The converted weights are integers 2v with scales 2^(E-128) in the Q8_0
// packed layout: the W8A8 GEMM and layer call run them unchanged.
qg_status qg_gemm_w4a8_mxfp4(const int8_t* q, const uint16_t* q16, const float* scale,
                             int64_t M, int64_t K, const void* w_packed, int64_t N, void* out,
                             qg_dtype out_dtype, int64_t ldo, void* stream) {
  return gemm_q8_0(q, q16, scale, M, K, w_packed, N, out, out_dtype, ldo, QG_PATH_AUTO, nullptr,
                   stream);
}

qg_status qg_linear_w4a8_mxfp4(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                               int64_t ldx, const void* w_packed, int64_t N, void* out,
                               qg_dtype out_dtype, int64_t ldo, float* scale_out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return linear(false, x, x_dtype, M, K, ldx, w_packed, N, out, out_dtype, ldo, scale_out,
                workspace, workspace_bytes, stream);
}

qg_status qg_linear_w8a8_q8_0_noalloc(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                                      int64_t ldx, const void* w_packed, int64_t N, void* out,
                                      qg_dtype out_dtype, int64_t ldo, float* scale_out,
                                      void* stream) {
  // 0 when M or K is invalid: linear() then reports which, before any use of
  // the workspace
  const size_t need = qg_linear_workspace_bytes(0, M, K);
  if (need > QG_LINEAR_NOALLOC_SCRATCH_BYTES)
    return fail(QG_EINVAL,
                "M=%lld, K=%lld need %llu bytes of scratch, more than the %llu of the static "
                "scratch; call qg_linear_w8a8_q8_0 with a workspace",
                (long long)M, (long long)K, (unsigned long long)need,
                (unsigned long long)QG_LINEAR_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  if (need > 0) {
    ws = linear_scratch();
    if (!ws) return fail(QG_ECUDA, "no device address for the static scratch on this device");
  }
  return linear(false, x, x_dtype, M, K, ldx, w_packed, N, out, out_dtype, ldo, scale_out, ws,
                ws ? QG_LINEAR_NOALLOC_SCRATCH_BYTES : 0, stream);
}

// A single bounded wait on a barrier that nothing arrives at: after `polls`
// polls it records a timeout in the device error word and returns.
__global__ void wait_timeout_probe_kernel(uint32_t polls, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, polls);
}

qg_status qg_debug_wait_timeout(uint32_t polls, void* stream) {
  if (polls == 0 || polls > (1u << 20)) return fail(QG_EINVAL, "polls must be in [1, 2^20]");
  uint32_t* err = error_word();
  if (!err) return fail(QG_ECUDA, "no device error word on the current device");
  wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(polls, err);
  return from_cuda(cudaGetLastError(), "timeout probe launch");
}

static qg_status check_debug(const int32_t* isum, int64_t M, int64_t K, int64_t N) {
  if (!isum) return fail(QG_EINVAL, "null isum");
  if (M < 1 || N < 1 || K < kBlk) return fail(QG_EINVAL, "bad sizes");
  if (M * N * (K / kBlk) > (int64_t(1) << 28)) return fail(QG_EINVAL, "debug export too large");
  return QG_OK;
}

qg_status qg_debug_block_sums_q8_0(const int8_t* q, const uint16_t* q16, int64_t M, int64_t K,
                                   const void* w_packed, int64_t N, int32_t* isum, qg_path path,
                                   void* stream) {
  qg_status s = check_debug(isum, M, K, N);
  if (s != QG_OK) return s;
  // scale is unused in debug mode; pass q as a non-null 4-byte aligned stand-in
  return gemm_q8_0(q, q16, reinterpret_cast<const float*>(isum), M, K, w_packed, N, nullptr,
                   QG_F32, N, path, isum, stream);
}

qg_status qg_debug_block_sums_q4k(const int8_t* q, const uint16_t* q16, int64_t M, int64_t K,
                                  const void* w_packed, int64_t N, int32_t* isum, qg_path path,
                                  void* stream) {
  qg_status s = check_debug(isum, M, K, N);
  if (s != QG_OK) return s;
  return gemm_q4k(q, q16, reinterpret_cast<const float*>(isum), isum, M, K, w_packed, N, nullptr,
                  QG_F32, N, path, isum, stream);
}

}  // extern "C"
