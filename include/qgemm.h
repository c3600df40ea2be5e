/*
 * qgemm.h -- C ABI of the exact int8 (W8A8) / W4A8 quantized linear layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the StartLux-Prism README describes:
 *   - "Why StartLux-Prism", bullet "The released files as they are": Q8_0
 *     weights run as int8 (W8A8), Q4_K_M weights on their own 4-bit values
 *     (W4A8), with no conversion of the file's numbers;
 *   - "Why StartLux-Prism", bullet "Reproducible to the bit", and "How it
 *     works", bullet on int8 tensor cores: integer products are summed
 *     exactly in int32, so a row's result does not depend on the other rows
 *     of its batch.
 * The pages print no formula or layout; this library fixes them as follows.
 *
 *   Activation quantization, per row m (token):
 *     s[m] = absmax_k |x[m,k]| / 127            (fp32, correctly rounded)
 *     q[m,k] = clamp(rint(x[m,k] / s[m]), -127, 127)   (IEEE division,
 *                                                  ties to even)
 *     an all-zero row gives s = 0 and q = 0.
 *   W8A8 with Q8_0 weights (block b = 32 consecutive k, scale d[n,b]):
 *     isum = sum_{k in b} q[m,k] * qw[n,k]          (exact int32)
 *     acc  = fmaf((float)isum, d[n,b], acc)          for b = 0, 1, ... in order
 *     y    = acc * s[m];  out = bf16(y) (round to nearest even) or y (fp32)
 *   W4A8 with Q4_K weights (sub-block b = 32 k, super-block = 8 sub-blocks):
 *     ds = d * sc_b, dm = dmin * m_b                 (exact fp32 products)
 *     isum = sum q[m,k] * qw[n,k],  asum = sum q[m,k] (exact int32)
 *     acc = fmaf((float)isum, ds, acc); acc = fmaf(-(float)asum, dm, acc)
 *     y = acc * s[m];  out as above.
 * Every path of this library produces these bits exactly, so results are
 * identical whatever the batch size M, the rows' positions, or the path
 * (decode or prefill kernel) chosen.
 *
 * Conventions for every call below.
 *   - All data pointers are DEVICE pointers, allocated and owned by the
 *     caller; the library allocates no memory and keeps no state between
 *     calls. Sizes are element counts unless stated otherwise.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream; no call
 *     synchronizes.
 *   - Arguments are validated on the host before any launch. A rejected call
 *     launches nothing and returns QG_EINVAL / QG_EALIGN / QG_EUNSUPPORTED;
 *     qg_last_error() then holds a one-line reason (thread-local).
 *   - A failed launch returns QG_ECUDA. Device-side waits are bounded: a wait
 *     that gives up records itself in a device error word, which
 *     qg_check_device_error() reads (it synchronizes its stream).
 *   - Nothing aborts and nothing prints.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QG_OK = 0,
  QG_EINVAL = 1,        /* null pointer, non-positive or inconsistent size  */
  QG_EALIGN = 2,        /* pointer or leading dimension not aligned         */
  QG_EUNSUPPORTED = 3,  /* valid request that no kernel here implements     */
  QG_ECUDA = 4,         /* CUDA runtime/launch error                        */
  QG_ETIMEOUT = 5,      /* a bounded device-side wait gave up               */
  QG_ERANGE = 6         /* a packed value outside its format's range        */
} qg_status;

typedef enum { QG_BF16 = 0, QG_F32 = 1 } qg_dtype;

/* Kernel selection for the *_ex GEMM calls. AUTO picks the weight-streaming
 * decode kernel for M <= qg_small_m_max() and the tensor-memory prefill
 * kernel above it. Both give identical bits; forcing one is for tests and
 * measurements. */
typedef enum { QG_PATH_AUTO = 0, QG_PATH_SMALL = 1, QG_PATH_LARGE = 2 } qg_path;

const char* qg_status_string(qg_status s);
/* One-line reason for the last non-OK status returned on this thread. */
const char* qg_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int qg_version(void);
/* Largest M the AUTO path sends to the decode kernel. */
int64_t qg_small_m_max(void);
/* Synchronizes `stream`, then reads and clears the device error word of the
 * current device: QG_OK, or QG_ETIMEOUT if a bounded wait gave up. */
qg_status qg_check_device_error(void* stream);
/* Number of kernel launches one qg_gemm_w8a8_q8_0(_ex) (weights_kind 0) or
 * qg_gemm_w4a8_q4k(_ex) (weights_kind 1) call with these sizes and path
 * makes on the current device: the decode kernel takes up to 16 rows per
 * launch; the prefill kernel runs as one launch, or, for W8A8 shapes whose
 * last wave of 256-token tiles would leave most SMs idle, as two (the rows
 * that fill whole waves, then the rest as narrow tiles). 0 if the sizes or
 * the path are invalid. Host-only: launches nothing; reads the SM count. */
int qg_gemm_launch_count(int weights_kind, int64_t M, int64_t K, int64_t N, qg_path path);

/* ------------------------------------------------------------------------ */
/* Activation quantization (per token, dynamic absmax; see the definition    */
/* above).                                                                   */
/*   x          [M][ldx] of x_dtype (QG_BF16 or QG_F32), rows of K values;   */
/*              16-byte aligned, ldx >= K, ldx*elem_size % 16 == 0.          */
/*   q          [M][K] int8 out, 16-byte aligned, or NULL when only q16 is   */
/*              wanted (the prefill kernel reads q16 alone).                 */
/*   scale      [M] fp32 out.                                                */
/*   block_sums [M][K/32] int32 out (sum of q over each 32-wide block, needed */
/*              by the W4A8 GEMM), or NULL.                                   */
/*   q16        [M][K] fp16 out holding the same integers as q (exact), the  */
/*              operand of the prefill tensor-core kernel, or NULL. 16-byte   */
/*              aligned. q and q16 are not both NULL (QG_EINVAL).             */
/* K must be a positive multiple of 32 and at most 65536; M >= 1.             */
/* ------------------------------------------------------------------------ */
qg_status qg_quantize_act(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                          int8_t* q, float* scale, int32_t* block_sums, uint16_t* q16,
                          void* stream);

/* ------------------------------------------------------------------------ */
/* Activation quantization with given scales (ranges calibrated once and     */
/* cached, as the StartLux-Prism README's engine does at its first start,    */
/* "Quick start"; the calibration itself is the caller's).                   */
/*   row m uses s = scale[m * scale_stride] (scale_stride 1: per row, [M];    */
/*   0: one scale for every row, [1]);                                        */
/*   q = clamp(rint(x / s), -127, 127), IEEE division, ties to even; values  */
/*   beyond the calibrated range saturate; s == 0 gives q = 0.               */
/* x, q, block_sums, q16 as for qg_quantize_act (block_sums 16-byte aligned).*/
/* The GEMMs take the same scale array as their activation scale ([M]; pass  */
/* a per-row array when the calibration is per tensor).                      */
/* ------------------------------------------------------------------------ */
qg_status qg_quantize_act_static(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                                 int64_t ldx, const float* scale, int64_t scale_stride, int8_t* q,
                                 int32_t* block_sums, uint16_t* q16, void* stream);

/* ------------------------------------------------------------------------ */
/* Q8_0 weights (W8A8).                                                      */
/* Input format: the weight matrix W [N][K] as N*K/32 blocks of 34 bytes,    */
/* row-major over (n, b): {fp16 d (little endian); int8 q[32]}, weight =     */
/* d*q. qg_pack_q8_0 rearranges them once into the library's opaque packed   */
/* buffer (qg_q8_0_packed_bytes(N, K) bytes, 256-byte aligned, caller-owned), */
/* which holds the int8 values in the decode kernels' order, the            */
/* scales, and an fp16 copy of the values for the prefill kernel. The values  */
/* are never changed: d and q reach the arithmetic bit for bit.              */
/*   blocks  device, [N][K/32][34] bytes (no alignment needed).              */
/*   K % 32 == 0, 32 <= K <= 65536, 1 <= N <= 2^24.                          */
/* ------------------------------------------------------------------------ */
size_t qg_q8_0_packed_bytes(int64_t N, int64_t K);
qg_status qg_pack_q8_0(const void* blocks, int64_t N, int64_t K, void* packed, void* stream);

/* out[m][n] = the W8A8 result above for m < M, n < N.
 *   q, scale  from qg_quantize_act ([M][K] int8, [M] fp32). q is read only by
 *             the decode kernel (M <= qg_small_m_max() under AUTO, or
 *             QG_PATH_SMALL) and may be NULL when the prefill kernel runs.
 *   q16       the fp16 copy from qg_quantize_act; required when the prefill
 *             kernel runs (M > qg_small_m_max() under AUTO), else may be NULL.
 *   w_packed  from qg_pack_q8_0 with the same N, K.
 *   out       [M][ldo] of out_dtype, 16-byte aligned, ldo >= N.
 * Rows are independent: the bits of row m depend only on q[m], scale[m] and
 * the weights. */
qg_status qg_gemm_w8a8_q8_0(const int8_t* q, const uint16_t* q16, const float* scale,
                            int64_t M, int64_t K, const void* w_packed, int64_t N,
                            void* out, qg_dtype out_dtype, int64_t ldo, void* stream);
qg_status qg_gemm_w8a8_q8_0_ex(const int8_t* q, const uint16_t* q16, const float* scale,
                               int64_t M, int64_t K, const void* w_packed, int64_t N,
                               void* out, qg_dtype out_dtype, int64_t ldo, qg_path path,
                               void* stream);

/* ------------------------------------------------------------------------ */
/* Q4_K weights (W4A8).                                                      */
/* Input format: W [N][K] as N*K/256 super-blocks of 144 bytes (this         */
/* library's canonical packing; the pages give none):                        */
/*   bytes 0-1 d, 2-3 dmin (fp16, little endian);                            */
/*   bytes 4-15 a 96-bit little-endian string of sixteen 6-bit fields, field */
/*     f at bits [6f, 6f+6): sc_0..sc_7 then m_0..m_7;                        */
/*   bytes 16-143 4-bit q: weight j (0..255) is the low nibble of byte       */
/*     16 + j/2 for even j, the high nibble for odd j.                       */
/*   weight(j) = d*sc_i*q_j - dmin*m_i, i = j/32.                            */
/*   K % 256 == 0, 256 <= K <= 65536, 1 <= N <= 2^24.                         */
/* ------------------------------------------------------------------------ */
size_t qg_q4k_packed_bytes(int64_t N, int64_t K);
qg_status qg_pack_q4k(const void* superblocks, int64_t N, int64_t K, void* packed, void* stream);

/* out[m][n] = the W4A8 result above.
 *   block_sums  [M][K/32] int32 from qg_quantize_act (required, 16-byte
 *               aligned).
 *   Other arguments as for qg_gemm_w8a8_q8_0. */
qg_status qg_gemm_w4a8_q4k(const int8_t* q, const uint16_t* q16, const float* scale,
                           const int32_t* block_sums, int64_t M, int64_t K,
                           const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                           int64_t ldo, void* stream);
qg_status qg_gemm_w4a8_q4k_ex(const int8_t* q, const uint16_t* q16, const float* scale,
                              const int32_t* block_sums, int64_t M, int64_t K,
                              const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                              int64_t ldo, qg_path path, void* stream);

/* ------------------------------------------------------------------------ */
/* The whole layer in one call: x in, y out. qg_quantize_act (the dynamic    */
/* per-token scales) into the caller's workspace, then the GEMM (AUTO), with */
/* the bits of those two calls made separately.                              */
/*   The GEMM's first launch (decode kernel for M <= qg_small_m_max(),      */
/*     prefill or 16-row kernel above) is a programmatic dependent of the    */
/*     quantize kernel: its CTAs start while the rows are quantized, request */
/*     their first weight stages, and read activations and scales only after */
/*     the quantize grid has completed.                                      */
/*   x          [M][ldx] of x_dtype, 16-byte aligned, ldx >= K,              */
/*              ldx*elem_size % 16 == 0.                                      */
/*   w_packed   from qg_pack_q8_0 / qg_pack_q4k with the same N, K.          */
/*   out        [M][ldo] of out_dtype, 16-byte aligned, ldo >= N.             */
/*   scale_out  [M] fp32: receives the row scales s[m] (else they stay in    */
/*              the workspace), or NULL.                                      */
/*   workspace  device memory of at least qg_linear_workspace_bytes(kind, M, */
/*              K) bytes, 256-byte aligned, owned by the caller: the row      */
/*              scales, the quantized activations (int8 for the decode        */
/*              kernel, fp16 for the prefill kernel) and, for W4A8, the       */
/*              block sums.                                                   */
/* K as for the GEMM (multiple of 32; of 256 for Q4_K), M >= 1.               */
/* ------------------------------------------------------------------------ */
/* Workspace bytes for qg_linear_w8a8_q8_0 (weights_kind 0) or               */
/* qg_linear_w4a8_q4k (weights_kind 1) with these sizes; 0 if the sizes are  */
/* invalid. Host-only. */
size_t qg_linear_workspace_bytes(int weights_kind, int64_t M, int64_t K);
qg_status qg_linear_w8a8_q8_0(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                              const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                              int64_t ldo, float* scale_out, void* workspace,
                              size_t workspace_bytes, void* stream);
qg_status qg_linear_w4a8_q4k(const void* x, qg_dtype x_dtype, int64_t M, int64_t K, int64_t ldx,
                             const void* w_packed, int64_t N, void* out, qg_dtype out_dtype,
                             int64_t ldo, float* scale_out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* MXFP4 weights from Q8_0 (StartLux-Prism README, "Supported models and     */
/* GPUs" and "Blackwell MXFP4": --precision mxfp4 runs the MLP's projections */
/* in MXFP4, from a Q8_0 file, at lower precision). Lossy in the conversion  */
/* only: qg_pack_mxfp4_q8_0 rounds each Q8_0 block to MXFP4 -- 32 values     */
/* sharing X = 2^(E-127), E = floor(log2 max|w|) - 2 + 127 (an all-zero       */
/* block: 127), each w/X to the nearest E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4, */
/* 6, signed; ties to the even mantissa; saturating at 6). Twice an E2M1     */
/* value is an integer in [-12, 12], so the GEMM is the W8A8 one on integer  */
/* weights 2v with block scales X/2 = 2^(E-128): exact int32 block sums and  */
/* the same fixed-order fp32 epilogue, bit-reproducible like W8A8.           */
/*   qg_mxfp4_packed_bytes / qg_pack_mxfp4_q8_0: as qg_q8_0_packed_bytes /   */
/*     qg_pack_q8_0 (the same layout and buffer rules); the packed values    */
/*     are the converted ones. A block whose X/2 lies outside fp16's range   */
/*     (2^-24 .. 2^15; the decode kernels hold block scales in fp16) makes   */
/*     the next qg_check_device_error() return QG_ERANGE; such a buffer must */
/*     not be used by the decode kernel (M <= qg_small_m_max()).             */
/*   qg_gemm_w4a8_mxfp4, qg_linear_w4a8_mxfp4: as qg_gemm_w8a8_q8_0 and       */
/*     qg_linear_w8a8_q8_0 (workspace kind 0), on a buffer from               */
/*     qg_pack_mxfp4_q8_0.                                                    */
/* The pages ran this on Blackwell's block-scaled tensor cores; here the     */
/* integer sums run on the int8 paths and the power-of-two block scale is     */
/* applied in the fixed-order fp32 epilogue, so the bits stay reproducible.   */
/* ------------------------------------------------------------------------ */
size_t qg_mxfp4_packed_bytes(int64_t N, int64_t K);
qg_status qg_pack_mxfp4_q8_0(const void* blocks, int64_t N, int64_t K, void* packed,
                             void* stream);
qg_status qg_gemm_w4a8_mxfp4(const int8_t* q, const uint16_t* q16, const float* scale,
                             int64_t M, int64_t K, const void* w_packed, int64_t N, void* out,
                             qg_dtype out_dtype, int64_t ldo, void* stream);
qg_status qg_linear_w4a8_mxfp4(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                               int64_t ldx, const void* w_packed, int64_t N, void* out,
                               qg_dtype out_dtype, int64_t ldo, float* scale_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* The W8A8 layer call without a workspace argument and without allocating   */
/* (the pages have no counterpart: this is a convenience of this library).   */
/* For callers that cannot call cudaMalloc: a host that hands a plug-in only  */
/* its input and output buffers across a C interface, or a latency-critical   */
/* loop where an allocation (cudaMalloc and cudaFree synchronize the device)  */
/* is not acceptable. The scratch that qg_linear_w8a8_q8_0 takes from its     */
/* caller lives here in one module-scope device array of                     */
/* QG_LINEAR_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the     */
/* library holds until the process exits.                                    */
/*   Arguments, results and bits as for qg_linear_w8a8_q8_0 (scale_out may   */
/*   be NULL).                                                               */
/*   Limit: qg_linear_workspace_bytes(0, M, K) <= QG_LINEAR_NOALLOC_SCRATCH_  */
/*   BYTES (every M <= qg_small_m_max() at any K; larger M while M*K*2 plus  */
/*   the row scales fit); larger sizes return QG_EINVAL and launch nothing.  */
/*   The first call on a device looks the array's device address up for that */
/*   device (the device current at the call); make that first call before   */
/*   any stream capture. It returns QG_ECUDA if the lookup fails.            */
/*   Every call on a device shares the one array, and it keeps the last      */
/*   call's contents: nothing in it needs to start at zero (the quantize     */
/*   kernel writes every byte the GEMM then reads). Calls whose work overlaps */
/*   on the GPU (other streams, other threads) race on it and give wrong     */
/*   results; order them on one stream or use qg_linear_w8a8_q8_0 with a     */
/*   workspace each.                                                         */
/* ------------------------------------------------------------------------ */
#define QG_LINEAR_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
qg_status qg_linear_w8a8_q8_0_noalloc(const void* x, qg_dtype x_dtype, int64_t M, int64_t K,
                                      int64_t ldx, const void* w_packed, int64_t N, void* out,
                                      qg_dtype out_dtype, int64_t ldo, float* scale_out,
                                      void* stream);

/* ------------------------------------------------------------------------ */
/* Test support: the exact per-block integer sums as the chosen kernel sees   */
/* them, isum[m][n][b] (int32, [M][N][K/32]), taken from the same kernels     */
/* (decode: the int8 MMA accumulators; prefill: the tensor-memory block       */
/* accumulators), for checking exactness. Small shapes only:                 */
/* M*N*(K/32) <= 2^28. For Q4_K the same layout holds sum q_a*q (4-bit q).   */
/* ------------------------------------------------------------------------ */
qg_status qg_debug_block_sums_q8_0(const int8_t* q, const uint16_t* q16, int64_t M, int64_t K,
                                   const void* w_packed, int64_t N, int32_t* isum,
                                   qg_path path, void* stream);
qg_status qg_debug_block_sums_q4k(const int8_t* q, const uint16_t* q16, int64_t M, int64_t K,
                                  const void* w_packed, int64_t N, int32_t* isum,
                                  qg_path path, void* stream);

/* Test support: the wave plan of the W8A8 prefill kernel for an M x N GEMM on
 * a GPU of `sms` SMs, as qg_gemm_w8a8_q8_0 carries it out there (M above
 * qg_small_m_max(), AUTO). Host-only; launches nothing.
 *   rows_wide      weight rows [0, rows_wide) run as 256-token tiles in one
 *                  launch (N: the whole GEMM is that launch);
 *   narrow_kind    the remaining rows, all tokens, in a second launch: 0 none,
 *                  1 tensor-memory tiles, 2 16-row tiles (legacy fp16 MMA);
 *   narrow_tokens  that launch's token-tile width (0 when there is none).
 * The plan never changes a bit of the result. */
qg_status qg_debug_prefill_plan_q8_0(int64_t M, int64_t N, int sms, int64_t* rows_wide,
                                     int* narrow_kind, int* narrow_tokens);

/* Test support: the tiles of the W4A8 GEMM for M x N on a GPU of `sms` SMs,
 * as qg_gemm_w4a8_q4k carries it out there (M above qg_small_m_max(), AUTO;
 * one launch): *kind 1 = tensor-memory tiles of 128 weight rows, 2 = tiles of
 * 16 weight rows (legacy fp16 MMA); *tokens = the token-tile width (32, 64,
 * 128 or 256). Host-only; launches nothing. The tiles never change a bit of
 * the result. */
qg_status qg_debug_prefill_tile_q4k(int64_t M, int64_t N, int sms, int* kind, int* tokens);

/* Test support for failure detection: launches one bounded wait on a
 * barrier that nothing completes; after `polls` polls (1 .. 2^20) it records
 * a timeout in the device error word and returns, leaving the context usable.
 * The following qg_check_device_error() reports QG_ETIMEOUT and clears it. */
qg_status qg_debug_wait_timeout(uint32_t polls, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_H */
