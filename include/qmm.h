/*
 * qmm.h -- C ABI of the quantized projection matmul library for one GB300 (sm_103a).
 *
 * Two halves, and two widenings of the second:
 *   (I)   an exact int8 GEMM with zero-point correction, per-column weight
 *         scale, optional int32 bias and float or requantised output, and the
 *         int8 quantisation of its activations;
 *   (II)  a 4-bit block-weight GEMM/GEMV over 32x256 tiles of q4_1 blocks and
 *         its MUL_MAT_ID (mixture-of-experts) variant;
 *   (III) W8A16: int8 weights with block scales times bf16 activations;
 *   (IV)  more weight formats: Q4_K repacked into q4_1 tiles, and 8-bit (Q8)
 *         tiles in two code layouts.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *   except the size outputs (size_t*) and the epilogue struct, which are host
 *   pointers.
 * - The caller allocates and owns every buffer.  No entry point allocates or
 *   frees device memory, synchronises the stream, or keeps mutable state
 *   between calls.  There are three exceptions: a per-process cache of the
 *   driver entry point used to build TMA descriptors, a per-process cache of
 *   the grouped GEMV's launch plans (keyed by the problems' shapes), and the
 *   fixed scratch array of qmm_q4_gemm_id_noalloc (see there).  Pointers are
 *   borrowed until the work queued on `stream` has finished.
 * - Work is queued on `stream` and runs asynchronously.  Argument errors are
 *   found on the host and returned at once, and nothing is launched when a
 *   check fails.
 * - Errors found on the device go to `dev_status`, a device int32 that the
 *   caller sets to 0 (it may be NULL).  These are a bounded wait that ran out
 *   (QMM_ERR_TIMEOUT), an expert id outside [0, n_expert)
 *   (QMM_ERR_BAD_EXPERT_ID), a per-axis zero point outside its operand's
 *   domain (QMM_ERR_INVALID_ARG), and a weight block that the f16 tensor-core
 *   route cannot form (QMM_ERR_RANGE).  The library only ever replaces a 0
 *   there with an error code, so the caller reads it after synchronising.
 * - Shapes the library has no kernel for return QMM_ERR_UNSUPPORTED.  There
 *   is no fallback path.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QMM_OK = 0,
  QMM_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, type or zero point */
  QMM_ERR_UNSUPPORTED = 2,     /* valid request the library has no kernel for */
  QMM_ERR_OVERFLOW_BOUND = 3,  /* K*255*128 >= 2^31: int32 sums could overflow */
  QMM_ERR_CUDA = 4,            /* a CUDA runtime call failed (e.g. launch) */
  QMM_ERR_TIMEOUT = 5,         /* device: a bounded pipeline wait gave up */
  QMM_ERR_BAD_EXPERT_ID = 6,   /* device: an expert id was outside [0, n_expert) */
  QMM_ERR_WORKSPACE = 7,       /* workspace pointer NULL, misaligned or smaller than required */
  QMM_ERR_RANGE = 8            /* device: a weight block beyond f16's range (|w| could pass 65504) on a
                                  route that forms f16 weights; the results of that call are not valid */
} qmm_status;

typedef enum {
  QMM_U8 = 1,
  QMM_S8 = 2,
  QMM_S32 = 3,
  QMM_F32 = 4,
  QMM_BF16 = 5
} qmm_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* qmm_status_string(qmm_status s);

/* Library ABI version (major*10000 + minor*100 + patch). */
int qmm_version(void);

/* ========================================================================
 * (I) int8 GEMM
 *
 * Defined by "int8 inference" (recursiveai.org/onemodel/docs/int8/),
 * section "Product kernel (Int8Gemm)":
 *     A' = A - 128 for uint8 A, A for int8 (B the same);
 *     zA' = zA - 128 for uint8 A (zB' likewise);
 *     S[m,n] = sum_k A'[m,k] B'[k,n]                        (exact int32)
 *     Y[m,n] = S - zA' colSum[n] - zB' (rowSum[m] - K zA')   (= sum (A-zA)(B-zB))
 * followed by the epilogue, in this order: optional int32 bias, then the
 * output conversion.  "The ONNX pack: weights to Q4NX, matmuls to our
 * kernels, no VitisAI", sections "The three layers of the pack" and "What
 * works today", fixes packB's scale = amax/127, the float dequant
 * C = Cm * s_x[m] * s_w[n], and the fused QuantizeLinear
 * y_q = clamp(round_half_even(C * s_x s_w / s_y) + zp_y).
 * ======================================================================== */

/* Packed-weight size: N rows of Kp = K rounded up to 64 bytes. */
qmm_status qmm_pack_b_int8_size(int64_t K, int64_t N, size_t* packed_bytes);

/* packB: build the kernel's weight layout once per weight.
 *
 * B        [K][N] row-major, row stride `ldb` elements (ldb >= N).
 * b_type   QMM_F32: quantise each column, s = amax/127 (fp32, IEEE division),
 *                   q = clamp(round_half_even(W/s), -127, 127); a zero column
 *                   gets s = 0 and q = 0.  Scales go to col_scale[N].
 *          QMM_S8 / QMM_U8: integer weights, stored shifted (B' = B, or B-128
 *                   for uint8); col_scale is not touched (may be NULL).
 * packed   int8 [N][Kp], K-major (byte n*Kp + k holds B'[k][n]; bytes k >= K
 *          are 0).  Base 16-byte aligned, `packed_bytes` >= qmm_pack_b_int8_size.
 * col_sum  int32 [N]: colSum[n] = sum_k B'[k][n], kept beside the weight.
 * Errors: QMM_ERR_INVALID_ARG for null/misaligned pointers, K < 1, N < 1,
 * ldb < N or a bad type; QMM_ERR_OVERFLOW_BOUND when K*255*128 >= 2^31.
 */
qmm_status qmm_pack_b_int8(const void* B, qmm_dtype b_type, int64_t K, int64_t N, int64_t ldb,
                           void* packed, size_t packed_bytes, float* col_scale, int32_t* col_sum,
                           cudaStream_t stream);

/* Epilogue of qmm_int8_gemm (all pointers device, [N] or [M] fp32/int32). */
typedef struct {
  qmm_dtype out_type;      /* QMM_S32 (Y + bias), QMM_F32, QMM_S8 or QMM_U8 */
  const int32_t* bias;     /* [N] int32 added to Y before any conversion, or NULL */
  const float* s_x;        /* activation scale: NULL means 1.0 */
  int64_t s_x_stride;      /* 0: per-tensor s_x[0]; 1: per-row s_x[m] */
  const float* s_w;        /* [N] per-column weight scale, or NULL for 1.0 */
  float s_y;               /* output scale (S8/U8 only), > 0 */
  int32_t zp_y;            /* output zero point (S8/U8 only), added after rounding */
} qmm_epilogue;

/* Workspace the int8 GEMM needs for an (M, K, N) call (0 when none). */
qmm_status qmm_int8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);

/* Y = A (x) packB with zero points, bias and the chosen output.
 *
 * A        [M][K] uint8 or int8 (a_type), row stride lda bytes: lda >= K,
 *          lda % 16 == 0, base 16-byte aligned.  zA in A's own domain.  The
 *          kernels read whole 16-byte groups, so A must be readable for
 *          (M - 1) * lda + roundup(K, 16) bytes, as an [M][lda] tensor is;
 *          the bytes past K do not change the result.
 * packedB  from qmm_pack_b_int8 with the same K and N; col_sum from the same call.
 * b_orig_type  the b_type given to packB (QMM_U8, QMM_S8 or QMM_F32); zB is in
 *          that domain and must be 0 for QMM_F32 weights (symmetric).
 * ep       epilogue (host pointer to the struct; its arrays are device).
 * out      [M][N] with row stride ldo elements of the output type (ldo >= N).
 * workspace / ws_bytes  device scratch of at least
 *          qmm_int8_gemm_workspace_size(M, K, N) bytes, 256-byte aligned
 *          (may be NULL when that size is 0).
 * Output conversions (fp32 IEEE, round-to-nearest-even, no contraction):
 *   S32: Yb = Y + bias
 *   F32: fl(fl(fl(Yb) * s_x[m]) * s_w[n])
 *   S8/U8: Mq = fl(fl(s_x[m] * s_w[n]) / s_y); q = rint_even(fl(fl(Yb) * Mq)) + zp_y,
 *          clamped to the output type's range.
 * The result is bit-exact and independent of the kernel chosen.  The caller
 * must keep |Y|, |Y + bias| < 2^31.
 * Errors: as packB, plus QMM_ERR_OVERFLOW_BOUND for K*255*128 >= 2^31,
 * QMM_ERR_INVALID_ARG for zero points outside the operand domain, and
 * QMM_ERR_WORKSPACE.  Device status: QMM_ERR_TIMEOUT.
 */
qmm_status qmm_int8_gemm(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda,
                         int32_t zA, const void* packedB, const int32_t* col_sum, int64_t N,
                         qmm_dtype b_orig_type, int32_t zB, const qmm_epilogue* ep, void* out,
                         int64_t ldo, void* workspace, size_t ws_bytes, int32_t* dev_status,
                         cudaStream_t stream);

/* Static weights widened once ("int8 inference", "Product kernel (Int8Gemm)":
 * packB is a one-time weight transform, and so is this).  The tensor-core
 * route (M >= 65) multiplies f16 copies of the codes, exact for every int8
 * value; qmm_int8_gemm widens the packed weights on every call, while
 * qmm_int8_gemm_b16 reads a copy made here once, so a call only widens A.
 *
 * qmm_widen_b_int8_size: bytes of that copy, N * roundup(K, 64) * 2.
 * qmm_widen_b_int8: packedB (from qmm_pack_b_int8 with the same K and N,
 *          16-byte aligned) -> b16, f16 [N][roundup(K, 64)] of the packed
 *          codes B' (the padding columns are zeros), device, 16-byte aligned,
 *          b16_bytes at least the size above; owned by the caller and valid as
 *          long as packedB is unchanged.  Asynchronous on `stream`.
 * qmm_int8_gemm_b16_workspace_size: workspace of qmm_int8_gemm_b16 (smaller
 *          than qmm_int8_gemm's: no room for the widened weights).
 * qmm_int8_gemm_b16: exactly qmm_int8_gemm (same arguments, checks, routes
 *          and results, bit for bit), with b16 (non-NULL) the copy of
 *          packedB.  M <= 64 routes read packedB and ignore b16.
 * Errors: QMM_ERR_INVALID_ARG for a NULL or misaligned b16 or a short
 *          b16_bytes, else as qmm_int8_gemm / qmm_pack_b_int8.
 */
qmm_status qmm_widen_b_int8_size(int64_t K, int64_t N, size_t* b16_bytes);
qmm_status qmm_widen_b_int8(const void* packedB, int64_t K, int64_t N, void* b16, size_t b16_bytes,
                            int32_t* dev_status, cudaStream_t stream);
qmm_status qmm_int8_gemm_b16_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);
qmm_status qmm_int8_gemm_b16(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda, int32_t zA,
                             const void* packedB, const void* b16, const int32_t* col_sum, int64_t N,
                             qmm_dtype b_orig_type, int32_t zB, const qmm_epilogue* ep, void* out, int64_t ldo,
                             void* workspace, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream);

/* One int8 GEMM of a grouped call: the arguments of qmm_int8_gemm, with the
 * epilogue held by value. */
typedef struct qmm_int8_problem {
  const void* A;
  qmm_dtype a_type;
  int64_t M, K, lda;
  int32_t zA;
  const void* packedB;
  const int32_t* col_sum;
  int64_t N;
  qmm_dtype b_orig_type;
  int32_t zB;
  qmm_epilogue ep;
  void* out;
  int64_t ldo;
} qmm_int8_problem;

/* Several independent small-M int8 GEMMs in one launch (one per 16 problems):
 * each computes exactly what qmm_int8_gemm computes for its arguments,
 * bit-exact.  Small batches of tokens run several projections whose weight
 * streams are each too short to keep the GPU busy ("The ONNX pack: weights to
 * Q4NX, matmuls to our kernels, no VitisAI", "What works today": the per-call
 * cost of the M = 16 / 32 projection GEMMs); one launch streams them together.
 *
 * problems  HOST array of `count` descriptors, read during the call only.
 *           Every problem needs M <= 64 (else QMM_ERR_UNSUPPORTED) and passes
 *           qmm_int8_gemm's checks (the first failing status is returned
 *           before anything is queued).  No workspace is used.  An output
 *           must not overlap any input or other output of the group.
 */
qmm_status qmm_int8_gemm_group(const qmm_int8_problem* problems, int64_t count, int32_t* dev_status,
                               cudaStream_t stream);

/* Workspace of qmm_int8_gemm_axis_zp: the int32 product [M][N] and the row
 * sums [M], each rounded up to 256 bytes, plus qmm_int8_gemm_workspace_size. */
qmm_status qmm_int8_gemm_axis_zp_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);

/* qmm_int8_gemm with per-axis zero points: one per activation row and one per
 * weight column ("The ONNX pack...", "What works today": the asymmetric
 * corrections come per tensor, or per row and per column wherever the scales are,
 * exact in integers):
 *     Y[m,n] = sum_k (A[m,k] - zA[m]) (B[k,n] - zB[n])
 *            = S - zA'[m] colSum[n] - zB'[n] (rowSum[m] - K zA'[m])
 * then the same bias and output conversion as qmm_int8_gemm (bit-exact).
 *
 * zA   device int32 [M], each in A's domain (0..255 for QMM_U8, -128..127 for
 *      QMM_S8), or NULL for all zeros.
 * zB   device int32 [N] in the domain of b_orig_type (QMM_U8 / QMM_S8), or NULL
 *      for all zeros; must be NULL for QMM_F32 weights (symmetric).
 * All other arguments as qmm_int8_gemm, except the workspace, which must hold
 * qmm_int8_gemm_axis_zp_workspace_size(M, K, N) bytes (256-byte aligned).
 * The exact product goes through the per-tensor GEMM into the workspace
 * (int32), and one more pass applies the corrections, the bias and the output
 * conversion: the call costs an int32 write and read of M x N more than
 * qmm_int8_gemm.
 * Errors: as qmm_int8_gemm.  Zero points are device data: one outside its
 * domain sets QMM_ERR_INVALID_ARG in dev_status, and the outputs are then
 * unspecified.
 */
qmm_status qmm_int8_gemm_axis_zp(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda,
                                 const int32_t* zA, const void* packedB, const int32_t* col_sum, int64_t N,
                                 qmm_dtype b_orig_type, const int32_t* zB, const qmm_epilogue* ep, void* out,
                                 int64_t ldo, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 cudaStream_t stream);

/* Workspace of qmm_quantize_act_int8: 256 bytes for per-tensor scaling, 0 per row. */
qmm_status qmm_quantize_act_int8_workspace_size(int64_t M, int64_t K, int per_row, size_t* ws_bytes);

/* Symmetric int8 quantisation of activations for qmm_int8_gemm ("int8
 * inference", "Product kernel (Int8Gemm)": per-tensor symmetric activations
 * with scale amax/127; the ONNX pack page, "What works today": the per-row
 * scale vector s_x[m] of the float epilogue).  The rule is packB's, applied to
 * each row (per_row = 1) or to the whole tensor (per_row = 0):
 *   s    = fl(amax / 127), amax = max |X| over the row or the tensor;
 *   A[m][k] = clamp(rint_even(fl(X[m][k] / s)), -127, 127), and 0 where s == 0.
 * Every step is IEEE fp32, so the codes and scales are bit-exact.
 *
 * X        [M][K] fp32 (x_type QMM_F32) or bf16 (QMM_BF16), row stride ldx
 *          elements (ldx >= K), base aligned to its element size.
 * A        int8 [M][K] out, row stride lda bytes: lda >= K, lda % 16 == 0, base
 *          16-byte aligned (what qmm_int8_gemm takes, with a_type QMM_S8 and
 *          zA = 0).  Bytes past K in a row are not written.
 * s_x      fp32 out: [M] per row, [1] per tensor.  Pass it as the epilogue's s_x
 *          with s_x_stride = per_row.
 * workspace / ws_bytes  at least qmm_quantize_act_int8_workspace_size bytes,
 *          16-byte aligned (NULL when that size is 0).
 * X must be finite: for an inf or NaN input the codes and scales are
 * unspecified.
 * Errors: QMM_ERR_INVALID_ARG for null or misaligned pointers, M < 1, K < 1,
 * ldx < K, a bad lda or x_type, per_row not 0 or 1; QMM_ERR_WORKSPACE.
 */
qmm_status qmm_quantize_act_int8(const void* X, qmm_dtype x_type, int64_t M, int64_t K, int64_t ldx,
                                 int per_row, void* A, int64_t lda, float* s_x, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream);

/* ========================================================================
 * (II) 4-bit block weights
 *
 * Tile geometry from "NPU engine: full ELFs, no xclbin", section "Q4NX
 * chunks".  A weight of N rows (outputs) x K columns (inputs) is a grid of
 * 32-row x 256-column tiles, 5120 bytes each, stored row-major over the grid
 * ([N/32][K/256] tiles).  The q4_1 semantics come from "Zaya 8B Q4NX on the
 * AMD NPU", round 26: w = q * scale + min, where q is a 4-bit code 0..15 and
 * scale and min are bf16, one pair per (row, 32-column block).
 *
 * The byte map inside a tile is this library's own, because the pages do not
 * print one:
 *   bytes [0, 4096)    codes: row r owns bytes [128 r, 128 r + 128); block b
 *                      (columns 32 b .. 32 b + 31) is the 16 bytes at
 *                      128 r + 16 b, as 4 little-endian uint32 words; word t
 *                      (t = 0..3) holds the codes of columns 32 b + 8 t + j,
 *                      j = 0..7, with code j = 2i in bits [4i, 4i+4) and code
 *                      j = 2i+1 in bits [16+4i, 16+4i+4).
 *   bytes [4096, 5120) (scale, min) bf16 pairs: the pair of (row r, block b)
 *                      sits at byte 4096 + 4 (8 r + b), scale in the low half.
 * ======================================================================== */

/* Tile bytes of an N x K weight: (N/32) * (K/256) * 5120. */
qmm_status qmm_pack_q4_size(int64_t N, int64_t K, size_t* tile_bytes);

/* Quantise fp32 W [N][K] (row stride ldw elements, ldw >= K) into tiles.
 * Per block of 32 consecutive k of one row (fp32 IEEE steps):
 *   s = bf16_rne((max - min) / 15), m = bf16_rne(min),
 *   q = clamp(rint_even((x - m) / s), 0, 15), q = 0 where s == 0.
 * Requires N % 32 == 0 and K % 256 == 0 (else QMM_ERR_UNSUPPORTED); tiles
 * 16-byte aligned with tile_bytes >= qmm_pack_q4_size.
 */
qmm_status qmm_pack_q4(const float* W, int64_t N, int64_t K, int64_t ldw, void* tiles,
                       size_t tile_bytes, cudaStream_t stream);

/* Workspace of qmm_q4_gemm: 0 for M <= 16 (the decode GEMV), else the
 * activations as f16 rows (M*K*2 bytes) and one fp32 scale per row, each
 * rounded up to 256 bytes. */
qmm_status qmm_q4_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);

/* Y[m][n] = sum_k X[m][k] * w[n][k] with fp32 accumulation.
 *
 * tiles  one N x K tile set (16-byte aligned).  N % 32 == 0, K % 256 == 0.
 * X      bf16 [M][K], row stride ldx elements (ldx >= K, ldx % 8 == 0, base
 *        16-byte aligned).
 * Y      fp32 [M][N], row stride ldy elements (ldy >= N).
 * workspace / ws_bytes  qmm_q4_gemm_workspace_size bytes, 256-byte aligned
 *        (NULL when that size is 0), rewritten by the call.
 * Small M (<= 16) runs the decode GEMV, which never rounds a weight: only
 * fp32 summation rounds, within 2e-5 * sum_k |x||w|.  Larger M runs the
 * tensor-core GEMM on f16 operands: each weight is rounded once to f16
 * (<= 2^-11 of itself), and each activation row is scaled by a power of two
 * before its f16 conversion, which makes that conversion exact for every
 * element within a factor 2^31 of the row's largest.  With every block's
 * scale and min in f16's normal range (|s|, |m| >= 2^-14, or 0), each weight
 * is within max(2^-11 |w|, 2^-25) of its exact value, so for every input
 *     |y - y_exact| <= (2^-11 + K * 2^-23) * sum_k |x||w| + 2^-25 * sum' |x|,
 * where sum' runs over the weights with |w| < 2^-14 (K * 2^-23 bounds the
 * fp32 accumulation even if every addition truncates).  The first term is
 * below 2e-3 * sum_k |x||w| for K <= 12,544.  A block whose scale or min is
 * below 2^-14 adds at most 17 * 2^-25 * |x| per weight.  A block with
 * |m| + 15 |s| > 65504 cannot be formed in f16: dev_status gets QMM_ERR_RANGE.
 */
qmm_status qmm_q4_gemm(const void* tiles, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                       int32_t* dev_status, cudaStream_t stream);

/* One decode GEMV (M = 1) of a grouped call: y = W x for one q4 tile set. */
typedef struct qmm_q4_gemv_problem {
  const void* tiles; /* device: one N x K tile set, 16-byte aligned */
  int64_t N;         /* N % 32 == 0 */
  int64_t K;         /* K % 256 == 0 */
  const void* x;     /* device: bf16 [K], 16-byte aligned */
  float* y;          /* device: fp32 [N], 4-byte aligned */
} qmm_q4_gemv_problem;

/* Several independent decode GEMVs in one launch: y_i[n] = sum_k x_i[k] w_i[n][k]
 * for each problem i, the function qmm_q4_gemm computes at M = 1 and with the
 * same bound (weights never rounded; fp32 summation only, within
 * 2e-5 * sum_k |x||w|).  Decode runs many small projections, each too small to
 * keep the memory system busy by itself ("Zaya 8B Q4NX on the AMD NPU", round
 * 25n: a launch-bound step; round 25p: one stream of packed weights feeding
 * several matmuls).  The call spreads the tile rows of all problems over the
 * GPU's SMs, balanced by bytes, so that the group streams as one weight set.
 *
 * problems  HOST array of `count` descriptors, read during the call only.
 *           A y buffer must not overlap any tiles, x or other y of the group.
 * count     1 <= count; any number of problems (the call launches one kernel
 *           per 32 problems or per 6,144 tile rows; a problem with K > 16,384
 *           or more than 6,144 tile rows runs as its own qmm_q4_gemm launch).
 * Sizes are checked on the host; a bad descriptor returns QMM_ERR_INVALID_ARG
 * (null pointer, misalignment) or QMM_ERR_UNSUPPORTED (N % 32, K % 256) before
 * anything is queued.  Results are deterministic: each output is summed in a
 * fixed order, with no atomics.
 */
qmm_status qmm_q4_gemv_group(const qmm_q4_gemv_problem* problems, int64_t count, int32_t* dev_status,
                             cudaStream_t stream);

/* Workspace of qmm_q4_gemm_id: routing tables for n_expert experts and
 * P = T*n_used (token, slot) pairs (int32 offsets [n_expert+1], int32 pair ids
 * [P] and fp32 activation-row scales [P], each padded to 256 bytes), followed
 * by the pairs' activation rows packed in expert order as f16 [P][K]. */
qmm_status qmm_q4_gemm_id_workspace_size(int64_t n_expert, int64_t n_used, int64_t T, int64_t K,
                                         size_t* ws_bytes);

/* MUL_MAT_ID over q4 experts ("Zaya 8B Q4NX on the AMD NPU": the new
 * MUL_MAT_ID_Q4NX op; "The bugs that were the work"; the down-projection fix
 * of the rounds 24-28 notes).  It runs the tensor-core route of qmm_q4_gemm
 * (f16 operands) with the same accuracy bound and QMM_ERR_RANGE report.
 *
 * tiles     n_expert consecutive N x K tile sets (expert e starts at byte
 *           e * qmm_pack_q4_size(N, K)).
 * X         bf16 activations.  Slot i of token t reads the row at element
 *           offset t*ldx_token + i*ldx_slot: ldx_slot = 0 gives the shared src1
 *           of gate/up ([T][K]); ldx_slot = K gives the per-slot src1 of down
 *           ([T][n_used][K]).  ldx_token and ldx_slot % 8 == 0.
 * ids       int32, a STRIDED view: the expert of (t, i) is ids[t*ld_ids + i]
 *           (ld_ids >= n_used, e.g. 17 for the top-8 of 17 sorted ids).
 * Y         fp32; row (t, i) starts at element t*ldy_token + i*ldy_slot.
 * workspace device scratch (256-byte aligned), rewritten on every call.
 *           qmm_q4_gemm_id_workspace_size bytes run the fastest path, which
 *           packs the activation rows in expert order.  A workspace that holds
 *           only the routing tables and row scales runs a path that gathers
 *           the rows inside the grouped kernel (same results); anything
 *           smaller returns QMM_ERR_WORKSPACE.
 * Y[t][i][n] = sum_k x(t,i)[k] * w_{ids(t,i)}[n][k].  A pair whose id is
 * outside [0, n_expert) is skipped (its output row is left untouched) and
 * dev_status gets QMM_ERR_BAD_EXPERT_ID.
 */
qmm_status qmm_q4_gemm_id(const void* tiles, int64_t n_expert, int64_t N, int64_t K,
                          const void* X, int64_t ldx_token, int64_t ldx_slot, const int32_t* ids,
                          int64_t ld_ids, int64_t n_used, int64_t T, float* Y, int64_t ldy_token,
                          int64_t ldy_slot, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, cudaStream_t stream);

/* The gate/up pair of a mixture-of-experts layer in one MUL_MAT_ID call:
 * Y_gate = MUL_MAT_ID(tiles_gate) and Y_up = MUL_MAT_ID(tiles_up), each exactly
 * what qmm_q4_gemm_id computes for its weights (same bound).  Both weight sets
 * read the same ids and the same shared src1 row of each token, so the
 * routing and the packed activations are built once and one grouped launch
 * streams both sets ("Zaya 8B Q4NX on the AMD NPU", round 25p: one packed
 * activation stream feeding several matmuls).
 *
 * tiles_gate, tiles_up  n_expert consecutive N x K tile sets each (same N, K).
 * X       bf16 [T][K] with row stride ldx_token (the shared src1).
 * Y_gate, Y_up  fp32 [T][n_used][N], both with strides ldy_token / ldy_slot.
 * workspace  qmm_q4_gemm_id_workspace_size(n_expert, n_used, T, K) bytes (the
 *         same as one qmm_q4_gemm_id call); a tables-only workspace runs the
 *         gather mode as there.
 * Other arguments, checks and device status as qmm_q4_gemm_id.
 */
qmm_status qmm_q4_gemm_id_pair(const void* tiles_gate, const void* tiles_up, int64_t n_expert, int64_t N,
                               int64_t K, const void* X, int64_t ldx_token, const int32_t* ids, int64_t ld_ids,
                               int64_t n_used, int64_t T, float* Y_gate, float* Y_up, int64_t ldy_token,
                               int64_t ldy_slot, void* workspace, size_t ws_bytes, int32_t* dev_status,
                               cudaStream_t stream);

/* MUL_MAT_ID for callers that cannot allocate device memory.  No counterpart
 * on the pages: this is a convenience of this library.
 *
 * Callers that cannot call cudaMalloc use this entry point.  Examples are a
 * plugin whose host framework owns every device buffer and passes it only
 * inputs and outputs, and a latency-critical path where an allocation (which
 * may synchronise the device) is not allowed.  The call computes exactly what
 * qmm_q4_gemm_id computes, with the same arguments minus the workspace.  The
 * routing tables and activation-row scales live in a fixed scratch array
 * inside the library's own device memory (528,640 bytes, held on every GPU
 * that loads the library until the process exits), so the call allocates
 * nothing.  When the packed activation rows fit in the rest of the array
 * (small calls) they are packed there; larger calls gather the rows inside
 * the grouped kernel.
 *
 * Limits: n_expert <= 1024 and T * n_used <= 65536; larger requests return
 * QMM_ERR_WORKSPACE.
 * - The first call on each device looks up the scratch array's device
 *   address and caches it.  Make that first call before any stream capture.
 * - Every call on a device shares the one array.  Calls that overlap on the
 *   GPU (other streams, other host threads) race on it, so serialise them.
 *   The array keeps the last call's tables; nothing in it needs to start at
 *   zero, because each call rewrites what it reads.
 */
qmm_status qmm_q4_gemm_id_noalloc(const void* tiles, int64_t n_expert, int64_t N, int64_t K,
                                  const void* X, int64_t ldx_token, int64_t ldx_slot,
                                  const int32_t* ids, int64_t ld_ids, int64_t n_used, int64_t T,
                                  float* Y, int64_t ldy_token, int64_t ldy_slot,
                                  int32_t* dev_status, cudaStream_t stream);

/* ========================================================================
 * (III) W8A16: int8 weights with block scales, bf16 activations
 *
 * "llama.cpp-xdna -- CPU, iGPU and XDNA1 NPU on AMD Ryzen APUs", sections
 * "The NPU worker" and "Running": in the GGML_XDNA_NPU_W8 mode each
 * 1,024-weight block of a row is int8 with its own scale, and that scale
 * multiplies the block's partial sum.
 *
 * Layout (this library's own; the page gives the block size, not the bytes):
 *   codes   int8 [N][Kp], Kp = K rounded up to 64, row n = output n, zeros in
 *           the padding columns.
 *   scales  fp32 [N][nb], nb = ceil(K / 1024): scale of (row n, block b)
 *           covers columns 1024 b .. min(K, 1024 b + 1024) - 1.
 * ======================================================================== */

/* Bytes of the codes (N * Kp) and of the scales (N * nb * 4).  K <= 65536,
 * N <= 2^31 - 1, else QMM_ERR_UNSUPPORTED. */
qmm_status qmm_pack_w8_size(int64_t N, int64_t K, size_t* code_bytes, size_t* scale_bytes);

/* Quantise fp32 W [N][K] (row stride ldw elements, ldw >= K).  Per (row n,
 * block b), with IEEE fp32 steps (the same rule as qmm_pack_b_int8):
 *   s = fl(amax / 127), amax = max |W[n][k]| over the block;
 *   q = clamp(rint_even(fl(W[n][k] / s)), -127, 127), 0 where s == 0.
 * codes 16-byte aligned with code_bytes >= the size above; scales 4-byte
 * aligned.  W must be finite.  Errors: QMM_ERR_INVALID_ARG for null or
 * misaligned pointers, short buffers, N < 1, K < 1 or ldw < K.
 */
qmm_status qmm_pack_w8(const float* W, int64_t N, int64_t K, int64_t ldw, void* codes, size_t code_bytes,
                       float* scales, size_t scale_bytes, cudaStream_t stream);

/* Workspace of qmm_w8_gemm: 0 for M <= 16 (the decode GEMV), else N * Kp * 2
 * bytes (the codes widened to bf16 for the tensor cores). */
qmm_status qmm_w8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);

/* Y[m][n] = sum_b scales[n][b] * sum_{k in block b} codes[n][k] * X[m][k],
 * with fp32 accumulation.
 *
 * X      bf16 [M][K], row stride ldx elements (ldx >= K, ldx % 8 == 0, base
 *        16-byte aligned).
 * Y      fp32 [M][N], row stride ldy elements (ldy >= N), 4-byte aligned.
 * workspace / ws_bytes  qmm_w8_gemm_workspace_size bytes, 256-byte aligned
 *        (NULL when that size is 0), rewritten by the call.
 * M <= 16 runs the decode GEMV (codes streamed once; M = 1 over many rows
 * streams 32-row items through a shared-memory ring with bounded waits, which
 * report QMM_ERR_TIMEOUT into dev_status); larger M the tensor-core GEMM (the codes widened to bf16, which is exact;
 * each 1,024-k block summed in the tensor cores' fp32 accumulator, then
 * scaled).  Both compute the same function, within
 * max |y - y_exact| <= 2e-4 * sum_k |x| |w|: the products code * x are exact
 * in fp32, so the only error is fp32 summation over at most 1,024 terms per
 * block (1,024 * 2^-23 < 1.3e-4 even if every addition truncates) and over
 * the at most 64 blocks.
 * Errors: QMM_ERR_INVALID_ARG for null or misaligned pointers and bad sizes or
 * strides; QMM_ERR_WORKSPACE for a missing or short workspace;
 * QMM_ERR_UNSUPPORTED for K > 65536.
 */
qmm_status qmm_w8_gemm(const void* codes, const float* scales, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* dev_status,
                       cudaStream_t stream);

/* ========================================================================
 * (IV) More weight formats
 *
 * "NPU engine: full ELFs, no xclbin", section "Q4NX chunks":
 *   - Q4_K weights convert to q4_1 tiles, which the 4-bit kernels above then
 *     run; the only loss is the bf16 rounding of the two per-sub-block
 *     products (scale and min);
 *   - Q8 weights use the same 32 x 256 tile grid with 8-bit codes in one of
 *     two layouts: code (row r, column k) at byte k*32 + r, or at
 *     (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16.
 * ======================================================================== */

/* Repack Q4_K super-blocks into q4_1 tiles (the format of qmm_pack_q4).
 *
 * q4k       N rows of K/256 super-blocks (GGML's k-quant layout, 144 bytes per
 *           256 weights of a row: fp16 d, fp16 dmin, twelve bytes of 6-bit
 *           scale/min codes, 128 bytes of 4-bit codes; w = d*sc*q - dmin*mn).
 *           Row n starts at byte n*row_bytes; row_bytes >= (K/256)*144 and a
 *           multiple of 16, base 16-byte aligned.
 * tiles     out, qmm_pack_q4_size(N, K) bytes, 16-byte aligned.
 * Each 32-weight sub-block keeps its codes and gets scale bf16(d*sc) and min
 * bf16(-(dmin*mn)), rounded to nearest even from the exact fp32 products, so
 * every decoded weight is within 2^-8 (q|d*sc| + |dmin*mn|) of the Q4_K one.
 * Errors: QMM_ERR_INVALID_ARG for null or misaligned pointers, a short row
 * stride or tile buffer, N < 1 or K < 1; QMM_ERR_UNSUPPORTED unless N % 32 == 0
 * and K % 256 == 0.
 */
qmm_status qmm_repack_q4k(const void* q4k, int64_t N, int64_t K, int64_t row_bytes, void* tiles,
                          size_t tile_bytes, cudaStream_t stream);

/* Q8 code layouts (the two of "Q4NX chunks"). */
typedef enum {
  QMM_Q8_LAYOUT_KR = 0,     /* code (r, k) at byte k*32 + r */
  QMM_Q8_LAYOUT_SLAB16 = 1  /* code (r, k) at byte (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16 */
} qmm_q8_layout;

/* Q8 tile bytes of an N x K weight: (N/32) * (K/256) * 8704.  Each tile holds
 * the 8192 code bytes (int8, in the chosen layout) followed by this library's
 * scale bytes, which the pages do not give: one bf16 scale per (row r, block
 * g of 32 columns) at byte 8192 + 2*(32 g + r).  w = code * scale. */
qmm_status qmm_pack_q8_size(int64_t N, int64_t K, size_t* tile_bytes);

/* Quantise fp32 W [N][K] (row stride ldw elements, ldw >= K, W finite) into
 * Q8 tiles.  Per block of 32 consecutive k of one row (IEEE fp32 steps):
 *   s = bf16_rne(amax / 127); q = clamp(rint_even(W / s), -127, 127), 0 where s == 0.
 * Requires N % 32 == 0 and K % 256 == 0 (else QMM_ERR_UNSUPPORTED); tiles
 * 16-byte aligned with tile_bytes >= qmm_pack_q8_size; QMM_ERR_INVALID_ARG for
 * a bad layout or pointer.
 */
qmm_status qmm_pack_q8(const float* W, int64_t N, int64_t K, int64_t ldw, qmm_q8_layout layout, void* tiles,
                       size_t tile_bytes, cudaStream_t stream);

/* Workspace of qmm_q8_gemm: 0 for M <= 16, else N*K*2 bytes of f16 weights,
 * N*ceil(K/1024)*4 bytes of chunk scales, M*K*2 bytes of f16 activation rows
 * and M*4 bytes of row scales, each rounded up to 256. */
qmm_status qmm_q8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes);

/* Y[m][n] = sum_k X[m][k] * w[n][k] over Q8 tiles, fp32 accumulation.
 *
 * tiles  from qmm_pack_q8 (or any Q8 tile set) in the given layout, 16-byte
 *        aligned; N % 32 == 0, K % 256 == 0.
 * X      bf16 [M][K], row stride ldx elements (ldx >= K, ldx % 8 == 0, base
 *        16-byte aligned).
 * Y      fp32 [M][N], row stride ldy elements (ldy >= N), 4-byte aligned.
 * workspace / ws_bytes  qmm_q8_gemm_workspace_size bytes, 256-byte aligned
 *        (NULL when that size is 0), rewritten by the call.
 * M <= 16 runs the decode GEMV, which forms every weight exactly
 * (code * scale in fp32), so only fp32 summation rounds: about
 * (K/256 + 14) * 2^-24 * sum_k |x||w| at worst, within 2e-5 * sum_k |x||w|
 * for K <= 65536.  Larger M decodes the tiles to f16 weights (one rounding,
 * <= 2^-11 relative per weight) and the activation rows to power-of-two
 * scaled f16 (exact, as for qmm_q4_gemm) for the tensor-core GEMM, which sums
 * each 1,024-k chunk in fp32: the worst case is
 * (2^-11 + 1024 * 2^-23 + K/1024 * 2^-24) * sum_k |x||w| < 6.2e-4 * sum_k |x||w|
 * for scales in f16's normal range.  A block with 128 |s| > 65504 gives
 * QMM_ERR_RANGE.
 * Errors: QMM_ERR_INVALID_ARG for null or misaligned pointers, bad sizes,
 * strides or layout; QMM_ERR_WORKSPACE; QMM_ERR_UNSUPPORTED for N % 32 != 0,
 * K % 256 != 0, or K > 65536 when M > 16.  Device status: QMM_ERR_TIMEOUT,
 * QMM_ERR_RANGE (M > 16 only).
 */
qmm_status qmm_q8_gemm(const void* tiles, qmm_q8_layout layout, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* dev_status,
                       cudaStream_t stream);

/* ========================================================================
 * Diagnostics
 * ======================================================================== */

/* Load-only read of `bytes` of device memory (a multiple of 32768, at least
 * 32768; buf 16-byte aligned): the bandwidth a kernel that only streams data
 * reaches, the roofline of the decode GEMVs besides the copy bandwidth ("Zaya
 * 8B Q4NX on the AMD NPU", round 25q: a load-only kernel over a rotating ring
 * of buffers).  mode 0 reads with per-thread 16-byte loads, mode 1 with bulk
 * copies into a shared-memory ring (the two ways the GEMVs read).  The data
 * is folded into one word; `sink` (device uint32) is written only when that
 * word equals a fixed constant, so normally nothing is stored.  dev_status:
 * QMM_ERR_TIMEOUT (mode 1).  QMM_ERR_INVALID_ARG for a bad pointer, size or
 * mode. */
qmm_status qmm_probe_hbm_read(const void* buf, size_t bytes, int mode, uint32_t* sink, int32_t* dev_status,
                              cudaStream_t stream);

/* Self-test of the device error path (no counterpart on the pages).
 *
 * Every pipeline wait of the tensor-core kernels is bounded in time: a wait
 * that gives up raises its thread block's abort flag and writes
 * QMM_ERR_TIMEOUT to dev_status, the block's other waits return at once, and
 * the kernel frees its tensor memory and exits, leaving the context usable.
 * This call runs that path on purpose in a one-block kernel: one wait with
 * limit limit_ns (1 us .. 100 ms) on a barrier nothing arrives on, a second
 * wait (with the kernels' normal limit) that must leave on the abort flag,
 * and a tensor-memory allocation held across the abort and freed.
 * out      device int64 [4]: [0] 1 if the short wait completed (it must not),
 *          [1] 1 if the second wait completed (it must not), [2] ns the short
 *          wait took, [3] ns from the abort to the second wait's return.
 * dev_status gets QMM_ERR_TIMEOUT.  QMM_ERR_INVALID_ARG for a null or
 * misaligned pointer or a limit outside the range.
 */
qmm_status qmm_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_status, int64_t* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
