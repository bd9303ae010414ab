// C-ABI entry points: argument validation, kernel choice, launch.
//
// Every check runs on the host before anything is queued.  Kernel choice is
// by shape only: every route computes the same function (bit-exact for the
// int8 half, within the stated bound for the 4-bit half).  A shape with no
// kernel returns QMM_ERR_UNSUPPORTED.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "int8_axis.h"
#include "qmm_internal.h"

using namespace qmm;

namespace {

qmm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QMM_OK;
  if (std::getenv("QMM_LOG")) std::fprintf(stderr, "qmm: CUDA error %s\n", cudaGetErrorString(e));
  return QMM_ERR_CUDA;
}

bool k_bound_ok(int64_t K) { return K * 255 * 128 < (int64_t(1) << 31); }

bool zp_in_domain(int32_t z, qmm_dtype t) {
  if (t == QMM_U8) return z >= 0 && z <= 255;
  if (t == QMM_S8) return z >= -128 && z <= 127;
  return false;
}

}  // namespace

extern "C" {

const char* qmm_status_string(qmm_status s) {
  switch (s) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_INVALID_ARG: return "QMM_ERR_INVALID_ARG";
    case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED";
    case QMM_ERR_OVERFLOW_BOUND: return "QMM_ERR_OVERFLOW_BOUND";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT";
    case QMM_ERR_BAD_EXPERT_ID: return "QMM_ERR_BAD_EXPERT_ID";
    case QMM_ERR_WORKSPACE: return "QMM_ERR_WORKSPACE";
    case QMM_ERR_RANGE: return "QMM_ERR_RANGE";
  }
  return "QMM_ERR_UNKNOWN";
}

int qmm_version(void) { return 200; }

// ---------------------------------------------------------------------------
// int8
// ---------------------------------------------------------------------------

qmm_status qmm_pack_b_int8_size(int64_t K, int64_t N, size_t* packed_bytes) {
  if (packed_bytes == nullptr || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  *packed_bytes = (size_t)(N * padded_k(K));
  return QMM_OK;
}

qmm_status qmm_pack_b_int8(const void* B, qmm_dtype b_type, int64_t K, int64_t N, int64_t ldb,
                           void* packed, size_t packed_bytes, float* col_scale, int32_t* col_sum,
                           cudaStream_t stream) {
  if (B == nullptr || packed == nullptr || col_sum == nullptr) return QMM_ERR_INVALID_ARG;
  if (K < 1 || N < 1 || ldb < N) return QMM_ERR_INVALID_ARG;
  if (b_type != QMM_F32 && b_type != QMM_S8 && b_type != QMM_U8) return QMM_ERR_INVALID_ARG;
  if (b_type == QMM_F32 && col_scale == nullptr) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  if (!aligned(packed, 16) || !aligned(col_sum, 4)) return QMM_ERR_INVALID_ARG;
  if (b_type == QMM_F32 && (!aligned(B, 4) || !aligned(col_scale, 4))) return QMM_ERR_INVALID_ARG;
  if (packed_bytes < (size_t)(N * padded_k(K))) return QMM_ERR_INVALID_ARG;
  if (N > (int64_t)1 << 30) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_pack_b_int8(B, b_type, K, N, ldb, static_cast<int8_t*>(packed),
                                        padded_k(K), col_scale, col_sum, stream));
}

qmm_status qmm_int8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  *ws_bytes = int8_umma_workspace_bytes(M, K, N);
  return QMM_OK;
}

}  // extern "C"

namespace {

// Host checks shared by qmm_int8_gemm and qmm_int8_gemm_group; fills the
// kernel arguments.
qmm_status int8_args(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda, int32_t zA,
                     const void* packedB, const int32_t* col_sum, int64_t N, qmm_dtype b_orig_type, int32_t zB,
                     const qmm_epilogue* ep, void* out, int64_t ldo, Int8GemmArgs& a) {
  if (A == nullptr || packedB == nullptr || col_sum == nullptr || ep == nullptr || out == nullptr)
    return QMM_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (a_type != QMM_U8 && a_type != QMM_S8) return QMM_ERR_INVALID_ARG;
  if (b_orig_type != QMM_U8 && b_orig_type != QMM_S8 && b_orig_type != QMM_F32)
    return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  if (lda < K || lda % 16 != 0 || !aligned(A, 16) || !aligned(packedB, 16)) return QMM_ERR_INVALID_ARG;
  if (!zp_in_domain(zA, a_type)) return QMM_ERR_INVALID_ARG;
  if (b_orig_type == QMM_F32 ? zB != 0 : !zp_in_domain(zB, b_orig_type)) return QMM_ERR_INVALID_ARG;
  const qmm_dtype ot = ep->out_type;
  if (ot != QMM_S32 && ot != QMM_F32 && ot != QMM_S8 && ot != QMM_U8) return QMM_ERR_INVALID_ARG;
  if (ldo < N) return QMM_ERR_INVALID_ARG;
  if (ep->s_x != nullptr && ep->s_x_stride != 0 && ep->s_x_stride != 1) return QMM_ERR_INVALID_ARG;
  if ((ot == QMM_S8 || ot == QMM_U8) && !(ep->s_y > 0.0f)) return QMM_ERR_INVALID_ARG;
  const size_t osz = (ot == QMM_S32 || ot == QMM_F32) ? 4 : 1;
  if (!aligned(out, osz)) return QMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX) return QMM_ERR_UNSUPPORTED;

  a = Int8GemmArgs{};
  a.A = static_cast<const int8_t*>(A);
  a.a_u8 = (a_type == QMM_U8);
  a.M = (int)M;
  a.K = (int)K;
  a.N = (int)N;
  a.lda = lda;
  a.B = static_cast<const int8_t*>(packedB);
  a.Kp = padded_k(K);
  const int32_t zAp = a_type == QMM_U8 ? zA - 128 : zA;
  const int32_t zBp = b_orig_type == QMM_U8 ? zB - 128 : zB;
  a.need_rowsum = (zBp != 0);
  a.epi.out_type = (int)ot;
  a.epi.bias = ep->bias;
  a.epi.s_x = ep->s_x;
  a.epi.s_x_stride = (int)ep->s_x_stride;
  a.epi.s_w = ep->s_w;
  a.epi.s_y = ep->s_y;
  a.epi.zp_y = ep->zp_y;
  a.epi.zAp = (uint32_t)zAp;
  a.epi.zBp = (uint32_t)zBp;
  a.epi.Kz = (uint32_t)((int64_t)K * zAp);
  a.epi.col_sum = col_sum;
  a.epi.out = out;
  a.epi.ldo = ldo;
  return QMM_OK;
}

qmm_status int8_gemm_impl(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda, int32_t zA,
                          const void* packedB, const void* b16, const int32_t* col_sum, int64_t N,
                          qmm_dtype b_orig_type, int32_t zB, const qmm_epilogue* ep, void* out, int64_t ldo,
                          void* workspace, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  Int8GemmArgs a;
  const qmm_status st = int8_args(A, a_type, M, K, lda, zA, packedB, col_sum, N, b_orig_type, zB, ep, out, ldo, a);
  if (st != QMM_OK) return st;
  if (b16 != nullptr && !aligned(b16, 16)) return QMM_ERR_INVALID_ARG;
  if (int8_umma_eligible(M, K, N)) {
    // tensor-core route: needs the caller's workspace (never a silent switch)
    const size_t need = int8_umma_workspace_bytes(M, K, N, b16 != nullptr);
    if (need > 0 && (workspace == nullptr || ws_bytes < need || !aligned(workspace, 256))) return QMM_ERR_WORKSPACE;
    if ((M + 127) / 128 > INT32_MAX || (N + 255) / 256 > 65535) return QMM_ERR_UNSUPPORTED;
    return cuda_status(launch_int8_gemm_umma(a, workspace, dev_status, stream, static_cast<const __half*>(b16)));
  }
  if (int8_small_eligible(M, K, N)) return cuda_status(launch_int8_small(a, dev_status, stream));
  if ((M + 31) / 32 > 65535) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_int8_gemm_mma(a, stream));
}

}  // namespace

extern "C" {

qmm_status qmm_int8_gemm(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda,
                         int32_t zA, const void* packedB, const int32_t* col_sum, int64_t N,
                         qmm_dtype b_orig_type, int32_t zB, const qmm_epilogue* ep, void* out,
                         int64_t ldo, void* workspace, size_t ws_bytes, int32_t* dev_status,
                         cudaStream_t stream) {
  return int8_gemm_impl(A, a_type, M, K, lda, zA, packedB, nullptr, col_sum, N, b_orig_type, zB, ep, out, ldo,
                        workspace, ws_bytes, dev_status, stream);
}

qmm_status qmm_widen_b_int8_size(int64_t K, int64_t N, size_t* b16_bytes) {
  if (b16_bytes == nullptr || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  *b16_bytes = (size_t)(N * padded_k(K) * 2);
  return QMM_OK;
}

qmm_status qmm_widen_b_int8(const void* packedB, int64_t K, int64_t N, void* b16, size_t b16_bytes,
                            int32_t* dev_status, cudaStream_t stream) {
  if (packedB == nullptr || b16 == nullptr || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  if (!aligned(packedB, 16) || !aligned(b16, 16)) return QMM_ERR_INVALID_ARG;
  if (b16_bytes < (size_t)(N * padded_k(K) * 2)) return QMM_ERR_INVALID_ARG;
  if (N > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_widen_b_int8(static_cast<const int8_t*>(packedB), (int)K, (int)N,
                                         static_cast<__half*>(b16), dev_status, stream));
}

qmm_status qmm_int8_gemm_b16_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  *ws_bytes = int8_umma_workspace_bytes(M, K, N, true);
  return QMM_OK;
}

qmm_status qmm_int8_gemm_b16(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda, int32_t zA,
                             const void* packedB, const void* b16, const int32_t* col_sum, int64_t N,
                             qmm_dtype b_orig_type, int32_t zB, const qmm_epilogue* ep, void* out, int64_t ldo,
                             void* workspace, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  if (b16 == nullptr) return QMM_ERR_INVALID_ARG;
  return int8_gemm_impl(A, a_type, M, K, lda, zA, packedB, b16, col_sum, N, b_orig_type, zB, ep, out, ldo,
                        workspace, ws_bytes, dev_status, stream);
}

qmm_status qmm_int8_gemm_group(const qmm_int8_problem* problems, int64_t count, int32_t* dev_status,
                               cudaStream_t stream) {
  if (problems == nullptr || count < 1 || count > INT32_MAX) return QMM_ERR_INVALID_ARG;
  std::vector<Int8GemmArgs> args((size_t)count);
  for (int64_t i = 0; i < count; ++i) {
    const qmm_int8_problem& q = problems[i];
    const qmm_status st = int8_args(q.A, q.a_type, q.M, q.K, q.lda, q.zA, q.packedB, q.col_sum, q.N, q.b_orig_type,
                                    q.zB, &q.ep, q.out, q.ldo, args[(size_t)i]);
    if (st != QMM_OK) return st;
    if (!int8_small_eligible(q.M, q.K, q.N)) return QMM_ERR_UNSUPPORTED;
  }
  return cuda_status(launch_int8_small_group(args.data(), (int)count, dev_status, stream));
}

namespace {
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
}  // namespace

qmm_status qmm_int8_gemm_axis_zp_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  if (M > INT32_MAX || N > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  *ws_bytes = round256((size_t)M * N * 4) + round256((size_t)M * 4) + int8_umma_workspace_bytes(M, K, N);
  return QMM_OK;
}

qmm_status qmm_int8_gemm_axis_zp(const void* A, qmm_dtype a_type, int64_t M, int64_t K, int64_t lda,
                                 const int32_t* zA, const void* packedB, const int32_t* col_sum, int64_t N,
                                 qmm_dtype b_orig_type, const int32_t* zB, const qmm_epilogue* ep, void* out,
                                 int64_t ldo, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 cudaStream_t stream) {
  if (A == nullptr || packedB == nullptr || col_sum == nullptr || ep == nullptr || out == nullptr)
    return QMM_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (a_type != QMM_U8 && a_type != QMM_S8) return QMM_ERR_INVALID_ARG;
  if (b_orig_type != QMM_U8 && b_orig_type != QMM_S8 && b_orig_type != QMM_F32)
    return QMM_ERR_INVALID_ARG;
  if (b_orig_type == QMM_F32 && zB != nullptr) return QMM_ERR_INVALID_ARG;   // symmetric weights
  if (!k_bound_ok(K)) return QMM_ERR_OVERFLOW_BOUND;
  if (lda < K || lda % 16 != 0 || !aligned(A, 16) || !aligned(packedB, 16)) return QMM_ERR_INVALID_ARG;
  if ((zA != nullptr && !aligned(zA, 4)) || (zB != nullptr && !aligned(zB, 4)) || !aligned(col_sum, 4))
    return QMM_ERR_INVALID_ARG;
  const qmm_dtype ot = ep->out_type;
  if (ot != QMM_S32 && ot != QMM_F32 && ot != QMM_S8 && ot != QMM_U8) return QMM_ERR_INVALID_ARG;
  if (ldo < N) return QMM_ERR_INVALID_ARG;
  if (ep->s_x != nullptr && ep->s_x_stride != 0 && ep->s_x_stride != 1) return QMM_ERR_INVALID_ARG;
  if ((ot == QMM_S8 || ot == QMM_U8) && !(ep->s_y > 0.0f)) return QMM_ERR_INVALID_ARG;
  const size_t osz = (ot == QMM_S32 || ot == QMM_F32) ? 4 : 1;
  if (!aligned(out, osz)) return QMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  const size_t s_bytes = round256((size_t)M * N * 4), r_bytes = round256((size_t)M * 4);
  const size_t g_bytes = int8_umma_workspace_bytes(M, K, N);
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < s_bytes + r_bytes + g_bytes)
    return QMM_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  int32_t* S = reinterpret_cast<int32_t*>(ws);
  int32_t* row_sum = reinterpret_cast<int32_t*>(ws + s_bytes);
  // S' = sum_k A'B' exactly: zero points that shift to 0, int32 output, no bias
  const qmm_epilogue eps = {QMM_S32, nullptr, nullptr, 0, nullptr, 1.0f, 0};
  const qmm_status st = qmm_int8_gemm(A, a_type, M, K, lda, a_type == QMM_U8 ? 128 : 0, packedB, col_sum, N,
                                      b_orig_type, b_orig_type == QMM_U8 ? 128 : 0, &eps, S, N,
                                      g_bytes ? ws + s_bytes + r_bytes : nullptr, g_bytes, dev_status, stream);
  if (st != QMM_OK) return st;
  Int8AxisArgs a{};
  a.A = static_cast<const uint8_t*>(A);
  a.lda = lda;
  a.a_u8 = a_type == QMM_U8;
  a.b_u8 = b_orig_type == QMM_U8;
  a.M = (int)M;
  a.K = (int)K;
  a.N = (int)N;
  a.zA = zA;
  a.zB = zB;
  a.S = S;
  a.row_sum = row_sum;
  a.epi.out_type = (int)ot;
  a.epi.bias = ep->bias;
  a.epi.s_x = ep->s_x;
  a.epi.s_x_stride = (int)ep->s_x_stride;
  a.epi.s_w = ep->s_w;
  a.epi.s_y = ep->s_y;
  a.epi.zp_y = ep->zp_y;
  a.epi.col_sum = col_sum;
  a.epi.out = out;
  a.epi.ldo = ldo;
  a.dev_status = dev_status;
  return cuda_status(launch_int8_axis_zp(a, stream));
}

qmm_status qmm_quantize_act_int8_workspace_size(int64_t M, int64_t K, int per_row, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || (per_row != 0 && per_row != 1)) return QMM_ERR_INVALID_ARG;
  *ws_bytes = per_row ? 0 : 256;
  return QMM_OK;
}

qmm_status qmm_quantize_act_int8(const void* X, qmm_dtype x_type, int64_t M, int64_t K, int64_t ldx,
                                 int per_row, void* A, int64_t lda, float* s_x, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream) {
  if (X == nullptr || A == nullptr || s_x == nullptr) return QMM_ERR_INVALID_ARG;
  if (x_type != QMM_F32 && x_type != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || ldx < K || lda < K || lda % 16 != 0 || (per_row != 0 && per_row != 1))
    return QMM_ERR_INVALID_ARG;
  if (!aligned(X, x_type == QMM_F32 ? 4 : 2) || !aligned(A, 16) || !aligned(s_x, 4)) return QMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  if (!per_row && (workspace == nullptr || ws_bytes < 256 || !aligned(workspace, 16))) return QMM_ERR_WORKSPACE;
  return cuda_status(launch_quantize_act(X, x_type == QMM_BF16, (int)M, (int)K, ldx, per_row == 1,
                                         static_cast<int8_t*>(A), lda, s_x, workspace, stream));
}

// ---------------------------------------------------------------------------
// W8A16: int8 weights, an fp32 scale for every 1,024 weights of a row
// ---------------------------------------------------------------------------

qmm_status qmm_pack_w8_size(int64_t N, int64_t K, size_t* code_bytes, size_t* scale_bytes) {
  if (code_bytes == nullptr || scale_bytes == nullptr || N < 1 || K < 1) return QMM_ERR_INVALID_ARG;
  if (N > INT32_MAX || K > kW8MaxK) return QMM_ERR_UNSUPPORTED;
  *code_bytes = (size_t)N * w8_padded_k(K);
  *scale_bytes = (size_t)N * w8_blocks(K) * sizeof(float);
  return QMM_OK;
}

qmm_status qmm_pack_w8(const float* W, int64_t N, int64_t K, int64_t ldw, void* codes, size_t code_bytes,
                       float* scales, size_t scale_bytes, cudaStream_t stream) {
  if (W == nullptr || codes == nullptr || scales == nullptr || N < 1 || K < 1 || ldw < K)
    return QMM_ERR_INVALID_ARG;
  if (N > INT32_MAX || K > kW8MaxK) return QMM_ERR_UNSUPPORTED;
  if (!aligned(W, 4) || !aligned(codes, 16) || !aligned(scales, 4)) return QMM_ERR_INVALID_ARG;
  if (code_bytes < (size_t)N * w8_padded_k(K) || scale_bytes < (size_t)N * w8_blocks(K) * sizeof(float))
    return QMM_ERR_INVALID_ARG;
  return cuda_status(launch_pack_w8(W, (int)N, (int)K, ldw, static_cast<int8_t*>(codes), scales, stream));
}

qmm_status qmm_w8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (K > kW8MaxK) return QMM_ERR_UNSUPPORTED;
  *ws_bytes = M > kW8GemvMaxM ? w8_umma_workspace_bytes(K, N) : 0;
  return QMM_OK;
}

qmm_status qmm_w8_gemm(const void* codes, const float* scales, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* dev_status,
                       cudaStream_t stream) {
  if (codes == nullptr || scales == nullptr || X == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || M < 1 || ldx < K || ldy < N) return QMM_ERR_INVALID_ARG;
  if (ldx % 8 != 0 || !aligned(X, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(Y, 4))
    return QMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > kW8MaxK) return QMM_ERR_UNSUPPORTED;
  const int8_t* c = static_cast<const int8_t*>(codes);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
  if (M <= kW8GemvMaxM)
    return cuda_status(launch_w8_gemv(c, scales, (int)N, (int)K, x, ldx, (int)M, Y, ldy, dev_status, stream));
  const size_t need = w8_umma_workspace_bytes(K, N);
  if (workspace == nullptr || ws_bytes < need || !aligned(workspace, 256)) return QMM_ERR_WORKSPACE;
  if ((N + 255) / 256 > 65535) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_w8_gemm_umma(c, scales, (int)N, (int)K, x, ldx, (int)M, Y, ldy, workspace, dev_status,
                                         stream));
}

// ---------------------------------------------------------------------------
// 4-bit
// ---------------------------------------------------------------------------

qmm_status qmm_pack_q4_size(int64_t N, int64_t K, size_t* tile_bytes) {
  if (tile_bytes == nullptr || N < 1 || K < 1) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  *tile_bytes = (size_t)((N / kTileRows) * (K / kTileCols) * kTileBytes);
  return QMM_OK;
}

qmm_status qmm_pack_q4(const float* W, int64_t N, int64_t K, int64_t ldw, void* tiles,
                       size_t tile_bytes, cudaStream_t stream) {
  if (W == nullptr || tiles == nullptr || N < 1 || K < 1 || ldw < K) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (!aligned(W, 4) || !aligned(tiles, 16)) return QMM_ERR_INVALID_ARG;
  if (tile_bytes < (size_t)((N / kTileRows) * (K / kTileCols) * kTileBytes)) return QMM_ERR_INVALID_ARG;
  if (N * (K / 32) > (int64_t)INT32_MAX * 64) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_pack_q4(W, N, K, ldw, static_cast<uint8_t*>(tiles), stream));
}

qmm_status qmm_q4_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (M > INT32_MAX || K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  *ws_bytes = q4_umma_eligible(M, N, K) ? act_f16_bytes(M, K) : 0;
  return QMM_OK;
}

qmm_status qmm_q4_gemm(const void* tiles, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                       int32_t* dev_status, cudaStream_t stream) {
  if (tiles == nullptr || X == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || M < 1 || ldx < K || ldy < N) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (ldx % 8 != 0 || !aligned(X, 16) || !aligned(tiles, 16) || !aligned(Y, 4))
    return QMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  Q4DenseArgs a{};
  a.tiles = static_cast<const uint8_t*>(tiles);
  a.N = (int)N;
  a.K = (int)K;
  a.M = (int)M;
  a.X = static_cast<const __nv_bfloat16*>(X);
  a.ldx = ldx;
  a.Y = Y;
  a.ldy = ldy;
  if (q4_umma_eligible(M, N, K)) {
    if ((M + 255) / 256 > 65535) return QMM_ERR_UNSUPPORTED;
    if (workspace == nullptr || ws_bytes < act_f16_bytes(M, K) || !aligned(workspace, 256))
      return QMM_ERR_WORKSPACE;
    a.act16 = workspace;
    return cuda_status(launch_q4_gemm_umma(a, dev_status, stream));
  }
  return cuda_status(launch_q4_gemv(a, dev_status, stream));
}

qmm_status qmm_q4_gemv_group(const qmm_q4_gemv_problem* problems, int64_t count, int32_t* dev_status,
                             cudaStream_t stream) {
  if (problems == nullptr || count < 1) return QMM_ERR_INVALID_ARG;
  for (int64_t i = 0; i < count; ++i) {
    const qmm_q4_gemv_problem& q = problems[i];
    if (q.tiles == nullptr || q.x == nullptr || q.y == nullptr || q.N < 1 || q.K < 1) return QMM_ERR_INVALID_ARG;
    if (q.N % kTileRows != 0 || q.K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
    if (q.N > INT32_MAX || q.K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
    if (!aligned(q.tiles, 16) || !aligned(q.x, 16) || !aligned(q.y, 4)) return QMM_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Consecutive problems share a launch while it holds at most
  // kMaxGroupProblems problems and kMaxGroupRows tile rows; a problem too
  // large for the grouped kernel runs the single-problem GEMV.
  std::vector<GemvGroupProblem> batch;
  int rows = 0;
  auto flush = [&]() -> cudaError_t {
    cudaError_t e = cudaSuccess;
    if (!batch.empty()) e = launch_q4_gemv_group(batch.data(), (int)batch.size(), sms, dev_status, stream);
    batch.clear();
    rows = 0;
    return e;
  };
  for (int64_t i = 0; i < count; ++i) {
    const qmm_q4_gemv_problem& q = problems[i];
    const int r = (int)(q.N / kTileRows);
    if (q.K > kMaxGroupK || r > kMaxGroupRows) {
      Q4DenseArgs a{};
      a.tiles = static_cast<const uint8_t*>(q.tiles);
      a.N = (int)q.N;
      a.K = (int)q.K;
      a.M = 1;
      a.X = static_cast<const __nv_bfloat16*>(q.x);
      a.ldx = q.K;
      a.Y = q.y;
      a.ldy = q.N;
      const cudaError_t e = launch_q4_gemv(a, dev_status, stream);
      if (e != cudaSuccess) return cuda_status(e);
      continue;
    }
    if ((int)batch.size() == kMaxGroupProblems || rows + r > kMaxGroupRows) {
      const cudaError_t e = flush();
      if (e != cudaSuccess) return cuda_status(e);
    }
    batch.push_back({static_cast<const uint8_t*>(q.tiles), static_cast<const __nv_bfloat16*>(q.x), q.y,
                     (int)q.N, (int)q.K});
    rows += r;
  }
  return cuda_status(flush());
}

qmm_status qmm_q4_gemm_id_workspace_size(int64_t n_expert, int64_t n_used, int64_t T, int64_t K,
                                         size_t* ws_bytes) {
  if (ws_bytes == nullptr || n_expert < 1 || n_used < 1 || T < 1 || K < 1) return QMM_ERR_INVALID_ARG;
  if (K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (n_expert > kMaxExperts || T * n_used > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  *ws_bytes = q4_moe_workspace_bytes(n_expert, n_used, T, K);
  return QMM_OK;
}

}  // extern "C"

namespace {

// MUL_MAT_ID over one weight set, or over two (tiles2, Y2) that share the
// routing and the packed activations: the gate/up pair.
qmm_status q4_gemm_id_sets(const void* tiles, const void* tiles2, int64_t n_expert, int64_t N, int64_t K,
                           const void* X, int64_t ldx_token, int64_t ldx_slot, const int32_t* ids, int64_t ld_ids,
                           int64_t n_used, int64_t T, float* Y, float* Y2, int64_t ldy_token, int64_t ldy_slot,
                           void* workspace, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  if (tiles == nullptr || X == nullptr || ids == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
  if (n_expert < 1 || N < 1 || K < 1 || n_used < 1 || T < 1 || ld_ids < n_used)
    return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (n_expert > kMaxExperts || n_expert > 65535 || T * n_used > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  if (ldx_token < 0 || ldx_slot < 0 || ldx_token % 8 != 0 || ldx_slot % 8 != 0)
    return QMM_ERR_INVALID_ARG;
  if (ldx_slot == 0 ? ldx_token < K : (ldx_slot < K || ldx_token < ldx_slot * n_used))
    return QMM_ERR_INVALID_ARG;
  if (ldy_token < 0 || ldy_slot < 0) return QMM_ERR_INVALID_ARG;
  if (!(ldy_slot >= N && ldy_token >= ldy_slot * n_used)) return QMM_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(tiles, 16) || !aligned(Y, 4) || !aligned(ids, 4))
    return QMM_ERR_INVALID_ARG;
  // The routing tables are the minimum; the full size adds the packed
  // activations, which the fast path needs.
  const size_t tables = q4_moe_table_bytes(n_expert, n_used, T);
  if (workspace == nullptr || ws_bytes < tables || !aligned(workspace, 256)) return QMM_ERR_WORKSPACE;
  const bool packed = ws_bytes >= q4_moe_workspace_bytes(n_expert, n_used, T, K);
  Q4MoEArgs a{};
  a.tiles = static_cast<const uint8_t*>(tiles);
  a.tiles2 = static_cast<const uint8_t*>(tiles2);
  a.Y2 = Y2;
  a.n_expert = (int)n_expert;
  a.N = (int)N;
  a.K = (int)K;
  a.X = static_cast<const __nv_bfloat16*>(X);
  a.ldx_token = ldx_token;
  a.ldx_slot = ldx_slot;
  a.ids = ids;
  a.ld_ids = ld_ids;
  a.n_used = (int)n_used;
  a.T = (int)T;
  a.Y = Y;
  a.ldy_token = ldy_token;
  a.ldy_slot = ldy_slot;
  char* ws = static_cast<char*>(workspace);
  const size_t off_bytes = ((size_t)(n_expert + 1) * 4 + 255) / 256 * 256;
  const size_t pair_bytes = ((size_t)(T * n_used) * 4 + 255) / 256 * 256;
  a.offsets = reinterpret_cast<int32_t*>(ws);
  a.pairs = reinterpret_cast<int32_t*>(ws + off_bytes);
  a.xup = reinterpret_cast<float*>(ws + off_bytes + pair_bytes);
  a.xperm = packed ? reinterpret_cast<__half*>(ws + tables) : nullptr;
  a.dev_status = dev_status;
  return cuda_status(launch_q4_moe(a, stream));
}

}  // namespace

extern "C" {

qmm_status qmm_q4_gemm_id(const void* tiles, int64_t n_expert, int64_t N, int64_t K,
                          const void* X, int64_t ldx_token, int64_t ldx_slot, const int32_t* ids,
                          int64_t ld_ids, int64_t n_used, int64_t T, float* Y, int64_t ldy_token,
                          int64_t ldy_slot, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, cudaStream_t stream) {
  return q4_gemm_id_sets(tiles, nullptr, n_expert, N, K, X, ldx_token, ldx_slot, ids, ld_ids, n_used, T, Y, nullptr,
                         ldy_token, ldy_slot, workspace, ws_bytes, dev_status, stream);
}

qmm_status qmm_q4_gemm_id_pair(const void* tiles_gate, const void* tiles_up, int64_t n_expert, int64_t N,
                               int64_t K, const void* X, int64_t ldx_token, const int32_t* ids, int64_t ld_ids,
                               int64_t n_used, int64_t T, float* Y_gate, float* Y_up, int64_t ldy_token,
                               int64_t ldy_slot, void* workspace, size_t ws_bytes, int32_t* dev_status,
                               cudaStream_t stream) {
  if (tiles_up == nullptr || Y_up == nullptr) return QMM_ERR_INVALID_ARG;
  if (!aligned(tiles_up, 16) || !aligned(Y_up, 4)) return QMM_ERR_INVALID_ARG;
  return q4_gemm_id_sets(tiles_gate, tiles_up, n_expert, N, K, X, ldx_token, 0, ids, ld_ids, n_used, T, Y_gate, Y_up,
                         ldy_token, ldy_slot, workspace, ws_bytes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// More weight formats: Q4_K repack, Q8 tiles
// ---------------------------------------------------------------------------

qmm_status qmm_repack_q4k(const void* q4k, int64_t N, int64_t K, int64_t row_bytes, void* tiles,
                          size_t tile_bytes, cudaStream_t stream) {
  if (q4k == nullptr || tiles == nullptr || N < 1 || K < 1) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  if (row_bytes < (K / kTileCols) * 144 || row_bytes % 16 != 0) return QMM_ERR_INVALID_ARG;
  if (!aligned(q4k, 16) || !aligned(tiles, 16)) return QMM_ERR_INVALID_ARG;
  if (tile_bytes < (size_t)((N / kTileRows) * (K / kTileCols) * kTileBytes)) return QMM_ERR_INVALID_ARG;
  if ((N * (K / kTileCols) + 255) / 256 > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  return cuda_status(launch_repack_q4k(static_cast<const uint8_t*>(q4k), row_bytes, (int)N, (int)K,
                                       static_cast<uint8_t*>(tiles), stream));
}

qmm_status qmm_pack_q8_size(int64_t N, int64_t K, size_t* tile_bytes) {
  if (tile_bytes == nullptr || N < 1 || K < 1) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  *tile_bytes = (size_t)((N / kTileRows) * (K / kTileCols)) * kQ8TileBytes;
  return QMM_OK;
}

qmm_status qmm_pack_q8(const float* W, int64_t N, int64_t K, int64_t ldw, qmm_q8_layout layout, void* tiles,
                       size_t tile_bytes, cudaStream_t stream) {
  if (W == nullptr || tiles == nullptr || N < 1 || K < 1 || ldw < K) return QMM_ERR_INVALID_ARG;
  if (layout != QMM_Q8_LAYOUT_KR && layout != QMM_Q8_LAYOUT_SLAB16) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX || (N / kTileRows) * (K / kTileCols) > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  if (!aligned(W, 4) || !aligned(tiles, 16)) return QMM_ERR_INVALID_ARG;
  if (tile_bytes < (size_t)((N / kTileRows) * (K / kTileCols)) * kQ8TileBytes) return QMM_ERR_INVALID_ARG;
  return cuda_status(launch_pack_q8(W, ldw, (int)N, (int)K, (int)layout, static_cast<uint8_t*>(tiles), stream));
}

qmm_status qmm_q8_gemm_workspace_size(int64_t M, int64_t K, int64_t N, size_t* ws_bytes) {
  if (ws_bytes == nullptr || M < 1 || K < 1 || N < 1) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (M > kQ8GemvMaxM && K > kQ8MaxK) return QMM_ERR_UNSUPPORTED;
  *ws_bytes = M <= kQ8GemvMaxM ? 0 : q8_gemm_workspace_bytes(M, N, K);
  return QMM_OK;
}

qmm_status qmm_q8_gemm(const void* tiles, qmm_q8_layout layout, int64_t N, int64_t K, const void* X, int64_t M,
                       int64_t ldx, float* Y, int64_t ldy, void* workspace, size_t ws_bytes, int32_t* dev_status,
                       cudaStream_t stream) {
  if (tiles == nullptr || X == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || M < 1 || ldx < K || ldy < N) return QMM_ERR_INVALID_ARG;
  if (layout != QMM_Q8_LAYOUT_KR && layout != QMM_Q8_LAYOUT_SLAB16) return QMM_ERR_INVALID_ARG;
  if (ldx % 8 != 0 || !aligned(X, 16) || !aligned(tiles, 16) || !aligned(Y, 4)) return QMM_ERR_INVALID_ARG;
  if (N % kTileRows != 0 || K % kTileCols != 0) return QMM_ERR_UNSUPPORTED;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QMM_ERR_UNSUPPORTED;
  if (M > kQ8GemvMaxM) {
    if (K > kQ8MaxK || (N + 255) / 256 > 65535 || (N / kTileRows) * (K / kTileCols) > INT32_MAX)
      return QMM_ERR_UNSUPPORTED;
    if (workspace == nullptr || ws_bytes < q8_gemm_workspace_bytes(M, N, K) || !aligned(workspace, 256))
      return QMM_ERR_WORKSPACE;
  }
  return cuda_status(launch_q8_gemm(static_cast<const uint8_t*>(tiles), (int)layout, (int)N, (int)K,
                                    static_cast<const __nv_bfloat16*>(X), ldx, (int)M, Y, ldy, workspace, dev_status,
                                    stream));
}

// ---------------------------------------------------------------------------
// Diagnostics
// ---------------------------------------------------------------------------

qmm_status qmm_probe_hbm_read(const void* buf, size_t bytes, int mode, uint32_t* sink, int32_t* dev_status,
                              cudaStream_t stream) {
  if (buf == nullptr || sink == nullptr || !aligned(buf, 16) || !aligned(sink, 4)) return QMM_ERR_INVALID_ARG;
  if (mode != 0 && mode != 1) return QMM_ERR_INVALID_ARG;
  if (bytes < 32768 || bytes % 32768 != 0) return QMM_ERR_INVALID_ARG;
  return cuda_status(launch_probe_hbm_read(buf, bytes, mode, sink, dev_status, stream));
}

qmm_status qmm_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_status, int64_t* out, cudaStream_t stream) {
  if (dev_status == nullptr || out == nullptr || !aligned(out, 8)) return QMM_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 100000000ull) return QMM_ERR_INVALID_ARG;
  return cuda_status(launch_wait_timeout_selftest(limit_ns, dev_status, out, stream));
}

}  // extern "C"
