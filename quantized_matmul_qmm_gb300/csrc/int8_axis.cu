// Per-axis zero points for the int8 GEMM: one zero point per activation row
// (zA[m]) and one per weight column (zB[n]) ("The ONNX pack: weights to Q4NX,
// matmuls to our kernels, no VitisAI", section "What works today": the
// asymmetric corrections come per tensor or per axis, laid out like the
// scales, and are exact in integers).
//
//   Y[m,n] = S'[m,n] - zA'[m] colSum'[n] - zB'[n] (rowSum'[m] - K zA'[m])
//
// with the shifted operands and zero points of the per-tensor GEMM (uint8
// values minus 128).  The two correction terms are outer products of a row
// vector and a column vector, which the per-tensor epilogues cannot hold:
// the tensor-core kernel's per-column constants fill its shared memory.  So
// the product S' runs through the exact GEMM unchanged (zero points that
// shift to 0, int32 output, into the workspace), a warp per row forms
// rowSum'[m], and one elementwise pass applies both corrections, the bias and
// the output conversion of the per-tensor path (int8_store).  Integer steps
// run modulo 2^32, exact whenever the final Y fits in int32.
#include <algorithm>

#include "int8_axis.h"

namespace qmm {
namespace {

constexpr int kRowSumWarps = 8;
constexpr int kEpiThreads = 256;

__global__ void __launch_bounds__(kRowSumWarps * 32)
axis_rowsum_kernel(const uint8_t* __restrict__ A, int64_t lda, int M, int K, bool a_u8, int32_t* __restrict__ row_sum) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (int)gridDim.x * kRowSumWarps;
  for (int m = (int)blockIdx.x * kRowSumWarps + ((int)threadIdx.x >> 5); m < M; m += nwarps) {
    const uint8_t* row = A + (int64_t)m * lda;
    uint32_t su = 0;   // sum of the bytes read as uint8
    int32_t ss = 0;    // sum of the bytes read as int8
    for (int c = 16 * lane; c < K; c += 512) {
      // lda is a multiple of 16 and >= K, so the 16 bytes at c stay in the row
      const uint4 v = ldg128(row + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int valid = K - (c + 4 * i);
        const uint32_t mask = valid >= 4 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : (1u << (8 * valid)) - 1u);
        if (a_u8) su = __dp4a(w[i] & mask, 0x01010101u, su);
        else ss = __dp4a((int)(w[i] & mask), 0x01010101, ss);
      }
    }
    int32_t t = a_u8 ? (int32_t)su : ss;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) row_sum[m] = a_u8 ? t - 128 * K : t;
  }
}

// Four consecutive columns per thread (one 16-byte load of S' when the row
// stride allows), rows strided over the grid's y dimension.
__global__ void __launch_bounds__(kEpiThreads)
axis_epilogue_kernel(const int32_t* __restrict__ S, int M, int N, int K, const int32_t* __restrict__ zA, int a_shift,
                     int za_lo, int za_hi, const int32_t* __restrict__ zB, int b_shift, int zb_lo, int zb_hi,
                     const int32_t* __restrict__ row_sum, const Int8Epi e, int32_t* dev_status) {
  const bool vec = (N & 3) == 0;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const int32_t za = zA != nullptr ? zA[m] : 0;
    if ((za < za_lo || za > za_hi) && blockIdx.x == 0 && threadIdx.x == 0) set_status(dev_status, QMM_ERR_INVALID_ARG);
    const uint32_t zap = (uint32_t)(za - a_shift);
    const uint32_t r = (uint32_t)row_sum[m] - (uint32_t)K * zap;
    const int32_t* srow = S + (int64_t)m * N;
    for (int n0 = 4 * ((int)blockIdx.x * kEpiThreads + (int)threadIdx.x); n0 < N;
         n0 += 4 * (int)gridDim.x * kEpiThreads) {
      int32_t sv[4];
      if (vec) {
        const int4 v = *reinterpret_cast<const int4*>(srow + n0);
        sv[0] = v.x;
        sv[1] = v.y;
        sv[2] = v.z;
        sv[3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) sv[i] = n0 + i < N ? srow[n0 + i] : 0;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + i;
        if (n >= N) break;
        const int32_t zb = zB != nullptr ? zB[n] : 0;
        if ((zb < zb_lo || zb > zb_hi) && m == (int)blockIdx.y) set_status(dev_status, QMM_ERR_INVALID_ARG);
        const uint32_t zbp = (uint32_t)(zb - b_shift);
        const uint32_t y = (uint32_t)sv[i] - zap * (uint32_t)e.col_sum[n] - zbp * r;
        int8_store(e, m, n, (int32_t)y);
      }
    }
  }
}

}  // namespace

cudaError_t launch_int8_axis_zp(const Int8AxisArgs& a, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int rgrid = std::max(1, std::min((a.M + kRowSumWarps - 1) / kRowSumWarps, 8 * sms));
  axis_rowsum_kernel<<<rgrid, kRowSumWarps * 32, 0, stream>>>(a.A, a.lda, a.M, a.K, a.a_u8, a.row_sum);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int gx = std::max(1, std::min((a.N + 4 * kEpiThreads - 1) / (4 * kEpiThreads), 16));
  const int gy = std::max(1, std::min(a.M, 1024));
  const int za_lo = a.a_u8 ? 0 : -128, za_hi = a.a_u8 ? 255 : 127;
  const int zb_lo = a.b_u8 ? 0 : -128, zb_hi = a.b_u8 ? 255 : 127;
  axis_epilogue_kernel<<<dim3(gx, gy), kEpiThreads, 0, stream>>>(a.S, a.M, a.N, a.K, a.zA, a.a_u8 ? 128 : 0, za_lo,
                                                                  za_hi, a.zB, a.b_u8 ? 128 : 0, zb_lo, zb_hi,
                                                                  a.row_sum, a.epi, a.dev_status);
  return cudaGetLastError();
}

}  // namespace qmm
