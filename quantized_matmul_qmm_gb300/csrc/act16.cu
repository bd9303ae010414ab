// Activation rows to f16 operands for the tensor-core routes that take f16
// weights: each bf16 row is multiplied by the power of two that puts its
// largest magnitude in [2^14, 2^15), rounded to f16 (exact for every element
// within a factor 2^31 of that magnitude), and the inverse power of two is
// kept for the epilogue.
#include "f16_operands.cuh"
#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kActThreads = 256;
constexpr int kActWarps = kActThreads / 32;

// One warp per row: X bf16 [rows][K] (row stride ldx) -> Xh f16 [rows][K]
// (row stride K) and up[r].  K % 8 == 0.
__global__ void __launch_bounds__(kActThreads)
act_to_f16_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int rows, int K, __half* __restrict__ Xh,
                  float* __restrict__ up) {
  // the GEMM that reads Xh starts its prologue now and waits for this grid
  umma::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int chunks = K / 8;
  const int nw = (int)gridDim.x * kActWarps;
  for (int r = (int)blockIdx.x * kActWarps + ((int)threadIdx.x >> 5); r < rows; r += nw) {
    const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)r * ldx);
    uint32_t am = 0;
#pragma unroll 4
    for (int c = lane; c < chunks; c += 32) {
      const uint4 v = ldg128(src + c);
      am = bf16x2_absmax_bits(am, v.x);
      am = bf16x2_absmax_bits(am, v.y);
      am = bf16x2_absmax_bits(am, v.z);
      am = bf16x2_absmax_bits(am, v.w);
    }
    const uint32_t amax = __reduce_max_sync(0xffffffffu, bf16x2_absmax_fold(am));
    float down, u;
    f16_row_scale(amax, down, u);
    uint4* dst = reinterpret_cast<uint4*>(Xh + (int64_t)r * K);
#pragma unroll 4
    for (int c = lane; c < chunks; c += 32) dst[c] = bf16x8_to_f16x8_scaled(ldg128(src + c), down);
    if (lane == 0) up[r] = u;
  }
}

}  // namespace

size_t act_f16_bytes(int64_t rows, int64_t K) {
  return ((size_t)rows * (size_t)K * 2 + 255) / 256 * 256 + ((size_t)rows * 4 + 255) / 256 * 256;
}

cudaError_t launch_act_to_f16(const __nv_bfloat16* X, int64_t ldx, int rows, int K, void* out,
                              cudaStream_t stream) {
  __half* Xh = static_cast<__half*>(out);
  float* up = reinterpret_cast<float*>(static_cast<char*>(out) + ((size_t)rows * K * 2 + 255) / 256 * 256);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::max(1, std::min((rows + kActWarps - 1) / kActWarps, 4 * sms));
  act_to_f16_kernel<<<grid, kActThreads, 0, stream>>>(X, ldx, rows, K, Xh, up);
  return cudaGetLastError();
}

}  // namespace qmm
