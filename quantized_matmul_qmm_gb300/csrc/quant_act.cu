// Symmetric int8 quantisation of activations for the int8 GEMM ("int8
// inference", "Product kernel (Int8Gemm)": activations per-tensor symmetric
// with scale amax/127; "The ONNX pack: weights to Q4NX, matmuls to our
// kernels, no VitisAI", "What works today": the float epilogue's per-row
// activation scale s_x[m]).  The rule is packB's, applied to rows or to the
// whole tensor:
//     s = fl(amax / 127);  q = clamp(rint_even(fl(x / s)), -127, 127), 0 where s == 0.
//
// Per row: one block per row, two passes over the row (its max, then the
// codes; the second pass hits L1/L2).  Per tensor: a grid of row-block maxima
// folded into one word with atomicMax on the fp32 bits (non-negative floats
// order like their bit patterns), then the quantising grid as that grid's
// programmatic dependent.
#include <cuda_bf16.h>

#include <algorithm>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kQThreads = 256;

template <bool kBf16>
__device__ __forceinline__ float ld_x(const void* X, int64_t i) {
  if constexpr (kBf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(X)[i]);
  return reinterpret_cast<const float*>(X)[i];
}

// Max over the block of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();   // red is reused by the next call
  return m;
}

template <bool kBf16>
__device__ __forceinline__ float row_absmax(const void* X, int64_t xrow, int K) {
  float a = 0.f;
  for (int k = threadIdx.x; k < K; k += kQThreads) a = fmaxf(a, fabsf(ld_x<kBf16>(X, xrow + k)));
  return a;
}

// Codes of one row, four per thread per step, stored as 32-bit words (the row
// base is 16-byte aligned); bytes at k >= K are not touched.
template <bool kBf16>
__device__ __forceinline__ void quant_row(const void* X, int64_t xrow, int K, float s, int8_t* arow) {
  for (int k = 4 * (int)threadIdx.x; k < K; k += 4 * kQThreads) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (k + i < K) {
        int q = 0;
        if (s > 0.f) q = min(max(__float2int_rn(__fdiv_rn(ld_x<kBf16>(X, xrow + k + i), s)), -127), 127);
        w |= ((uint32_t)q & 0xFFu) << (8 * i);
      }
    }
    if (k + 4 <= K) {
      *reinterpret_cast<uint32_t*>(arow + k) = w;
    } else {
      for (int i = 0; k + i < K; ++i) arow[k + i] = (int8_t)(w >> (8 * i));
    }
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kQThreads)
quant_rows_kernel(const void* __restrict__ X, int64_t ldx, int K, int8_t* __restrict__ A, int64_t lda,
                  float* __restrict__ s_x) {
  __shared__ float red[kQThreads / 32];
  const int m = blockIdx.x;
  const int64_t xrow = (int64_t)m * ldx;
  const float s = __fdiv_rn(block_max(row_absmax<kBf16>(X, xrow, K), red), 127.0f);
  if (threadIdx.x == 0) s_x[m] = s;
  quant_row<kBf16>(X, xrow, K, s, A + (int64_t)m * lda);
}

template <bool kBf16>
__global__ void __launch_bounds__(kQThreads)
tensor_absmax_kernel(const void* __restrict__ X, int64_t ldx, int M, int K, uint32_t* __restrict__ amax_bits) {
  __shared__ float red[kQThreads / 32];
  umma::pdl_launch_dependents();   // the quantising grid waits for this one
  float a = 0.f;
  for (int m = blockIdx.x; m < M; m += gridDim.x) a = fmaxf(a, row_absmax<kBf16>(X, (int64_t)m * ldx, K));
  a = block_max(a, red);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(a));
}

template <bool kBf16>
__global__ void __launch_bounds__(kQThreads)
quant_tensor_kernel(const void* __restrict__ X, int64_t ldx, int M, int K, int8_t* __restrict__ A, int64_t lda,
                    const uint32_t* __restrict__ amax_bits, float* __restrict__ s_x) {
  umma::pdl_wait();   // the tensor's max
  const float s = __fdiv_rn(__uint_as_float(*amax_bits), 127.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) s_x[0] = s;
  for (int m = blockIdx.x; m < M; m += gridDim.x) quant_row<kBf16>(X, (int64_t)m * ldx, K, s, A + (int64_t)m * lda);
}

template <bool kBf16>
cudaError_t launch_typed(const void* X, int M, int K, int64_t ldx, bool per_row, int8_t* A, int64_t lda,
                         float* s_x, uint32_t* ws, cudaStream_t stream) {
  if (per_row) {
    quant_rows_kernel<kBf16><<<M, kQThreads, 0, stream>>>(X, ldx, K, A, lda, s_x);
    return cudaGetLastError();
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(M, 8 * sms);
  cudaError_t err = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);
  if (err != cudaSuccess) return err;
  tensor_absmax_kernel<kBf16><<<grid, kQThreads, 0, stream>>>(X, ldx, M, K, ws);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_pdl(quant_tensor_kernel<kBf16>, dim3(grid), dim3(kQThreads), 0, stream, X, ldx, M, K, A, lda,
                    (const uint32_t*)ws, s_x);
}

}  // namespace

cudaError_t launch_quantize_act(const void* X, bool x_bf16, int M, int K, int64_t ldx, bool per_row, int8_t* A,
                                int64_t lda, float* s_x, void* workspace, cudaStream_t stream) {
  uint32_t* ws = static_cast<uint32_t*>(workspace);
  return x_bf16 ? launch_typed<true>(X, M, K, ldx, per_row, A, lda, s_x, ws, stream)
                : launch_typed<false>(X, M, K, ldx, per_row, A, lda, s_x, ws, stream);
}

}  // namespace qmm
