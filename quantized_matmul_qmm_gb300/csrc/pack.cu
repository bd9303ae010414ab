// Weight packers.
//
// packB: "The ONNX pack: weights to Q4NX, matmuls to our kernels, no VitisAI",
// section "The three layers of the pack": each weight column is quantised to
// int8 with scale = amax/127 and the column scales are stored beside the
// packed buffer.  Integer weights are shifted into int8 by the rule of "int8
// inference", section "Product kernel (Int8Gemm)" (uint8 minus 128).  Column
// sums are made here once per weight ("What works today": computed once and
// kept for the session).
//
// pack_q4: 32-row x 256-column tiles ("NPU engine: full ELFs, no xclbin",
// "Q4NX chunks") of q4_1 blocks (w = q*scale + min with bf16 scale/min,
// "Zaya 8B Q4NX on the AMD NPU", round 26).
#include <cuda_bf16.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kPackCols = 32;   // columns per block
constexpr int kPackRows = 8;    // k rows per pass (blockDim.y)
constexpr int kPackChunk = 64;  // k per SMEM transpose chunk

__device__ __forceinline__ float load_b_as_float(const void* B, qmm_dtype t, int64_t idx) {
  if (t == QMM_F32) return reinterpret_cast<const float*>(B)[idx];
  if (t == QMM_S8) return (float)reinterpret_cast<const int8_t*>(B)[idx];
  return (float)reinterpret_cast<const uint8_t*>(B)[idx];
}

__device__ __forceinline__ int load_b_code(const void* B, qmm_dtype t, int64_t idx) {
  if (t == QMM_S8) return (int)reinterpret_cast<const int8_t*>(B)[idx];
  return (int)reinterpret_cast<const uint8_t*>(B)[idx] - 128;
}

// One block packs 32 columns: amax (fp32 only), codes, and the K-major
// transposed rows through shared memory.
__global__ void __launch_bounds__(kPackCols * kPackRows)
pack_b_int8_kernel(const void* __restrict__ B, qmm_dtype b_type, int K, int N, int64_t ldb,
                   int8_t* __restrict__ packed, int64_t Kp, float* __restrict__ col_scale,
                   int32_t* __restrict__ col_sum) {
  __shared__ float red_f[kPackRows][kPackCols];
  __shared__ int red_i[kPackRows][kPackCols];
  __shared__ __align__(16) int8_t tile[kPackCols][kPackChunk];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int n0 = blockIdx.x * kPackCols;
  const int n = n0 + tx;
  const bool is_f32 = (b_type == QMM_F32);

  float scale = 0.0f;
  if (is_f32) {
    float amax = 0.0f;
    if (n < N)
      for (int k = ty; k < K; k += kPackRows)
        amax = fmaxf(amax, fabsf(load_b_as_float(B, b_type, (int64_t)k * ldb + n)));
    red_f[ty][tx] = amax;
    __syncthreads();
    if (ty == 0) {
      for (int r = 1; r < kPackRows; ++r) amax = fmaxf(amax, red_f[r][tx]);
      red_f[0][tx] = __fdiv_rn(amax, 127.0f);
    }
    __syncthreads();
    scale = red_f[0][tx];
    if (ty == 0 && n < N) col_scale[n] = scale;
  }

  int csum = 0;
  for (int kc = 0; kc < Kp; kc += kPackChunk) {
    for (int i = 0; i < kPackChunk / kPackRows; ++i) {
      const int kk = ty + kPackRows * i;
      const int k = kc + kk;
      int q = 0;
      if (k < K && n < N) {
        const int64_t idx = (int64_t)k * ldb + n;
        if (is_f32) {
          if (scale > 0.0f) {
            const float w = load_b_as_float(B, b_type, idx);
            q = __float2int_rn(__fdiv_rn(w, scale));
            q = min(max(q, -127), 127);
          }
        } else {
          q = load_b_code(B, b_type, idx);
        }
      }
      csum += q;
      tile[tx][kk] = (int8_t)q;
    }
    __syncthreads();
    const int tid = ty * kPackCols + tx;
    if (tid < kPackCols * (kPackChunk / 16)) {
      const int row = tid / (kPackChunk / 16), part = tid % (kPackChunk / 16);
      if (n0 + row < N)
        *reinterpret_cast<uint4*>(packed + (int64_t)(n0 + row) * Kp + kc + part * 16) =
            *reinterpret_cast<const uint4*>(&tile[row][part * 16]);
    }
    __syncthreads();
  }
  red_i[ty][tx] = csum;
  __syncthreads();
  if (ty == 0 && n < N) {
    for (int r = 1; r < kPackRows; ++r) csum += red_i[r][tx];
    col_sum[n] = csum;
  }
}

// One thread per (row, 32-column block): min/max, bf16 scale and min, codes.
__global__ void pack_q4_kernel(const float* __restrict__ W, int N, int K, int64_t ldw,
                               uint8_t* __restrict__ tiles) {
  const int nblk = K / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)N * nblk) return;
  const int n = (int)(idx / nblk), kb = (int)(idx % nblk);
  const float* w = W + (int64_t)n * ldw + (int64_t)kb * 32;
  float v[32];
  float mx = -INFINITY, mn = INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = w[j];
    mx = fmaxf(mx, v[j]);
    mn = fminf(mn, v[j]);
  }
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
  const __nv_bfloat16 mb = __float2bfloat16_rn(mn);
  const float s = __bfloat162float(sb), m = __bfloat162float(mb);
  const int tr = n / 32, r = n % 32, tc = kb / 8, b = kb % 8;
  uint8_t* tile = tiles + ((int64_t)tr * (K / 256) + tc) * kTileBytes;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int q = 0;
      if (s > 0.0f) {
        q = __float2int_rn(__fdiv_rn(__fsub_rn(v[8 * t + j], m), s));
        q = min(max(q, 0), 15);
      }
      const int sh = 4 * (j >> 1) + ((j & 1) ? 16 : 0);
      word |= (uint32_t)q << sh;
    }
    *reinterpret_cast<uint32_t*>(tile + r * 128 + 16 * b + 4 * t) = word;
  }
  const uint32_t pair =
      (uint32_t)__bfloat16_as_ushort(sb) | ((uint32_t)__bfloat16_as_ushort(mb) << 16);
  *reinterpret_cast<uint32_t*>(tile + 4096 + 4 * (8 * r + b)) = pair;
}

}  // namespace

cudaError_t launch_pack_b_int8(const void* B, qmm_dtype b_type, int64_t K, int64_t N, int64_t ldb,
                               int8_t* packed, int64_t Kp, float* col_scale, int32_t* col_sum,
                               cudaStream_t stream) {
  dim3 block(kPackCols, kPackRows);
  dim3 grid((unsigned)((N + kPackCols - 1) / kPackCols));
  pack_b_int8_kernel<<<grid, block, 0, stream>>>(B, b_type, (int)K, (int)N, ldb, packed, Kp,
                                                 col_scale, col_sum);
  return cudaGetLastError();
}

cudaError_t launch_pack_q4(const float* W, int64_t N, int64_t K, int64_t ldw, uint8_t* tiles,
                           cudaStream_t stream) {
  const int64_t items = N * (K / 32);
  const int threads = 256;
  pack_q4_kernel<<<(unsigned)((items + threads - 1) / threads), threads, 0, stream>>>(
      W, (int)N, (int)K, ldw, tiles);
  return cudaGetLastError();
}

}  // namespace qmm
