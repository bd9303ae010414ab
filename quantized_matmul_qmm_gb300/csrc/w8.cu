// W8A16: int8 weights with a scale for every 1,024 weights of a row, bf16
// activations ("llama.cpp-xdna -- CPU, iGPU and XDNA1 NPU on AMD Ryzen
// APUs", sections "The NPU worker" and "Running": in the GGML_XDNA_NPU_W8
// mode each 1,024-weight block of a row is int8 with its own scale, and the
// scale multiplies that block's partial sum).
//
// Pack: per (row n, block b of 1,024 k), packB's rule: s = fl(amax / 127),
// q = clamp(rint_even(fl(w / s)), -127, 127), 0 where s == 0.  Codes are
// [N][Kp] (Kp = K rounded up to 64, zero padding), scales [N][ceil(K/1024)].
//
// Decode GEMV (M <= 16): a warp streams 32/G rows at once with G lanes per
// row, G sized so that every lane has about eight 16-byte groups of its row
// (a K = 1024 row is 1 KB: four rows per warp, 4 KB in flight per warp).  Each
// lane converts its codes exactly with a byte permute and one add (the
// int-to-float unit runs at a quarter of the fma rate) and multiplies them
// with x read through the read-only cache, even and odd columns as the two
// lanes of packed f32x2 fmas.  Sixteen codes never straddle a 1,024 block, so
// each group's partial sum is scaled by its own block's scale.
#include <cuda_bf16.h>

#include <algorithm>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kW8Block = 1024;
constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads)
pack_w8_kernel(const float* __restrict__ W, int64_t ldw, int K, int Kp, int8_t* __restrict__ codes,
               float* __restrict__ scales, int nb) {
  __shared__ float red[kPackThreads / 32];
  const int n = blockIdx.x;
  const float* row = W + (int64_t)n * ldw;
  int8_t* out = codes + (int64_t)n * Kp;
  for (int b = 0; b < nb; ++b) {
    const int k0 = b * kW8Block, k1 = min(K, k0 + kW8Block);
    float a = 0.f;
    for (int k = k0 + (int)threadIdx.x; k < k1; k += kPackThreads) a = fmaxf(a, fabsf(row[k]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kPackThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) scales[(int64_t)n * nb + b] = s;
    for (int k = k0 + (int)threadIdx.x; k < k1; k += kPackThreads) {
      int q = 0;
      if (s > 0.f) q = min(max(__float2int_rn(__fdiv_rn(row[k], s)), -127), 127);
      out[k] = (int8_t)q;
    }
  }
  for (int k = K + (int)threadIdx.x; k < Kp; k += kPackThreads) out[k] = 0;
}

constexpr int kGvWarps = 8;
constexpr int kGvSteps = 8;   // 16-byte code groups in flight per lane

// 16 int8 codes as fp32 (exact), without the int-to-float unit.
__device__ __forceinline__ void codes16_to_f32(const uint4 v, float (&c)[16]) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[4 * i + j] = s8_byte_to_f32(w[i], j);
}

// A warp works on 32 / G rows at once, G lanes per row (G a power of two
// chosen so that a lane has about kGvSteps groups of its row): each load
// instruction of the warp reads G consecutive 16-byte groups of every one of
// its rows, and kGvSteps such loads are in flight before any is used.
template <int kM>
__global__ void __launch_bounds__(kGvWarps * 32)
w8_gemv_kernel(const int8_t* __restrict__ codes, const float* __restrict__ scales, int N, int K, int Kp, int nb,
               const __nv_bfloat16* __restrict__ X, int64_t ldx, float* __restrict__ Y, int64_t ldy, int M, int G) {
  const int lane = threadIdx.x & 31;
  const int R = 32 / G, sub = lane / G, sl = lane % G;
  const int warp_g = (int)blockIdx.x * kGvWarps + ((int)threadIdx.x >> 5);
  const int nwarps = (int)gridDim.x * kGvWarps;
  const int ngroups = Kp / 16;                       // 16-code groups of a row
  for (int n0 = warp_g * R; n0 < N; n0 += nwarps * R) {
    const int n = n0 + sub;
    const bool live = n < N;
    const uint4* row = reinterpret_cast<const uint4*>(codes + (int64_t)(live ? n : 0) * Kp);
    const float* srow = scales + (int64_t)(live ? n : 0) * nb;
    float acc[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) acc[m] = 0.f;
    for (int g0 = 0; g0 < ngroups; g0 += G * kGvSteps) {
      uint4 v[kGvSteps];
#pragma unroll
      for (int u = 0; u < kGvSteps; ++u) {
        const int g = g0 + G * u + sl;
        v[u] = (live && g < ngroups) ? ldg128_stream(row + g) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kGvSteps; ++u) {
        const int g = g0 + G * u + sl;
        if (!live || g >= ngroups) continue;
        const int k0 = 16 * g;
        if (k0 >= K) continue;   // padding codes are zero; x past K is not read
        float c[16];
        codes16_to_f32(v[u], c);
        const float s = __ldg(srow + k0 / kW8Block);
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          if (m >= M) break;
          const __nv_bfloat16* xr = X + (int64_t)m * ldx + k0;
          float part = 0.f;
          if (k0 + 16 <= K) {
            const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(xr));
            const uint4 x1 = __ldg(reinterpret_cast<const uint4*>(xr) + 1);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            // even and odd columns as the two lanes of packed f32x2 fmas
            uint64_t pp = f2_mul(f2_pack(c[0], c[1]), f2_pack(bf16lo_to_f32(xw[0]), bf16hi_to_f32(xw[0])));
#pragma unroll
            for (int i = 1; i < 8; ++i)
              pp = f2_fma(f2_pack(c[2 * i], c[2 * i + 1]), f2_pack(bf16lo_to_f32(xw[i]), bf16hi_to_f32(xw[i])), pp);
            float pe, po;
            f2_unpack(pp, pe, po);
            part = pe + po;
          } else {
            for (int i = 0; k0 + i < K; ++i) part = fmaf(c[i], __bfloat162float(xr[i]), part);
          }
          acc[m] = fmaf(part, s, acc[m]);
        }
      }
    }
    // sum over the G lanes of each row (G is a power of two: the xor partners
    // stay inside the row's lane group)
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      if (m >= M) break;
      float a = acc[m];
      for (int o = G >> 1; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (sl == 0 && live) Y[(int64_t)m * ldy + n] = a;
    }
  }
}

}  // namespace

int64_t w8_padded_k(int64_t K) { return (K + 63) / 64 * 64; }
int64_t w8_blocks(int64_t K) { return (K + kW8Block - 1) / kW8Block; }

cudaError_t launch_pack_w8(const float* W, int N, int K, int64_t ldw, int8_t* codes, float* scales,
                           cudaStream_t stream) {
  pack_w8_kernel<<<N, kPackThreads, 0, stream>>>(W, ldw, K, (int)w8_padded_k(K), codes, scales, (int)w8_blocks(K));
  return cudaGetLastError();
}

cudaError_t launch_w8_gemv(const int8_t* codes, const float* scales, int N, int K, const __nv_bfloat16* X,
                           int64_t ldx, int M, float* Y, int64_t ldy, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int Kp = (int)w8_padded_k(K), nb = (int)w8_blocks(K);
  // lanes per row: about kGvSteps groups each, at least 4 lanes, at most 32
  int G = 32;
  while (G > 4 && G * kGvSteps > Kp / 16) G >>= 1;
  const int R = 32 / G;
  const int rows_per_block = kGvWarps * R;
  const int grid = std::max(1, std::min((N + rows_per_block - 1) / rows_per_block, 8 * sms));
  if (M <= 1)
    w8_gemv_kernel<1><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  else if (M <= 4)
    w8_gemv_kernel<4><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  else
    w8_gemv_kernel<16><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  return cudaGetLastError();
}

}  // namespace qmm
