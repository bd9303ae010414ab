// Exact int8 GEMM on the legacy integer MMA (mma.sync m16n8k32 s8 -> s32).
//
// The small-M route of the int8 half ("int8 inference", "Product kernel
// (Int8Gemm)"): S = sum_k A'B' accumulates exactly in int32, and the zero-point
// correction, bias and output conversion follow in the epilogue.  With M of
// 16 or 32 rows the weight stream dominates, so the kernel reads packed int8
// weights straight from HBM, one 16-byte vector per thread and row.
//
// Inside a 64-column K block, thread t of a quad holds bytes 16t..16t+15 of
// each row it loads.  The MMA's logical k order is a permutation of those
// bytes, and it is the same permutation for A and B, so the sum over the
// block is unchanged.  The row sums of A' (needed when zB' != 0) are taken
// from the same registers with dp4a and reduced across the quad with warp
// shuffles.
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kWarps = 8;     // warps of a CTA split K between them
constexpr int kBM = 32;       // rows per CTA (two m16 tiles)
constexpr int kBN = 32;       // columns per CTA (four n8 tiles)

__global__ void __launch_bounds__(kWarps * 32) int8_gemm_mma_kernel(const Int8GemmArgs a) {
  __shared__ int red[kWarps][32][32];
  __shared__ int rsum[kWarps][kBM];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int K = a.K;
  const int K16 = (K + 15) & ~15;
  const int nkb = (K + 63) >> 6;
  const uint32_t xorv = a.a_u8 ? 0x80808080u : 0u;

  const int8_t* arow[4];
  bool aok[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = m0 + (r >> 1) * 16 + (r & 1) * 8 + g;
    aok[r] = row < a.M;
    arow[r] = a.A + (int64_t)(aok[r] ? row : 0) * a.lda;
  }
  const int8_t* brow[4];
  bool bok[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int col = n0 + 8 * j + g;
    bok[j] = col < a.N;
    brow[j] = a.B + (int64_t)(bok[j] ? col : 0) * a.Kp;
  }

  int acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][j][c] = 0;
  int rs[4] = {0, 0, 0, 0};

  for (int kb = warp; kb < nkb; kb += kWarps) {
    const int k = kb * 64 + t * 16;
    uint4 av[4], bv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (aok[r] && k < K16) {
        av[r] = ldg128(arow[r] + k);
        av[r].x ^= xorv; av[r].y ^= xorv; av[r].z ^= xorv; av[r].w ^= xorv;
        if (k + 16 > K) {            // clear the bytes past K (A' = 0 there)
          uint32_t w[4] = {av[r].x, av[r].y, av[r].z, av[r].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int valid = K - (k + 4 * q);
            if (valid <= 0) w[q] = 0u;
            else if (valid < 4) w[q] &= (1u << (8 * valid)) - 1u;
          }
          av[r] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        av[r] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      bv[j] = bok[j] ? ldg128_stream(brow[j] + k) : make_uint4(0u, 0u, 0u, 0u);
    if (a.need_rowsum) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        rs[r] = __dp4a((int)av[r].x, 0x01010101, rs[r]);
        rs[r] = __dp4a((int)av[r].y, 0x01010101, rs[r]);
        rs[r] = __dp4a((int)av[r].z, 0x01010101, rs[r]);
        rs[r] = __dp4a((int)av[r].w, 0x01010101, rs[r]);
      }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint32_t a0 = u4_get(av[2 * mt], 2 * s), a1 = u4_get(av[2 * mt + 1], 2 * s);
        const uint32_t a2 = u4_get(av[2 * mt], 2 * s + 1), a3 = u4_get(av[2 * mt + 1], 2 * s + 1);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_s8_16832(acc[mt][j], a0, a1, a2, a3, u4_get(bv[j], 2 * s), u4_get(bv[j], 2 * s + 1));
      }
  }

  // cross-warp reduction of the partial sums (exact int32 adds)
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[warp][lane][mt * 16 + j * 4 + c] = acc[mt][j][c];
  if (a.need_rowsum) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      int v = rs[r];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (t == 0) rsum[warp][(r >> 1) * 16 + (r & 1) * 8 + g] = v;
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < 32 * 32; idx += kWarps * 32) {
    const int l = idx >> 5, v = idx & 31;
    int s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w][l][v];
    const int gg = l >> 2, tt = l & 3;
    const int mt = v >> 4, j = (v >> 2) & 3, c = v & 3;
    const int rr = mt * 16 + gg + 8 * (c >> 1);
    const int row = m0 + rr;
    const int col = n0 + 8 * j + 2 * tt + (c & 1);
    if (row >= a.M || col >= a.N) continue;
    int rowsum = 0;
    if (a.need_rowsum)
#pragma unroll
      for (int w = 0; w < kWarps; ++w) rowsum += rsum[w][rr];
    const int32_t Y = zp_correct(s, a.epi.col_sum[col], rowsum, a.epi);
    int8_store(a.epi, row, col, Y);
  }
}

}  // namespace

cudaError_t launch_int8_gemm_mma(const Int8GemmArgs& a, cudaStream_t stream) {
  dim3 grid((unsigned)((a.N + kBN - 1) / kBN), (unsigned)((a.M + kBM - 1) / kBM));
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  int8_gemm_mma_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qmm
