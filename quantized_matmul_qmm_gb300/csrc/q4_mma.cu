// 4-bit decode GEMV for 2 <= M <= 16 tokens.
//
// The weights are 32x256 q4_1 tiles ("NPU engine: full ELFs, no xclbin", "Q4NX
// chunks"; w = q*scale + min, "Zaya 8B Q4NX on the AMD NPU", round 26).  At
// decode sizes the work is bound by the weight stream, so each warp streams
// whole tiles with 16-byte loads and never expands them in memory.
//
// The factored form keeps the per-weight work to one logic op per two codes.
// For one block (32 columns of one row):
//     sum_k x_k (q_k s + m) = s * sum_k (128 + q_k) x_k + (m - 128 s) * sum_k x_k
// A code ORed into the mantissa of bf16 128.0 is exactly 128 + q, so a single
// lop3 turns two codes into a bf16x2 MMA operand.  The tensor core
// (mma.sync m16n8k16, fp32 accumulate) forms sum (128+q) x.  The block scale
// and min are applied to the fp32 result, once per block.
//
// MMA fragment mapping: within block b, thread t of a quad owns code word t
// of the block (columns 32b + 8t .. 32b + 8t + 7) and the matching 16 bytes
// of x.  The logical k order inside the MMA is a permutation of these, the
// same for A and B.
#include "qmm_internal.h"

namespace qmm {
namespace {

// ---------------------------------------------------------------------------
// Decode GEMV (dense, M <= 16).  Each warp owns a 16-row slab of a tile row
// and walks its K range with the code words and (scale, min) pairs prefetched
// kPF tiles ahead in registers.  One quad thread loads the pairs of two
// blocks, and the quad shares them by shuffles.  The block sums of x are
// computed once per CTA into shared memory.  When N is small, S warps split
// the K range of a slab, and their partial sums are added in a fixed order
// through shared memory, so the result is deterministic.
// ---------------------------------------------------------------------------
constexpr int kGemvWarps = 8;
constexpr int kPF = 3;

struct Q4GemvParams {
  const uint8_t* tiles;
  int N, K, M;
  const __nv_bfloat16* X;
  int64_t ldx;
  float* Y;
  int64_t ldy;
  int S;            // warps per slab (K split)
};

struct SlabTile {
  uint32_t c[2][8]; // word t of blocks 0..7 of rows R0, R1
  uint2 p[2];       // (scale, min) of blocks 2t, 2t+1 of rows R0, R1
};

__device__ __forceinline__ void slab_load(SlabTile& d, const uint8_t* tile, int r0, int t, bool valid) {
  if (!valid) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint8_t* rowp = tile + (r0 + 8 * h) * 128 + 4 * t;
#pragma unroll
    for (int b = 0; b < 8; ++b) d.c[h][b] = ldg32(rowp + 16 * b);
    d.p[h] = *reinterpret_cast<const uint2*>(tile + 4096 + (r0 + 8 * h) * 32 + 8 * t);
  }
}

// One block of 32 columns for the two rows of this thread: MMA on the biased
// codes, then the block's scale and min.  kOneCol: only column 0 is real.
template <int NG, bool kOneCol>
__device__ __forceinline__ void gemv_block(const SlabTile& cur, int b, int lane, int t, int blk_x, const float* xs,
                                           const __nv_bfloat16* const (&xrow)[NG], float (&y)[NG][4]) {
  const int src = (lane & ~3) | (b >> 1);
  const uint32_t pA = __shfl_sync(0xffffffffu, (b & 1) ? cur.p[0].y : cur.p[0].x, src);
  const uint32_t pB = __shfl_sync(0xffffffffu, (b & 1) ? cur.p[1].y : cur.p[1].x, src);
  const float sA = bf16lo_to_f32(pA), sB = bf16lo_to_f32(pB);
  const float mA = fmaf(-128.0f, sA, bf16hi_to_f32(pA));
  const float mB = fmaf(-128.0f, sB, bf16hi_to_f32(pB));
  const uint32_t wA = cur.c[0][b];
  const uint32_t wB = cur.c[1][b];
  const uint32_t a00 = q4_pair_biased(wA, 0), a01 = q4_pair_biased(wB, 0);
  const uint32_t a02 = q4_pair_biased(wA, 1), a03 = q4_pair_biased(wB, 1);
  const uint32_t a10 = q4_pair_biased(wA, 2), a11 = q4_pair_biased(wB, 2);
  const uint32_t a12 = q4_pair_biased(wA, 3), a13 = q4_pair_biased(wB, 3);
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    const uint4 xv = xrow[ng] ? ldg128(xrow[ng] + blk_x + 8 * t) : make_uint4(0u, 0u, 0u, 0u);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16_16816(c, a00, a01, a02, a03, xv.x, xv.y);
    mma_bf16_16816(c, a10, a11, a12, a13, xv.z, xv.w);
    if (kOneCol) {
      const float x0 = xs[0];
      y[ng][0] = fmaf(sA, c[0], fmaf(mA, x0, y[ng][0]));
      y[ng][2] = fmaf(sB, c[2], fmaf(mB, x0, y[ng][2]));
    } else {
      const float2 xsv = *reinterpret_cast<const float2*>(xs + 8 * ng + 2 * t);
      y[ng][0] = fmaf(sA, c[0], fmaf(mA, xsv.x, y[ng][0]));
      y[ng][1] = fmaf(sA, c[1], fmaf(mA, xsv.y, y[ng][1]));
      y[ng][2] = fmaf(sB, c[2], fmaf(mB, xsv.x, y[ng][2]));
      y[ng][3] = fmaf(sB, c[3], fmaf(mB, xsv.y, y[ng][3]));
    }
  }
}

template <int NG>
__device__ __forceinline__ void gemv_xs_prologue(const Q4GemvParams& p, float* xs, int nblk) {
  for (int idx = threadIdx.x; idx < nblk * 8 * NG; idx += blockDim.x) {
    const int blk = idx / (8 * NG), col = idx % (8 * NG);
    float sum = 0.f;
    if (col < p.M) {
      const uint4* xp = reinterpret_cast<const uint4*>(p.X + (int64_t)col * p.ldx + blk * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 w = xp[v];
        sum += bf16lo_to_f32(w.x) + bf16hi_to_f32(w.x) + bf16lo_to_f32(w.y) + bf16hi_to_f32(w.y) +
               bf16lo_to_f32(w.z) + bf16hi_to_f32(w.z) + bf16lo_to_f32(w.w) + bf16hi_to_f32(w.w);
      }
    }
    xs[idx] = sum;
  }
}

template <int NG, bool kOneCol>
__device__ __forceinline__ void gemv_store(const Q4GemvParams& p, const float (&y)[NG][4], int nrow0, int g, int t) {
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int m = 8 * ng + 2 * t + (c & 1);
      const int n = nrow0 + g + 8 * (c >> 1);
      if (m < p.M && (!kOneCol || (c & 1) == 0)) p.Y[(int64_t)m * p.ldy + n] = y[ng][c];
    }
}

// K split across S warps of a CTA (small N).  Partial sums are added in a
// fixed order through shared memory.
template <int NG>
__global__ void __launch_bounds__(kGemvWarps * 32) q4_gemv_kernel(const Q4GemvParams p) {
  extern __shared__ float gsm[];
  const int nblk = p.K / 32;
  float* xs = gsm;                                   // [nblk][8*NG]
  float* red = gsm + nblk * 8 * NG;                  // [warps][32][4*NG]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int TC = p.K / 256;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // x and y may belong to the previous grid
  gemv_xs_prologue<NG>(p, xs, nblk);
  __syncthreads();

  const int slabs_per_cta = kGemvWarps / p.S;
  const int slab = blockIdx.x * slabs_per_cta + warp / p.S;
  const int ks = warp % p.S;
  const int nrow0 = slab * 16;
  float y[NG][4];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int c = 0; c < 4; ++c) y[ng][c] = 0.f;

  if (nrow0 < p.N) {
    const int tr = nrow0 / 32, r0 = (nrow0 & 31) + g;
    const uint8_t* rowtiles = p.tiles + (int64_t)tr * TC * kTileBytes;
    const __nv_bfloat16* xrow[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) xrow[ng] = (8 * ng + g < p.M) ? p.X + (int64_t)(8 * ng + g) * p.ldx : nullptr;
    SlabTile ring[kPF];
#pragma unroll
    for (int i = 0; i < kPF; ++i) {
      const int tc = ks + i * p.S;
      slab_load(ring[i], rowtiles + (int64_t)tc * kTileBytes, r0, t, tc < TC);
    }
    for (int it0 = 0; ks + it0 * p.S < TC; it0 += kPF) {
#pragma unroll
      for (int i = 0; i < kPF; ++i) {
        const int tc = ks + (it0 + i) * p.S;
        if (tc < TC) {
#pragma unroll
          for (int b = 0; b < 8; ++b)
            gemv_block<NG, false>(ring[i], b, lane, t, tc * 256 + b * 32, xs + (tc * 8 + b) * 8 * NG, xrow, y);
          const int tn = tc + kPF * p.S;
          slab_load(ring[i], rowtiles + (int64_t)tn * kTileBytes, r0, t, tn < TC);
        }
      }
    }
  }
  if (p.S > 1) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[(warp * 32 + lane) * 4 * NG + ng * 4 + c] = y[ng][c];
    __syncthreads();
    if (ks != 0) return;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float s = 0.f;
        for (int w = 0; w < p.S; ++w) s += red[((warp + w) * 32 + lane) * 4 * NG + ng * 4 + c];
        y[ng][c] = s;
      }
  }
  if (nrow0 >= p.N) return;
  gemv_store<NG, false>(p, y, nrow0, g, t);
}

}  // namespace

template <typename Kern>
cudaError_t launch_gemv_kernel(Kern kern, unsigned grid, size_t smem, const Q4GemvParams& p, cudaStream_t stream) {
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3(grid), dim3(kGemvWarps * 32), smem, stream, p);
}

cudaError_t launch_q4_gemv(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (a.M == 1) return launch_q4_gemv1(a, sms, dev_status, stream);
  Q4GemvParams p{};
  p.tiles = a.tiles;
  p.N = a.N;
  p.K = a.K;
  p.M = a.M;
  p.X = a.X;
  p.ldx = a.ldx;
  p.Y = a.Y;
  p.ldy = a.ldy;
  const int TC = a.K / 256;
  const int slabs = a.N / 16;
  const int NG = a.M <= 8 ? 1 : 2;
  const size_t xs_bytes = (size_t)(a.K / 32) * 8 * NG * sizeof(float);
  // split K across the warps of a CTA until the grid fills the GPU
  int S = 1;
  while (S < kGemvWarps && S < TC && (slabs * S) / kGemvWarps < 2 * sms) S *= 2;
  p.S = S;
  const int slabs_per_cta = kGemvWarps / S;
  const unsigned grid = (unsigned)((slabs + slabs_per_cta - 1) / slabs_per_cta);
  const size_t smem = xs_bytes + (size_t)kGemvWarps * 32 * 4 * NG * sizeof(float);
  if (NG == 1) return launch_gemv_kernel(q4_gemv_kernel<1>, grid, smem, p, stream);
  return launch_gemv_kernel(q4_gemv_kernel<2>, grid, smem, p, stream);
}

}  // namespace qmm
