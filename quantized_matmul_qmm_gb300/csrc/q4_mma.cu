// 4-bit GEMV / small-batch GEMM and the MUL_MAT_ID (mixture-of-experts) path.
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
// MMA fragment mapping: within one block, thread t of a quad owns code word
// (row, 8t + b) = columns 32b + 8t .. 32b + 8t + 7 and the matching 16 bytes
// of x.  The logical k order inside the MMA is a permutation of these, the
// same for A and B.
//
// MUL_MAT_ID ("The bugs that were the work"): the expert of (token t, slot i)
// is ids[t*ld_ids + i], a strided view.  Slot i of token t reads the
// activation row t*ldx_token + i*ldx_slot, which covers both the shared src1
// of gate/up (ldx_slot = 0) and the per-slot src1 of down (ldx_slot = K).
// A one-CTA router groups the (token, slot) pairs by expert.  The grouped
// kernel then runs the same tile loop over each expert's pairs, eight pairs
// per MMA column group.
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kMaxWarpsK = 8;

template <int NG>
struct Q4Acc {
  float y[2][NG][4];
};

// Process one tile (32 rows x 256 columns) for the calling warp.
// xrow[ng]: activation row of column g of group ng (nullptr = zero column).
template <int NG>
__device__ __forceinline__ void q4_tile(const uint8_t* __restrict__ tile, int64_t kbase,
                                        const __nv_bfloat16* const (&xrow)[NG], Q4Acc<NG>& acc,
                                        int g, int t) {
  // codes: rows g, g+8, g+16, g+24; word t of every block b (byte 16b + 4t of the row)
  uint32_t cw[4][8];
  uint4 pw[4][2];
#pragma unroll
  for (int rs = 0; rs < 4; ++rs) {
    const int r = g + 8 * rs;
    const uint8_t* rowp = tile + r * 128 + 4 * t;
#pragma unroll
    for (int b = 0; b < 8; ++b) cw[rs][b] = ldg32(rowp + 16 * b);
    const uint8_t* pp = tile + 4096 + r * 32;
    pw[rs][0] = ldg128(pp);
    pw[rs][1] = ldg128(pp + 16);
  }
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    uint4 xv[NG];
    float xs0[NG], xs1[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      xv[ng] = xrow[ng] ? ldg128(xrow[ng] + kbase + b * 32 + 8 * t) : make_uint4(0u, 0u, 0u, 0u);
      float s = bf16lo_to_f32(xv[ng].x) + bf16hi_to_f32(xv[ng].x) + bf16lo_to_f32(xv[ng].y) +
                bf16hi_to_f32(xv[ng].y) + bf16lo_to_f32(xv[ng].z) + bf16hi_to_f32(xv[ng].z) +
                bf16lo_to_f32(xv[ng].w) + bf16hi_to_f32(xv[ng].w);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      xs0[ng] = __shfl_sync(0xffffffffu, s, (2 * t) * 4);
      xs1[ng] = __shfl_sync(0xffffffffu, s, (2 * t + 1) * 4);
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint32_t wA = cw[2 * mt][b];
      const uint32_t wB = cw[2 * mt + 1][b];
      const uint32_t pA = u4_get(pw[2 * mt][b >> 2], b & 3);
      const uint32_t pB = u4_get(pw[2 * mt + 1][b >> 2], b & 3);
      const float sA = bf16lo_to_f32(pA), sB = bf16lo_to_f32(pB);
      const float mA = fmaf(-128.0f, sA, bf16hi_to_f32(pA));
      const float mB = fmaf(-128.0f, sB, bf16hi_to_f32(pB));
      const uint32_t a00 = q4_pair_biased(wA, 0), a01 = q4_pair_biased(wB, 0);
      const uint32_t a02 = q4_pair_biased(wA, 1), a03 = q4_pair_biased(wB, 1);
      const uint32_t a10 = q4_pair_biased(wA, 2), a11 = q4_pair_biased(wB, 2);
      const uint32_t a12 = q4_pair_biased(wA, 3), a13 = q4_pair_biased(wB, 3);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16_16816(c, a00, a01, a02, a03, xv[ng].x, xv[ng].y);
        mma_bf16_16816(c, a10, a11, a12, a13, xv[ng].z, xv[ng].w);
        float* y = acc.y[mt][ng];
        y[0] = fmaf(sA, c[0], fmaf(mA, xs0[ng], y[0]));
        y[1] = fmaf(sA, c[1], fmaf(mA, xs1[ng], y[1]));
        y[2] = fmaf(sB, c[2], fmaf(mB, xs0[ng], y[2]));
        y[3] = fmaf(sB, c[3], fmaf(mB, xs1[ng], y[3]));
      }
    }
  }
}

// Items are activation/output rows: dense mode uses row m directly; MoE mode
// maps item i of expert e to the pair pairs[offsets[e] + i] = t*n_used + slot.
struct Q4SmallParams {
  const uint8_t* tiles;     // expert 0 tiles (dense: the only set)
  int64_t expert_bytes;     // bytes per expert tile set
  int N, K;
  const __nv_bfloat16* X;
  int64_t ldx_token, ldx_slot;
  float* Y;
  int64_t ldy_token, ldy_slot;
  int n_items;              // dense: M
  int n_used;               // MoE: slots per token (dense: 1)
  const int32_t* offsets;   // MoE only
  const int32_t* pairs;     // MoE only
};

template <int NG, bool kMoE>
__global__ void __launch_bounds__(kMaxWarpsK * 32) q4_small_kernel(const Q4SmallParams p) {
  __shared__ float red[kMaxWarpsK][32][2 * NG * 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wk = blockDim.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int tr = blockIdx.x;
  const int TC = p.K / 256;

  int item0 = 0, n_items = p.n_items;
  const uint8_t* tiles = p.tiles;
  if (kMoE) {
    const int e = blockIdx.y;
    item0 = p.offsets[e];
    n_items = p.offsets[e + 1] - item0;
    tiles += (int64_t)e * p.expert_bytes;
  }
  const uint8_t* rowtiles = tiles + (int64_t)tr * TC * kTileBytes;

  for (int chunk = 0; chunk < n_items; chunk += 8 * NG) {
    const __nv_bfloat16* xrow[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int it = chunk + ng * 8 + g;
      xrow[ng] = nullptr;
      if (it < n_items) {
        int64_t off;
        if (kMoE) {
          const int pr = p.pairs[item0 + it];
          off = (int64_t)(pr / p.n_used) * p.ldx_token + (int64_t)(pr % p.n_used) * p.ldx_slot;
        } else {
          off = (int64_t)it * p.ldx_token;
        }
        xrow[ng] = p.X + off;
      }
    }
    Q4Acc<NG> acc;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc.y[mt][ng][c] = 0.f;

    for (int tc = warp; tc < TC; tc += wk)
      q4_tile<NG>(rowtiles + (int64_t)tc * kTileBytes, (int64_t)tc * 256, xrow, acc, g, t);

#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[warp][lane][(mt * NG + ng) * 4 + c] = acc.y[mt][ng][c];
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * 2 * NG * 4; idx += blockDim.x) {
      const int l = idx / (2 * NG * 4), v = idx % (2 * NG * 4);
      float s = 0.f;
      for (int w = 0; w < wk; ++w) s += red[w][l][v];
      const int gg = l >> 2, tt = l & 3;
      const int c = v & 3, ng = (v >> 2) % NG, mt = (v >> 2) / NG;
      const int n = tr * 32 + mt * 16 + gg + 8 * (c >> 1);
      const int it = chunk + ng * 8 + 2 * tt + (c & 1);
      if (it >= n_items) continue;
      int64_t off;
      if (kMoE) {
        const int pr = p.pairs[item0 + it];
        off = (int64_t)(pr / p.n_used) * p.ldy_token + (int64_t)(pr % p.n_used) * p.ldy_slot;
      } else {
        off = (int64_t)it * p.ldy_token;
      }
      p.Y[off + n] = s;
    }
    __syncthreads();
  }
}

// One CTA: count pairs per expert, prefix-sum, scatter pair ids by expert.
__global__ void __launch_bounds__(1024)
moe_route_kernel(const int32_t* __restrict__ ids, int64_t ld_ids, int n_used, int T, int n_expert,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ pairs, int32_t* dev_status) {
  extern __shared__ int sm[];
  int* cnt = sm;               // [n_expert]
  int* cursor = sm + n_expert; // [n_expert]
  const int tid = threadIdx.x;
  for (int e = tid; e < n_expert; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int npairs = T * n_used;
  bool bad = false;
  for (int p = tid; p < npairs; p += blockDim.x) {
    const int t = p / n_used, i = p % n_used;
    const int e = ids[(int64_t)t * ld_ids + i];
    if (e < 0 || e >= n_expert) { bad = true; continue; }
    atomicAdd(&cnt[e], 1);
  }
  if (bad) set_status(dev_status, QMM_ERR_BAD_EXPERT_ID);
  __syncthreads();
  if (tid < 32) {
    // warp scan over contiguous segments of the expert range
    const int per = (n_expert + 31) / 32;
    const int lo = min(tid * per, n_expert), hi = min(lo + per, n_expert);
    int seg = 0;
    for (int e = lo; e < hi; ++e) seg += cnt[e];
    int incl = seg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (tid >= d) incl += v;
    }
    int run = incl - seg;
    for (int e = lo; e < hi; ++e) {
      offsets[e] = run;
      cursor[e] = run;
      run += cnt[e];
    }
    if (tid == 31) offsets[n_expert] = incl;
  }
  __syncthreads();
  for (int p = tid; p < npairs; p += blockDim.x) {
    const int t = p / n_used, i = p % n_used;
    const int e = ids[(int64_t)t * ld_ids + i];
    if (e < 0 || e >= n_expert) continue;
    pairs[atomicAdd(&cursor[e], 1)] = p;
  }
}

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

template <int NG, bool kMoE>
cudaError_t launch_small(const Q4SmallParams& p, dim3 grid, int wk, cudaStream_t stream) {
  q4_small_kernel<NG, kMoE><<<grid, wk * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

template <typename Kern>
cudaError_t launch_gemv_kernel(Kern kern, unsigned grid, size_t smem, const Q4GemvParams& p, cudaStream_t stream) {
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kGemvWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_q4_gemv(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream) {
  (void)dev_status;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (a.M == 1) return launch_q4_gemv1(a, sms, stream);
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

size_t q4_moe_workspace_bytes(int64_t n_expert, int64_t n_used, int64_t T) {
  const size_t off = ((size_t)(n_expert + 1) * 4 + 255) / 256 * 256;
  return off + (size_t)(T * n_used) * 4;
}

cudaError_t launch_q4_moe(const Q4MoEArgs& a, cudaStream_t stream) {
  const size_t smem = (size_t)a.n_expert * 2 * sizeof(int);
  moe_route_kernel<<<1, 1024, smem, stream>>>(a.ids, a.ld_ids, a.n_used, a.T, a.n_expert,
                                              a.offsets, a.pairs, a.dev_status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  Q4SmallParams p{};
  p.tiles = a.tiles;
  p.expert_bytes = (int64_t)(a.N / 32) * (a.K / 256) * kTileBytes;
  p.N = a.N;
  p.K = a.K;
  p.X = a.X;
  p.ldx_token = a.ldx_token;
  p.ldx_slot = a.ldx_slot;
  p.Y = a.Y;
  p.ldy_token = a.ldy_token;
  p.ldy_slot = a.ldy_slot;
  p.n_used = a.n_used;
  p.offsets = a.offsets;
  p.pairs = a.pairs;
  const int TC = a.K / 256;
  const int wk = TC < kMaxWarpsK ? TC : kMaxWarpsK;
  dim3 grid((unsigned)(a.N / 32), (unsigned)a.n_expert);
  return launch_small<4, true>(p, grid, wk, stream);
}

}  // namespace qmm
