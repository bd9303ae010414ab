// 4-bit decode GEMV for 2 <= M <= 16 tokens.
//
// The weights are 32x256 q4_1 tiles ("NPU engine: full ELFs, no xclbin", "Q4NX
// chunks"; w = q*scale + min, "Zaya 8B Q4NX on the AMD NPU", round 26).  At
// decode sizes the work is bound by the weight stream, and the tiles are
// never expanded in memory.  Two kernels: over many tile rows, a producer
// thread streams whole tile rows into a shared ring (q4_gemv_ring_kernel);
// for fewer rows, each warp walks its slab's tiles with loads prefetched in
// registers and the warps of a CTA split K (q4_gemv_kernel).
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
#include <algorithm>

#include "qmm_internal.h"
#include "umma.cuh"

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
// xload(ng) gives this thread's 16 bytes of x (token 8 ng + g, the block's
// elements 8t .. 8t + 7).
template <int NG, bool kOneCol, typename XLoad>
__device__ __forceinline__ void gemv_block_x(const SlabTile& cur, int b, int lane, const float* xs, XLoad xload,
                                             float (&y)[NG][4]) {
  const int t = lane & 3;
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
    const uint4 xv = xload(ng);
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

template <int NG, bool kOneCol>
__device__ __forceinline__ void gemv_block(const SlabTile& cur, int b, int lane, int t, int blk_x, const float* xs,
                                           const __nv_bfloat16* const (&xrow)[NG], float (&y)[NG][4]) {
  gemv_block_x<NG, kOneCol>(cur, b, lane, xs, [&](int ng) {
    return xrow[ng] ? ldg128(xrow[ng] + blk_x + 8 * t) : make_uint4(0u, 0u, 0u, 0u);
  }, y);
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

// ---------------------------------------------------------------------------
// Streaming decode GEMV for 2 <= M <= 16 over many tile rows (the lm_head
// shape).  One producer thread fills a ring in shared memory with whole tile
// rows, as TMA boxes of up to six tiles seen as lines of 128 bytes with the
// 128-byte swizzle: 16-byte unit u of line l lands at unit u ^ (l & 7), so
// the eight rows a warp reads in one step sit in eight different bank
// groups.  x of every token is staged once in shared memory, each token's
// row padded by 64 bytes so that the two tokens of a quarter-warp read
// different banks.  Pairs of warps take the tile rows, one 16-row slab each,
// with the block step of the kernel above; the ring slot is released as soon
// as the pair has read it.
// ---------------------------------------------------------------------------
// Consumer warps, in pairs: 8 for one 8-token column group, 16 for two (the
// second group doubles the issue work per byte; measured on lm_head, 16 warps
// took M = 9..16 from 29.3-29.7 to 27.0-28.0 us, and 8 warps stayed faster at
// M = 8: 21.8 against 22.5-22.9 us).  The producer warp comes after them.
__host__ __device__ constexpr int ring_warps(int NG) { return NG == 1 ? 8 : 16; }
constexpr int kRMaxSlots = 16;
constexpr int kRBoxTiles = 6;                     // a box is at most 240 lines
constexpr size_t kRSmemCap = 227 * 1024;

struct Q4GemvRingParams {
  CUtensorMap tm;                                 // the tiles as lines of 128 bytes
  const uint8_t* tiles;
  int N, K, M;
  const __nv_bfloat16* X;
  int64_t ldx;
  float* Y;
  int64_t ldy;
  int slots;                                      // ring slots of one tile row each
  int box_tiles;                                  // tiles per TMA box (divides K / 256)
  int32_t* dev_status;
};

__host__ __device__ inline uint32_t ring_x_stride(int K) { return (uint32_t)K * 2 + 64; }

// Shared-memory bytes past the ring: x of 8 NG tokens, their block sums, the
// barriers and the abort flag.
__host__ __device__ inline size_t ring_tail_bytes(int K, int NG) {
  return (size_t)8 * NG * ring_x_stride(K) + (size_t)(K / 32) * 8 * NG * 4 + 2 * kRMaxSlots * 8 + 16;
}

// Fragment data of thread (g, t) from a swizzled tile (1024-byte aligned) in
// shared memory: word t of blocks 0..7 of rows r0 and r0 + 8 (r0 & 7 == g),
// and the (scale, min) pairs of blocks 2t, 2t + 1, which sit at byte
// 4096 + 32 r + 8 t of the tile.
QMM_DEV void slab_lds_swizzled(SlabTile& d, uint32_t tile, int r0, int t) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = r0 + 8 * h;
    const uint32_t line = tile + (uint32_t)r * 128u;
#pragma unroll
    for (int b = 0; b < 8; ++b) d.c[h][b] = umma::lds32(line + (uint32_t)(((b ^ (r & 7)) << 4) | (4 * t)));
    const int L = 32 + (r >> 2);                         // the pairs' line
    const int u = ((r & 3) << 1) | (t >> 1);             // their 16-byte unit in it
    uint2 pv;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                 : "=r"(pv.x), "=r"(pv.y)
                 : "r"(tile + (uint32_t)L * 128u + (uint32_t)((u ^ (L & 7)) << 4) + 8u * (uint32_t)(t & 1)));
    d.p[h] = pv;
  }
}

template <int NG>
__global__ void __launch_bounds__(32 * (ring_warps(NG) + 1), 1)
    q4_gemv_ring_kernel(const __grid_constant__ Q4GemvRingParams p) {
  using namespace umma;
  constexpr int kRWarps = ring_warps(NG);
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = smem_align(sm_raw, 1024);
  const int TC = p.K / 256;
  const uint32_t row_bytes = (uint32_t)TC * (uint32_t)kTileBytes;
  const uint32_t xstride = ring_x_stride(p.K);
  uint8_t* ring = sm;                                                          // [slots][row_bytes]
  uint8_t* xs = ring + (size_t)p.slots * row_bytes;                            // [8 NG][xstride]
  float* xsum = reinterpret_cast<float*>(xs + (size_t)8 * NG * xstride);       // [K / 32][8 NG]
  uint64_t* full = reinterpret_cast<uint64_t*>(xsum + (p.K / 32) * 8 * NG);    // [kRMaxSlots]
  uint64_t* empty = full + kRMaxSlots;                                         // [kRMaxSlots]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kRMaxSlots);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nrows = p.N / 32;
  const int my_rows = (int)blockIdx.x < nrows ? (nrows - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.tm);
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);   // the two warps of a pair
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kRWarps) {
    // ---- producer: tile rows blockIdx.x, blockIdx.x + gridDim.x, ... ----
    if (lane == 0) {
      // the first two rows into L2 while the previous grid finishes (the
      // copies into shared memory only start after the wait)
      for (int j = 0; j < my_rows && j < 2; ++j)
        bulk_prefetch_l2(p.tiles + (int64_t)((int)blockIdx.x + j * (int)gridDim.x) * row_bytes, row_bytes);
      pdl_wait();
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < my_rows; ++j) {
        const int s = j % p.slots;
        if (!mbar_wait(&empty[s], (uint32_t)(((j / p.slots) & 1) ^ 1), abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        const int tr = (int)blockIdx.x + j * (int)gridDim.x;
        mbar_arrive_expect_tx(&full[s], row_bytes);
        const uint32_t dst = smem_u32(ring) + (uint32_t)s * row_bytes;
        for (int tc = 0; tc < TC; tc += p.box_tiles)
          tma_load_2d_u32(dst + (uint32_t)tc * (uint32_t)kTileBytes, &p.tm, &full[s], 0, (tr * TC + tc) * 40);
        ++issued;
      }
      if (!ok) {
        // the rows already issued land before the CTA leaves: each slot's
        // last issued phase, whether or not it was consumed
        for (int s = 0; s < p.slots && s < issued; ++s) {
          const int last = issued - 1 - ((issued - 1 - s) % p.slots);
          mbar_drain(&full[s], (uint32_t)((last / p.slots) & 1));
        }
      }
    }
    return;
  }

  // ---- consumers: x of every token into shared memory (tokens M .. 8 NG - 1
  // as zeros), the block sums of x, then the tile rows ----
  pdl_wait();   // x and y may belong to the previous grid
  const int xunits = p.K / 8;   // 16-byte units of one token's x
  for (int i = threadIdx.x; i < 8 * NG * xunits; i += kRWarps * 32) {
    const int m = i / xunits, u = i - m * xunits;
    const uint4 v = m < p.M ? ldg128(p.X + (int64_t)m * p.ldx + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
    sts128(smem_u32(xs) + (uint32_t)m * xstride + 16u * (uint32_t)u, v);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kRWarps * 32) : "memory");
  for (int idx = threadIdx.x; idx < (p.K / 32) * 8 * NG; idx += kRWarps * 32) {
    const int blk = idx / (8 * NG), m = idx - blk * 8 * NG;
    const uint32_t xa = smem_u32(xs) + (uint32_t)m * xstride + 64u * (uint32_t)blk;
    float sum = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 w = lds128(xa + 16u * v);
      sum += bf16lo_to_f32(w.x) + bf16hi_to_f32(w.x) + bf16lo_to_f32(w.y) + bf16hi_to_f32(w.y) +
             bf16lo_to_f32(w.z) + bf16hi_to_f32(w.z) + bf16lo_to_f32(w.w) + bf16hi_to_f32(w.w);
    }
    xsum[idx] = sum;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kRWarps * 32) : "memory");

  // Pair q takes this CTA's rows q, q + P, ... (P = min(4, slots) pairs; the
  // launcher makes the slot count a multiple of P, so the rows sharing a slot
  // all belong to one pair and are consumed in order).
  const int pair = warp >> 1, slab = warp & 1;
  const int npairs = min(kRWarps / 2, p.slots);
  const uint32_t xthr = smem_u32(xs) + (uint32_t)g * xstride + 16u * (uint32_t)t;   // token g, elements 8t ..
  for (int j = pair < npairs ? pair : my_rows; j < my_rows; j += npairs) {
    const int s = j % p.slots;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)((j / p.slots) & 1), abort_flag, p.dev_status)))
      break;
    const uint32_t rowbase = smem_u32(ring) + (uint32_t)s * row_bytes;
    float y[NG][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 4; ++c) y[ng][c] = 0.f;
    for (int tc = 0; tc < TC; ++tc) {
      SlabTile d;
      slab_lds_swizzled(d, rowbase + (uint32_t)tc * (uint32_t)kTileBytes, 16 * slab + g, t);
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t xb = xthr + (uint32_t)(tc * 256 + 32 * b) * 2u;
        gemv_block_x<NG, false>(d, b, lane, xsum + (tc * 8 + b) * 8 * NG,
                                [&](int ng) { return lds128(xb + (uint32_t)(8 * ng) * xstride); }, y);
      }
    }
    // every lane's shared-memory reads of this slot are done
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const int nrow0 = ((int)blockIdx.x + j * (int)gridDim.x) * 32 + 16 * slab;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = 8 * ng + 2 * t + (c & 1);
        if (m < p.M) p.Y[(int64_t)m * p.ldy + nrow0 + g + 8 * (c >> 1)] = y[ng][c];
      }
  }
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
  const int NG = a.M <= 8 ? 1 : 2;
  if (a.N / 32 >= 2 * sms) {
    // many tile rows: the streaming ring kernel, where x and at least three
    // tile rows fit in shared memory
    const int TC = a.K / 256;
    const size_t row_bytes = (size_t)TC * kTileBytes;
    const size_t fixed = 1024 + ring_tail_bytes(a.K, NG);
    int slots = 0;
    if (fixed + 3 * row_bytes <= kRSmemCap) {
      slots = (int)std::min<size_t>((kRSmemCap - fixed) / row_bytes, kRMaxSlots);
      if (slots >= ring_warps(NG) / 2) slots -= slots % (ring_warps(NG) / 2);   // a multiple of the active pairs
    }
    if (slots >= 3) {
      Q4GemvRingParams p{};
      int bt = std::min(TC, kRBoxTiles);
      while (TC % bt != 0) --bt;   // boxes never cross a tile row
      if (!make_tmap_2d(&p.tm, false, const_cast<uint8_t*>(a.tiles), 64, (uint64_t)(a.N / 32) * TC * 40, 128, 64,
                        (uint32_t)(40 * bt)))
        return cudaErrorInvalidValue;
      p.tiles = a.tiles;
      p.N = a.N;
      p.K = a.K;
      p.M = a.M;
      p.X = a.X;
      p.ldx = a.ldx;
      p.Y = a.Y;
      p.ldy = a.ldy;
      p.slots = slots;
      p.box_tiles = bt;
      p.dev_status = dev_status;
      const size_t smem = fixed + (size_t)slots * row_bytes;
      auto kern = NG == 1 ? q4_gemv_ring_kernel<1> : q4_gemv_ring_kernel<2>;
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_pdl(kern, dim3((unsigned)sms), dim3(32 * (ring_warps(NG) + 1)), smem, stream, p);
    }
  }
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
