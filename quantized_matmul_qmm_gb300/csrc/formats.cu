// Two more weight formats ("NPU engine: full ELFs, no xclbin", section "Q4NX
// chunks").
//
// Q4_K -> q4_1.  The section converts Q4_K weights to q4_1 so that q4_1
// kernels can use them; the only loss is the bf16 rounding of the two
// per-sub-block products (super-block scale times scale code, super-block
// min scale times min code).  A Q4_K super-block (GGML's published k-quant layout)
// covers 256 weights of one row in 144 bytes: fp16 d and dmin, twelve bytes
// of 6-bit scale and min codes for the eight 32-weight sub-blocks, and 128
// bytes of 4-bit codes (byte 32c + l: weight 64c + l in the low nibble,
// weight 64c + 32 + l in the high one); w = d*sc_j*q - dmin*mn_j.  One
// super-block becomes one tile row of the q4 format: the same codes, scale
// bf16(d*sc_j) and min bf16(-(dmin*mn_j)).  Both products are exact in fp32,
// so each is rounded once.
//
// Q8 tiles.  The same 32 x 256 tile grid with 8-bit codes in one of the
// section's two layouts: code (r, k) at byte k*32 + r (layout 0) or at
// (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16 (layout 1).  Bytes
// [8192, 8704) of a tile hold one bf16 scale per (row r, block g of 32
// columns) at 8192 + 2*(32 g + r); w = code * scale.  In both layouts a
// 16-byte group is 16 consecutive rows (a slab) at one column k, which is what
// the decode GEMV reads.
//
// Decode GEMV (M <= 16): a warp owns one slab (16 output rows) of a tile row
// and walks its tiles, or every wpu-th of them when wpu warps share a slab
// (small N).  With one warp per slab the grid is one resident wave and each
// warp streams slab after slab, loading the next tile while it computes the
// current one, across slab boundaries too.
// Lane l reads the eight groups of columns 8l .. 8l+7 (one 32-column block,
// so one scale per row), forms each row's 8-term partial dot product per
// activation row, scales it, and a reduce-scatter across the warp (16 + 1
// shuffles for 16 rows) leaves row (l & 15)'s sum in lane l.  With one
// activation row the scaled partials stay in the lane across tiles and the
// warp reduces once per slab.  Rows go in pairs through the packed f32x2
// instructions.  Codes are converted exactly and code * x is exact in fp32;
// only the fp32 sums round.
//
// Larger M: the tiles are decoded to bf16 weights bf16(code * scale) (one
// rounding) in the workspace, and the pair tensor-core GEMM of the W8A16
// path runs on them with unit chunk scales.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "f16_operands.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kQ4KBytes = 144;
constexpr int kRepackThreads = 256;

// The byte i (0..11) of the scale field, which words w1..w3 hold.
__device__ __forceinline__ uint32_t q4k_scale_byte(uint32_t w1, uint32_t w2, uint32_t w3, int i) {
  const uint32_t w = i < 4 ? w1 : (i < 8 ? w2 : w3);
  return (w >> (8 * (i & 3))) & 0xFFu;
}

__global__ void __launch_bounds__(kRepackThreads)
repack_q4k_kernel(const uint8_t* __restrict__ src, int64_t row_bytes, int N, int nsb, uint8_t* __restrict__ tiles) {
  const int64_t idx = (int64_t)blockIdx.x * kRepackThreads + threadIdx.x;
  if (idx >= (int64_t)N * nsb) return;
  const int n = (int)(idx / nsb), j = (int)(idx % nsb);
  const uint4* blk = reinterpret_cast<const uint4*>(src + (int64_t)n * row_bytes + (int64_t)j * kQ4KBytes);
  uint32_t w[36];
#pragma unroll
  for (int t = 0; t < 9; ++t) {
    const uint4 v = ldg128_stream(blk + t);
    w[4 * t] = v.x;
    w[4 * t + 1] = v.y;
    w[4 * t + 2] = v.z;
    w[4 * t + 3] = v.w;
  }
  const float d = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(w[0] >> 16)));
  uint32_t pairs[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    uint32_t sc, mn;
    if (b < 4) {
      sc = q4k_scale_byte(w[1], w[2], w[3], b) & 63u;
      mn = q4k_scale_byte(w[1], w[2], w[3], b + 4) & 63u;
    } else {
      const uint32_t lo = q4k_scale_byte(w[1], w[2], w[3], b + 4);
      sc = (lo & 15u) | ((q4k_scale_byte(w[1], w[2], w[3], b - 4) >> 6) << 4);
      mn = (lo >> 4) | ((q4k_scale_byte(w[1], w[2], w[3], b) >> 6) << 4);
    }
    const __nv_bfloat16 s = __float2bfloat16_rn(__fmul_rn(d, (float)sc));
    const __nv_bfloat16 m = __float2bfloat16_rn(-__fmul_rn(dmin, (float)mn));
    pairs[b] = (uint32_t)__bfloat16_as_ushort(s) | ((uint32_t)__bfloat16_as_ushort(m) << 16);
  }
  const int tr = n / (int)kTileRows, r = n % (int)kTileRows;
  uint8_t* tile = tiles + ((int64_t)tr * nsb + j) * kTileBytes;
  // codes: block b of row r is 4 words; word t holds columns 32b + 8t + jj,
  // code jj = 2i at bits 4i and jj = 2i+1 at bits 16 + 4i.  The source byte of
  // column 32b + l is 32(b/2) + l (code words 4..35), nibble b % 2.
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const int c = b >> 1, sh = 4 * (b & 1);
    uint32_t out[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t lo = w[4 + 8 * c + 2 * t], hi = w[4 + 8 * c + 2 * t + 1];
      uint32_t o = 0;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t src_w = jj < 4 ? lo : hi;
        const uint32_t code = (src_w >> (8 * (jj & 3) + sh)) & 15u;
        o |= code << ((jj & 1) ? 16 + 4 * (jj >> 1) : 4 * (jj >> 1));
      }
      out[t] = o;
    }
    *reinterpret_cast<uint4*>(tile + 128 * r + 16 * b) = make_uint4(out[0], out[1], out[2], out[3]);
  }
  uint4* pdst = reinterpret_cast<uint4*>(tile + 4096 + 32 * r);
  pdst[0] = make_uint4(pairs[0], pairs[1], pairs[2], pairs[3]);
  pdst[1] = make_uint4(pairs[4], pairs[5], pairs[6], pairs[7]);
}

// ---------------------------------------------------------------------------
// Q8 tiles
// ---------------------------------------------------------------------------

template <int kLayout>
__device__ __forceinline__ int q8_offset(int r, int k) {
  if constexpr (kLayout == 0) return k * 32 + r;
  else return (r >> 4) * 4096 + (k >> 5) * 512 + (k & 31) * 16 + (r & 15);
}

constexpr int kTileThreads = 256;   // one thread per (row, 32-column block) of a tile

template <int kLayout>
__global__ void __launch_bounds__(kTileThreads)
pack_q8_kernel(const float* __restrict__ W, int64_t ldw, int TC, uint8_t* __restrict__ tiles) {
  __shared__ __align__(16) uint8_t img[kQ8TileBytes];
  const int tile_id = blockIdx.x;
  const int tr = tile_id / TC, tc = tile_id % TC;
  const int r = threadIdx.x & 31, g = threadIdx.x >> 5;
  const float* src = W + (int64_t)(32 * tr + r) * ldw + 256 * tc + 32 * g;
  float x[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    x[i] = __ldg(src + i);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(amax, 127.0f));
  const float s = __bfloat162float(sb);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int q = 0;
    if (s > 0.f) q = min(max(__float2int_rn(__fdiv_rn(x[i], s)), -127), 127);
    img[q8_offset<kLayout>(r, 32 * g + i)] = (uint8_t)(q & 0xFF);
  }
  reinterpret_cast<__nv_bfloat16*>(img + kQ8CodeBytes)[32 * g + r] = sb;
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(tiles + (int64_t)tile_id * kQ8TileBytes);
  for (int i = threadIdx.x; i < kQ8TileBytes / 16; i += kTileThreads) dst[i] = reinterpret_cast<const uint4*>(img)[i];
}

// Codes of rows 2p and 2p+1 (bytes of word xw, already XORed with 0x80) as an
// fp32 pair: each byte becomes the low mantissa byte of 2^23, and 2^23 + 128
// is subtracted (exact).
__device__ __forceinline__ uint64_t q8_code_pair(uint32_t xw, int p) {
  const uint32_t sel = 0x7540u + (uint32_t)(2 * (p & 1));
  const float lo = __uint_as_float(__byte_perm(xw, 0x4B000000u, sel));
  const float hi = __uint_as_float(__byte_perm(xw, 0x4B000000u, sel + 1));
  const float c = -8388736.0f;
  return f2_add(f2_pack(lo, hi), f2_pack(c, c));
}

// Reduce-scatter of 16 per-row values over the warp: lane l returns the sum,
// over all 32 lanes, of row (l & 15).
__device__ __forceinline__ float warp_rows16(float (&v)[16], int lane) {
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = up ? v[i] : v[i + 8];
      const float keep = up ? v[i + 8] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = up ? v[i] : v[i + 4];
      const float keep = up ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = up ? v[i] : v[i + 2];
      const float keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
  }
  {
    const bool up = lane & 1;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

constexpr int kQ8GvWarps = 8;

struct Q8Group {
  uint4 v[8];   // codes: v[j] = rows 16h .. 16h+15 at column 8 lane + j
  uint4 s[2];   // the 16 rows' bf16 scales of the lane's 32-column block
};

template <int kLayout>
__device__ __forceinline__ void q8_load(Q8Group& q, const uint8_t* tile, int lane, int h) {
  const int g = lane >> 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int off = kLayout == 0 ? (8 * lane + j) * 32 + 16 * h : h * 4096 + g * 512 + (lane & 3) * 128 + 16 * j;
    q.v[j] = ldg128_stream(tile + off);
  }
  const uint8_t* sp = tile + kQ8CodeBytes + 2 * (32 * g + 16 * h);
  q.s[0] = ldg128(sp);
  q.s[1] = ldg128(sp + 16);
}

// The lane's 16 row sums over its 8 columns for one activation row, as 8
// pairs (rows 2p, 2p+1): an 8-term fp32 fma chain per row, codes exact.
__device__ __forceinline__ void q8_rows_dot(const uint32_t (&xw)[8][4], const uint4 xv, uint64_t (&part)[8]) {
  const uint32_t xr[4] = {xv.x, xv.y, xv.z, xv.w};
  uint64_t xx[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = bf16lo_to_f32(xr[i]), hi = bf16hi_to_f32(xr[i]);
    xx[2 * i] = f2_pack(lo, lo);
    xx[2 * i + 1] = f2_pack(hi, hi);
  }
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    uint64_t a = f2_mul(q8_code_pair(xw[0][p >> 1], p), xx[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j) a = f2_fma(q8_code_pair(xw[j][p >> 1], p), xx[j], a);
    part[p] = a;
  }
}

// One tile of a slab: the lane's 16 row sums over its 8 columns, scaled.
// With one activation row they accumulate in racc (pairs of rows) for the
// reduction at the end of the slab; otherwise each activation row is reduced
// across the warp here and added to acc[m] (row l & 15 in lane l).
template <int kM>
__device__ __forceinline__ void q8_tile_compute(const Q8Group& cur, int tc, int lane, const __nv_bfloat16* X,
                                                int64_t ldx, int M, uint64_t (&racc)[8], float (&acc)[kM]) {
  uint64_t sc[8];   // scales of rows (2p, 2p+1)
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t sw = u4_get(cur.s[p >> 2], p & 3);
    sc[p] = f2_pack(bf16lo_to_f32(sw), bf16hi_to_f32(sw));
  }
  uint32_t xw[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    xw[j][0] = cur.v[j].x ^ 0x80808080u;
    xw[j][1] = cur.v[j].y ^ 0x80808080u;
    xw[j][2] = cur.v[j].z ^ 0x80808080u;
    xw[j][3] = cur.v[j].w ^ 0x80808080u;
  }
  const int k0 = 256 * tc + 8 * lane;
  if constexpr (kM == 1) {
    uint64_t pr[8];
    q8_rows_dot(xw, ldg128(X + k0), pr);
#pragma unroll
    for (int p = 0; p < 8; ++p) racc[p] = f2_fma(pr[p], sc[p], racc[p]);
  } else {
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      if (m >= M) break;
      uint64_t pr[8];
      q8_rows_dot(xw, ldg128(X + (int64_t)m * ldx + k0), pr);
      float v[16];
#pragma unroll
      for (int p = 0; p < 8; ++p) f2_unpack(f2_mul(pr[p], sc[p]), v[2 * p], v[2 * p + 1]);
      acc[m] += warp_rows16(v, lane);
    }
  }
}

// The slab's results: row 16u + l in lane l < 16.
template <int kM>
__device__ __forceinline__ void q8_slab_finish(int lane, uint64_t (&racc)[8], float (&acc)[kM]) {
  if constexpr (kM == 1) {
    float v[16];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      f2_unpack(racc[p], v[2 * p], v[2 * p + 1]);
      racc[p] = 0ull;
    }
    acc[0] = warp_rows16(v, lane);
  }
}

template <int kM, int kLayout>
__global__ void __launch_bounds__(kQ8GvWarps * 32)
q8_gemv_kernel(const uint8_t* __restrict__ tiles, int TR, int TC, const __nv_bfloat16* __restrict__ X, int64_t ldx,
               float* __restrict__ Y, int64_t ldy, int M, int wpu) {
  __shared__ float red[kQ8GvWarps][kM][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nunits = 2 * TR;
  uint64_t racc[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) racc[p] = 0ull;
  float acc[kM];
#pragma unroll
  for (int m = 0; m < kM; ++m) acc[m] = 0.f;

  if (wpu == 1) {
    // every warp on its own: one stream of (slab, tile) pairs, slab u, u + the
    // grid's warp count, ...; the next pair's loads are issued before the
    // current one is computed, across slab boundaries too
    const int tw = (int)gridDim.x * kQ8GvWarps;
    int u = (int)blockIdx.x * kQ8GvWarps + warp;
    if (u >= nunits) return;
    int tc = 0;
    Q8Group nxt;
    q8_load<kLayout>(nxt, tiles + (int64_t)(u >> 1) * TC * kQ8TileBytes, lane, u & 1);
    while (true) {
      const Q8Group cur = nxt;
      int nu = u, ntc = tc + 1;
      if (ntc == TC) {
        nu = u + tw;
        ntc = 0;
      }
      if (nu < nunits) q8_load<kLayout>(nxt, tiles + ((int64_t)(nu >> 1) * TC + ntc) * kQ8TileBytes, lane, nu & 1);
      q8_tile_compute<kM>(cur, tc, lane, X, ldx, M, racc, acc);
      if (ntc == 0) {
        q8_slab_finish<kM>(lane, racc, acc);
        if (lane < 16) {
          const int n = 16 * u + lane;
#pragma unroll
          for (int m = 0; m < kM; ++m)
            if (m < M) Y[(int64_t)m * ldy + n] = acc[m];
        }
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[m] = 0.f;
      }
      if (nu >= nunits) break;
      u = nu;
      tc = ntc;
    }
    return;
  }

  // wpu warps share a slab, each taking every wpu-th tile; the block adds
  // their partial sums in a fixed order
  const int upb = kQ8GvWarps / wpu;                 // slabs per block
  const int unit_l = warp / wpu, part = warp % wpu;
  const int ngroups = (nunits + upb - 1) / upb;
  for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
    const int u = grp * upb + unit_l;
    if (u < nunits) {
      const uint8_t* row_tiles = tiles + (int64_t)(u >> 1) * TC * kQ8TileBytes;
      Q8Group nxt;
      if (part < TC) q8_load<kLayout>(nxt, row_tiles + (int64_t)part * kQ8TileBytes, lane, u & 1);
      for (int tc = part; tc < TC; tc += wpu) {
        const Q8Group cur = nxt;
        if (tc + wpu < TC) q8_load<kLayout>(nxt, row_tiles + (int64_t)(tc + wpu) * kQ8TileBytes, lane, u & 1);
        q8_tile_compute<kM>(cur, tc, lane, X, ldx, M, racc, acc);
      }
      q8_slab_finish<kM>(lane, racc, acc);
    }
    if (lane < 16) {
#pragma unroll
      for (int m = 0; m < kM; ++m) red[warp][m][lane] = acc[m];
    }
    __syncthreads();
    if (part == 0 && u < nunits && lane < 16) {
      const int n = 16 * u + lane;
#pragma unroll
      for (int m = 0; m < kM; ++m) {
        if (m >= M) break;
        float a = 0.f;
        for (int p = 0; p < wpu; ++p) a += red[warp + p][m][lane];
        Y[(int64_t)m * ldy + n] = a;
      }
    }
#pragma unroll
    for (int m = 0; m < kM; ++m) acc[m] = 0.f;
    __syncthreads();
  }
}

// Q8 tiles -> f16 weights f16(code * scale) as rows [N][K] (the pair GEMM's
// B operand), and unit chunk scales [N][nb].  code * scale is exact in fp32
// (8 by 8 significant bits), so each weight is rounded once.  A block whose
// weights could pass f16's largest value (128 |s| > 65504) reports
// QMM_ERR_RANGE.
template <int kLayout>
__global__ void __launch_bounds__(kTileThreads)
q8_decode_f16_kernel(const uint8_t* __restrict__ tiles, int TC, int K, __half* __restrict__ W16,
                     float* __restrict__ ones, int nb, int32_t* dev_status) {
  __shared__ __align__(16) uint8_t img[kQ8TileBytes];
  const int tile_id = blockIdx.x;
  const int tr = tile_id / TC, tc = tile_id % TC;
  const uint4* src = reinterpret_cast<const uint4*>(tiles + (int64_t)tile_id * kQ8TileBytes);
  for (int i = threadIdx.x; i < kQ8TileBytes / 16; i += kTileThreads) reinterpret_cast<uint4*>(img)[i] = ldg128_stream(src + i);
  __syncthreads();
  const int r = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int n = 32 * tr + r;
  const float s = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(img + kQ8CodeBytes)[32 * g + r]);
  if (128.0f * fabsf(s) > kF16Max) set_status(dev_status, QMM_ERR_RANGE);
  uint4* dst = reinterpret_cast<uint4*>(W16 + (int64_t)n * K + 256 * tc + 32 * g);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 32 * g + 8 * c + 2 * i;
      const float w0 = __fmul_rn((float)(int8_t)img[q8_offset<kLayout>(r, k)], s);
      const float w1 = __fmul_rn((float)(int8_t)img[q8_offset<kLayout>(r, k + 1)], s);
      o[i] = (uint32_t)__half_as_ushort(__float2half_rn(w0)) | ((uint32_t)__half_as_ushort(__float2half_rn(w1)) << 16);
    }
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (tc == 0 && g == 0)
    for (int b = 0; b < nb; ++b) ones[(int64_t)n * nb + b] = 1.0f;
}

template <int kM>
cudaError_t q8_gemv_launch(int layout, int units, int sms, const uint8_t* tiles, int TR, int TC,
                           const __nv_bfloat16* X, int64_t ldx, float* Y, int64_t ldy, int M, int wpu,
                           cudaStream_t stream) {
  auto kern = layout == 0 ? q8_gemv_kernel<kM, 0> : q8_gemv_kernel<kM, 1>;
  const int upb = kQ8GvWarps / wpu;
  const int ngroups = (units + upb - 1) / upb;
  int grid = std::min(ngroups, 8 * sms);
  if (wpu == 1) {
    // one resident wave: each warp streams several slabs without a relaunch
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQ8GvWarps * 32, 0);
    if (err != cudaSuccess) return err;
    grid = std::min(ngroups, std::max(1, per_sm) * sms);
  }
  kern<<<std::max(1, grid), kQ8GvWarps * 32, 0, stream>>>(tiles, TR, TC, X, ldx, Y, ldy, M, wpu);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_repack_q4k(const uint8_t* src, int64_t row_bytes, int N, int K, uint8_t* tiles,
                              cudaStream_t stream) {
  const int nsb = K / (int)kTileCols;
  const int64_t total = (int64_t)N * nsb;
  const int64_t grid = (total + kRepackThreads - 1) / kRepackThreads;
  repack_q4k_kernel<<<(unsigned)grid, kRepackThreads, 0, stream>>>(src, row_bytes, N, nsb, tiles);
  return cudaGetLastError();
}

cudaError_t launch_pack_q8(const float* W, int64_t ldw, int N, int K, int layout, uint8_t* tiles,
                           cudaStream_t stream) {
  const int TR = N / (int)kTileRows, TC = K / (int)kTileCols;
  const int64_t ntiles = (int64_t)TR * TC;
  if (layout == 0) pack_q8_kernel<0><<<(unsigned)ntiles, kTileThreads, 0, stream>>>(W, ldw, TC, tiles);
  else pack_q8_kernel<1><<<(unsigned)ntiles, kTileThreads, 0, stream>>>(W, ldw, TC, tiles);
  return cudaGetLastError();
}

// f16 weights [N][K], unit chunk scales [N][nb], then the f16 activation
// rows and their scales, each padded to 256 bytes.
size_t q8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const size_t w16 = (size_t)N * K * 2;
  const size_t ones = (size_t)N * ((K + kPairChunkK - 1) / kPairChunkK) * 4;
  return (w16 + 255) / 256 * 256 + (ones + 255) / 256 * 256 + act_f16_bytes(M, K);
}

cudaError_t launch_q8_gemm(const uint8_t* tiles, int layout, int N, int K, const __nv_bfloat16* X, int64_t ldx,
                           int M, float* Y, int64_t ldy, void* workspace, int32_t* dev_status, cudaStream_t stream) {
  const int TR = N / (int)kTileRows, TC = K / (int)kTileCols;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (M <= kQ8GemvMaxM) {
    // slabs of 16 rows; more warps per slab while fewer than ~16 warps per SM
    const int units = 2 * TR;
    int wpu = 1;
    while (wpu < kQ8GvWarps && wpu < TC && (int64_t)units * wpu < (int64_t)16 * sms) wpu *= 2;
    if (M <= 1) return q8_gemv_launch<1>(layout, units, sms, tiles, TR, TC, X, ldx, Y, ldy, M, wpu, stream);
    if (M <= 2) return q8_gemv_launch<2>(layout, units, sms, tiles, TR, TC, X, ldx, Y, ldy, M, wpu, stream);
    if (M <= 4) return q8_gemv_launch<4>(layout, units, sms, tiles, TR, TC, X, ldx, Y, ldy, M, wpu, stream);
    if (M <= 8) return q8_gemv_launch<8>(layout, units, sms, tiles, TR, TC, X, ldx, Y, ldy, M, wpu, stream);
    return q8_gemv_launch<16>(layout, units, sms, tiles, TR, TC, X, ldx, Y, ldy, M, wpu, stream);
  }
  char* ws = static_cast<char*>(workspace);
  __half* W16 = reinterpret_cast<__half*>(ws);
  const size_t ones_off = ((size_t)N * K * 2 + 255) / 256 * 256;
  const int nb = (K + kPairChunkK - 1) / kPairChunkK;
  float* ones = reinterpret_cast<float*>(ws + ones_off);
  char* act = ws + ones_off + ((size_t)N * nb * 4 + 255) / 256 * 256;
  const int64_t ntiles = (int64_t)TR * TC;
  if (layout == 0)
    q8_decode_f16_kernel<0><<<(unsigned)ntiles, kTileThreads, 0, stream>>>(tiles, TC, K, W16, ones, nb, dev_status);
  else
    q8_decode_f16_kernel<1><<<(unsigned)ntiles, kTileThreads, 0, stream>>>(tiles, TC, K, W16, ones, nb, dev_status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if ((err = launch_act_to_f16(X, ldx, M, K, act, stream)) != cudaSuccess) return err;
  return launch_w16_gemm_umma(W16, true, ones, nb, N, K, act, K,
                              reinterpret_cast<const float*>(act + act_f16_scale_offset(M, K)), M, Y, ldy,
                              dev_status, stream);
}

}  // namespace qmm
