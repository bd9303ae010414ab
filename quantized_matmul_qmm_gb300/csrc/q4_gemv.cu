// Decode GEMV for one activation row (M = 1), the weight-streaming case.
//
// At decode sizes the q4 path is bound by the weight stream ("Zaya 8B Q4NX on
// the AMD NPU", round 25q: the access pattern, not the fabric, set the
// decode wall).  Weights stay packed as 32x256 q4_1 tiles ("NPU engine: full
// ELFs, no xclbin", "Q4NX chunks") and are read once, 16 bytes per load.
//
// Blocks as MMA columns.  For one output row r and one 32-column block b, the
// factored form needs
//     P[r][b] = sum_{e<32} (128 + q[r][b][e]) * x[b][e]
// and then y[r] += s[r][b] * P[r][b] + (min[r][b] - 128 s[r][b]) * sum_e x[b][e].
// One mma.sync m16n8k16 (bf16, fp32 accumulate) covers 16 rows and 8
// columns.  Here the 8 columns are the 8 blocks of a tile, not 8 activation
// rows.  Logical k = 2t'+u belongs to block t' and k = 2t'+8+u to block
// t'+4 (u = 0,1); MMA i takes elements 2i+u.  The B operand holds x[b][.] in
// column b and zeros elsewhere, so after 16 MMAs
// D[r][b] = P[r][b] for 16 rows x 8 blocks.  Every MMA column is useful, and
// each thread then applies the scale and min of exactly its own (row, block)
// pairs.
//
// Thread (g, t) of a warp works on rows g and g+8 of a 16-row slab.  It
// reads blocks t and t+4 of those rows (two 16-byte loads per row) and the
// (scale, min) pairs of blocks 2t and 2t+1 (its D columns).  Lanes with
// (g & 3) == t supply x of block g.
//
// Weight stream.  A tile row (32 outputs, all of K) is TC = K/256 contiguous
// tiles.  One producer thread copies whole tile rows into a ring in shared
// memory with bulk asynchronous copies (one TMA request of TC * 5120 bytes per
// row: TMA pays a fixed cost per request, so requests are made large).  Two
// consumer warps share each row (one 16-row slab each), four rows at a time.  Loads kept in registers
// (q4_gemv1_regs_kernel) remain for tile rows too long for a useful ring.
#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kWarps = 8;
constexpr int kPF = 3;                // tiles prefetched per warp (in registers)
constexpr int kCtasPerSm = 2;

struct Gemv1Params {
  const uint8_t* tiles;
  int N, K;
  const __nv_bfloat16* X;
  float* Y;
  int S;                              // warps sharing one slab (K split)
};

struct G1Tile {
  uint4 c[2][2];                      // [row g / g+8][block t / t+4]: 4 code words each
  uint2 p[2];                         // [row]: (scale, min) of blocks 2t, 2t+1
};

QMM_DEV uint2 ldg64(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// Fragment data of thread (g, t) straight from the tile in global memory:
// blocks t and t+4 of rows r0 and r0+8 (16 bytes each) and the pairs of
// blocks 2t, 2t+1, with plain 128-bit loads kept out of L1 (the path for tile
// rows too long for the streaming kernel's ring).
QMM_DEV void g1_load(G1Tile& d, const uint8_t* tile, int r0, int t) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint8_t* row = tile + (r0 + 8 * h) * 128;
    d.c[h][0] = ldg128_stream(row + 16 * t);
    d.c[h][1] = ldg128_stream(row + 16 * (t + 4));
    d.p[h] = ldg64(tile + 4096 + (r0 + 8 * h) * 32 + 8 * t);
  }
}

// One tile: 16 MMAs in four independent accumulator chains, then the scales
// of this thread's (row, block) pairs.  xsrc points at x of block g for the
// lanes that carry it and at a zero block otherwise (same for xsrc_hi).
QMM_DEV void g1_tile(const G1Tile& d, const __nv_bfloat16* xlo, const __nv_bfloat16* xhi, const float* xsum_tc,
                     int t, float& y0, float& y1) {
  uint32_t xa[16], xb[16];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 wa = reinterpret_cast<const uint4*>(xlo)[v];
    const uint4 wb = reinterpret_cast<const uint4*>(xhi)[v];
    xa[4 * v + 0] = wa.x; xa[4 * v + 1] = wa.y; xa[4 * v + 2] = wa.z; xa[4 * v + 3] = wa.w;
    xb[4 * v + 0] = wb.x; xb[4 * v + 1] = wb.y; xb[4 * v + 2] = wb.z; xb[4 * v + 3] = wb.w;
  }
  float acc[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int w = i >> 2, pi = i & 3;
    const uint32_t a0 = q4_pair_biased(u4_get(d.c[0][0], w), pi);   // row g,   block t
    const uint32_t a1 = q4_pair_biased(u4_get(d.c[1][0], w), pi);   // row g+8, block t
    const uint32_t a2 = q4_pair_biased(u4_get(d.c[0][1], w), pi);   // row g,   block t+4
    const uint32_t a3 = q4_pair_biased(u4_get(d.c[1][1], w), pi);   // row g+8, block t+4
    mma_bf16_16816(acc[i & 3], a0, a1, a2, a3, xa[i], xb[i]);
  }
  float r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) r[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
  // r: (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
  const float2 xsv = *reinterpret_cast<const float2*>(xsum_tc + 2 * t);
  const float s00 = bf16lo_to_f32(d.p[0].x), s01 = bf16lo_to_f32(d.p[0].y);
  const float s10 = bf16lo_to_f32(d.p[1].x), s11 = bf16lo_to_f32(d.p[1].y);
  y0 = fmaf(s00, r[0], fmaf(fmaf(-128.0f, s00, bf16hi_to_f32(d.p[0].x)), xsv.x, y0));
  y0 = fmaf(s01, r[1], fmaf(fmaf(-128.0f, s01, bf16hi_to_f32(d.p[0].y)), xsv.y, y0));
  y1 = fmaf(s10, r[2], fmaf(fmaf(-128.0f, s10, bf16hi_to_f32(d.p[1].x)), xsv.x, y1));
  y1 = fmaf(s11, r[3], fmaf(fmaf(-128.0f, s11, bf16hi_to_f32(d.p[1].y)), xsv.y, y1));
}

// Item cursor of one warp: (group iteration, position inside the group),
// advanced by increments so the hot loop does no division.
struct G1Cursor {
  int gi;       // group iteration (group = blockIdx.x + gi * gridDim.x)
  int pos;      // item inside the group: tile column tc = ks + pos * S
};

// Persistent: CTA b takes slab groups b, b + gridDim.x, ...  A group is
// kWarps / S slabs; the S warps of a slab split its tiles (tc = ks, ks + S,
// ...), and their partial sums are added in a fixed order through shared
// memory.  Each warp walks its (group, tile) items as one flat sequence, so
// the prefetch runs across group boundaries.
__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm) q4_gemv1_regs_kernel(const Gemv1Params p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int TC = p.K / 256;
  __nv_bfloat16* xs_sm = reinterpret_cast<__nv_bfloat16*>(sm);                 // [K] + 32 zeros
  float* xsum = reinterpret_cast<float*>(sm + (size_t)p.K * 2 + 64);           // [K/32]
  float* red = xsum + p.K / 32;                                                // [kWarps][32][2]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  umma::pdl_launch_dependents();
  umma::pdl_wait();
  for (int i = threadIdx.x; i < p.K / 8; i += blockDim.x)
    reinterpret_cast<uint4*>(xs_sm)[i] = reinterpret_cast<const uint4*>(p.X)[i];
  if (threadIdx.x < 4) reinterpret_cast<uint4*>(xs_sm + p.K)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  for (int b = threadIdx.x; b < p.K / 32; b += blockDim.x) {
    const uint4* xp = reinterpret_cast<const uint4*>(xs_sm + 32 * b);
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 w = xp[v];
      s += bf16lo_to_f32(w.x) + bf16hi_to_f32(w.x) + bf16lo_to_f32(w.y) + bf16hi_to_f32(w.y) +
           bf16lo_to_f32(w.z) + bf16hi_to_f32(w.z) + bf16lo_to_f32(w.w) + bf16hi_to_f32(w.w);
    }
    xsum[b] = s;
  }
  __syncthreads();

  const int S = p.S;
  const int slabs_per_group = kWarps / S;
  const int nslabs = p.N / 16;
  const int ngroups = (nslabs + slabs_per_group - 1) / slabs_per_group;
  const int my_groups = (int)blockIdx.x < ngroups ? (ngroups - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int ks = warp % S;
  const int per_warp = (TC - ks + S - 1) / S;        // tiles of one slab handled by this warp
  const int per_slot = (TC + S - 1) / S;             // items per group (uniform across warps)
  const int nitems = my_groups * per_slot;
  const int slab0 = (int)blockIdx.x * slabs_per_group + warp / S;
  const int slab_step = (int)gridDim.x * slabs_per_group;
  // x source of this lane: block g of each tile if it carries x, else the zero block
  const bool lo = (g == t), hi = (g == t + 4);
  const __nv_bfloat16* zero = xs_sm + p.K;

  G1Cursor ld{0, 0}, cu{0, 0};
  auto load_next = [&](G1Tile& dst) {
    if (ld.gi < my_groups) {
      const int slab = slab0 + ld.gi * slab_step;
      if (ld.pos < per_warp && slab < nslabs)
        g1_load(dst, p.tiles + ((int64_t)(slab >> 1) * TC + ks + ld.pos * S) * kTileBytes, ((slab & 1) << 4) + g,
                t);
    }
    if (++ld.pos == per_slot) { ld.pos = 0; ++ld.gi; }
  };

  G1Tile ring[kPF];
#pragma unroll
  for (int i = 0; i < kPF; ++i) load_next(ring[i]);
  float y0 = 0.f, y1 = 0.f;
  for (int j0 = 0; j0 < nitems; j0 += kPF) {
#pragma unroll
    for (int i = 0; i < kPF; ++i) {
      if (j0 + i < nitems) {
        const int slab = slab0 + cu.gi * slab_step;
        if (cu.pos < per_warp && slab < nslabs) {
          const int tc = ks + cu.pos * S;
          const __nv_bfloat16* xt = xs_sm + tc * 256 + 32 * g;
          g1_tile(ring[i], lo ? xt : zero, hi ? xt : zero, xsum + tc * 8, t, y0, y1);
        }
        load_next(ring[i]);
        if (++cu.pos == per_slot) {
          // end of this group: sum over the quad, then over the S warps of the slab
          y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
          y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
          y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
          y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
          if (S == 1) {
            if (t == 0 && slab < nslabs) {
              p.Y[slab * 16 + g] = y0;
              p.Y[slab * 16 + g + 8] = y1;
            }
          } else {
            red[(warp * 32 + lane) * 2 + 0] = y0;
            red[(warp * 32 + lane) * 2 + 1] = y1;
            __syncthreads();
            if (ks == 0 && t == 0 && slab < nslabs) {
              float a = 0.f, b = 0.f;
              for (int w = 0; w < S; ++w) {
                a += red[((warp + w) * 32 + lane) * 2 + 0];
                b += red[((warp + w) * 32 + lane) * 2 + 1];
              }
              p.Y[slab * 16 + g] = a;
              p.Y[slab * 16 + g + 8] = b;
            }
            __syncthreads();
          }
          y0 = 0.f;
          y1 = 0.f;
          cu.pos = 0;
          ++cu.gi;
        }
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Streaming M = 1 GEMV: bulk copies of whole tile rows into a shared ring.
// ---------------------------------------------------------------------------
constexpr int kSWarps = 8;                       // consumer warps, in pairs
constexpr int kSThreads = 32 * (kSWarps + 1);    // + the producer warp
constexpr size_t kRingBudget = 192 * 1024;
constexpr int kMaxSlots = 16;
constexpr int kPrefetchRows = 2;                 // rows warmed in L2 before the dependency wait

struct Gemv1SParams {
  const uint8_t* tiles;
  int N, K;
  const __nv_bfloat16* X;
  float* Y;
  int slots;                                     // ring slots of one tile row each
  int32_t* dev_status;
};

// Fragment data of thread (g, t) from a tile held in shared memory.
QMM_DEV void g1_lds(G1Tile& d, uint32_t tile, int r0, int t) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t row = tile + (uint32_t)((r0 + 8 * h) * 128);
    d.c[h][0] = umma::lds128(row + 16 * t);
    d.c[h][1] = umma::lds128(row + 16 * (t + 4));
    uint2 pv;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                 : "=r"(pv.x), "=r"(pv.y)
                 : "r"(tile + 4096u + (uint32_t)((r0 + 8 * h) * 32 + 8 * t)));
    d.p[h] = pv;
  }
}


__global__ void __launch_bounds__(kSThreads, 1) q4_gemv1_kernel(const Gemv1SParams p) {
  using namespace umma;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = smem_align(sm_raw, 128);
  const int TC = p.K / 256;
  const uint32_t row_bytes = (uint32_t)TC * (uint32_t)kTileBytes;
  uint8_t* ring = sm;                                                           // [slots][row_bytes]
  __nv_bfloat16* xs_sm = reinterpret_cast<__nv_bfloat16*>(ring + (size_t)p.slots * row_bytes);  // [K] + 32 zeros
  float* xsum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs_sm) + (size_t)p.K * 2 + 64);
  uint64_t* full = reinterpret_cast<uint64_t*>(xsum + p.K / 32 + 2);         // [slots]
  uint64_t* empty = full + kMaxSlots;                                         // [slots]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxSlots);
  float* red = reinterpret_cast<float*>(empty + kMaxSlots + 2);               // [pair][slab][g][2]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nrows = p.N / 32;                                                 // tile rows
  const int my_rows = (int)blockIdx.x < nrows ? (nrows - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);   // the two warps of a pair
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kSWarps) {
    // ---- producer: tile rows blockIdx.x, blockIdx.x + gridDim.x, ... ----
    if (lane == 0) {
      // While the previous grid finishes, pull the first two rows into L2.
      // L2 is where global memory is coherent, so a line warmed here and
      // written later by that grid is still read correctly: the copies into
      // shared memory are only issued after the wait below.  (More rows delay
      // the first copy: this SM's TMA unit works through the prefetch
      // requests first.)
      for (int j = 0; j < my_rows && j < kPrefetchRows; ++j)
        bulk_prefetch_l2(p.tiles + (int64_t)((int)blockIdx.x + j * (int)gridDim.x) * row_bytes, row_bytes);
      pdl_wait();
      for (int j = 0; j < my_rows; ++j) {
        const int s = j % p.slots;
        if (!mbar_wait(&empty[s], ((j / p.slots) & 1) ^ 1, abort_flag, p.dev_status)) break;
        const int tr = (int)blockIdx.x + j * (int)gridDim.x;
        mbar_arrive_expect_tx(&full[s], row_bytes);
        umma::bulk_g2s(smem_u32(ring + (size_t)s * row_bytes), p.tiles + (int64_t)tr * row_bytes, row_bytes, &full[s]);
      }
    }
    // the copies in flight land before the CTA exits: consumers wait for every row
    return;
  }

  // ---- consumers: x into shared memory, then rows j = warp, warp + 8, ... ----
  pdl_wait();   // x and y may belong to the previous grid
  for (int i = threadIdx.x; i < p.K / 8; i += kSWarps * 32)
    reinterpret_cast<uint4*>(xs_sm)[i] = reinterpret_cast<const uint4*>(p.X)[i];
  if (threadIdx.x < 4) reinterpret_cast<uint4*>(xs_sm + p.K)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("bar.sync 1, %0;" ::"n"(kSWarps * 32) : "memory");
  for (int b = threadIdx.x; b < p.K / 32; b += kSWarps * 32) {
    const uint4* xp = reinterpret_cast<const uint4*>(xs_sm + 32 * b);
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 w = xp[v];
      s += bf16lo_to_f32(w.x) + bf16hi_to_f32(w.x) + bf16lo_to_f32(w.y) + bf16hi_to_f32(w.y) +
           bf16lo_to_f32(w.z) + bf16hi_to_f32(w.z) + bf16lo_to_f32(w.w) + bf16hi_to_f32(w.w);
    }
    xsum[b] = s;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kSWarps * 32) : "memory");

  // A pair of warps takes each tile row, one 16-row slab each (its outputs are
  // its own); pair q takes rows q, q + P, ... with P = min(4, slots) active
  // pairs.  The launcher makes the slot count a multiple of P, so the rows
  // that share a slot (j, j + slots, ...) all belong to one pair and are
  // consumed in order: a pair never waits on a slot's phase before the
  // previous phase of that slot has completed, and the slot is free once both
  // warps of the pair have arrived on its empty barrier.
  const bool lo = (g == t), hi = (g == t + 4);
  const __nv_bfloat16* zero = xs_sm + p.K;
  const int pair = warp >> 1, slab = warp & 1;
  const int npairs = min(kSWarps / 2, p.slots);
  if (nrows <= (int)gridDim.x) {
    // One tile row per CTA (small N): all four pairs split the row's tiles
    // (tc = pair, pair + 4, ...; one row uses no slot twice) so that no pair
    // walks all of K alone, and their partial sums are added in pair order
    // through shared memory.
    constexpr int kSplit = kSWarps / 2;
    float y0 = 0.f, y1 = 0.f;
    if (my_rows == 1 &&
        __all_sync(0xffffffffu, mbar_wait(&full[0], 0, abort_flag, p.dev_status))) {
      const uint32_t rowbase = smem_u32(ring);
      for (int tc = pair; tc < TC; tc += kSplit) {
        G1Tile d;
        g1_lds(d, rowbase + (uint32_t)tc * kTileBytes, 16 * slab + g, t);
        const __nv_bfloat16* xt = xs_sm + tc * 256 + 32 * g;
        g1_tile(d, lo ? xt : zero, hi ? xt : zero, xsum + tc * 8, t, y0, y1);
      }
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t == 0) {
      red[((pair * 2 + slab) * 8 + g) * 2] = y0;
      red[((pair * 2 + slab) * 8 + g) * 2 + 1] = y1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kSWarps * 32) : "memory");
    if (pair == 0 && t == 0 && my_rows == 1 && !*abort_flag) {
      float s0 = 0.f, s1 = 0.f;
      for (int q = 0; q < kSplit; ++q) {
        s0 += red[((q * 2 + slab) * 8 + g) * 2];
        s1 += red[((q * 2 + slab) * 8 + g) * 2 + 1];
      }
      p.Y[(int)blockIdx.x * 32 + 16 * slab + g] = s0;
      p.Y[(int)blockIdx.x * 32 + 16 * slab + g + 8] = s1;
    }
  }
  for (int j = (pair < npairs && nrows > (int)gridDim.x) ? pair : my_rows; j < my_rows; j += npairs) {
    const int s = j % p.slots;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / p.slots) & 1, abort_flag, p.dev_status))) break;
    const uint32_t rowbase = smem_u32(ring + (size_t)s * row_bytes);
    // two tiles per iteration, independent until the final add (more ILP)
    float y0 = 0.f, y1 = 0.f, z0 = 0.f, z1 = 0.f;
    int tc = 0;
    for (; tc + 1 < TC; tc += 2) {
      G1Tile d, e;
      g1_lds(d, rowbase + (uint32_t)tc * kTileBytes, 16 * slab + g, t);
      g1_lds(e, rowbase + (uint32_t)(tc + 1) * kTileBytes, 16 * slab + g, t);
      const __nv_bfloat16* xt = xs_sm + tc * 256 + 32 * g;
      const __nv_bfloat16* xu = xt + 256;
      g1_tile(d, lo ? xt : zero, hi ? xt : zero, xsum + tc * 8, t, y0, y1);
      g1_tile(e, lo ? xu : zero, hi ? xu : zero, xsum + tc * 8 + 8, t, z0, z1);
    }
    if (tc < TC) {
      G1Tile d;
      g1_lds(d, rowbase + (uint32_t)tc * kTileBytes, 16 * slab + g, t);
      const __nv_bfloat16* xt = xs_sm + tc * 256 + 32 * g;
      g1_tile(d, lo ? xt : zero, hi ? xt : zero, xsum + tc * 8, t, y0, y1);
    }
    y0 += z0;
    y1 += z1;
    // every lane's shared-memory reads of this slot went into y0, y1
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t == 0) {
      const int tr = (int)blockIdx.x + j * (int)gridDim.x;
      p.Y[tr * 32 + 16 * slab + g] = y0;
      p.Y[tr * 32 + 16 * slab + g + 8] = y1;
    }
  }
  if (*abort_flag && threadIdx.x == 0) {
    // rows nobody consumed may still be landing: let them land first
    for (int j = 0; j < my_rows; ++j)
      mbar_wait(&full[j % p.slots], (j / p.slots) & 1, abort_flag, nullptr, 50000000ull) ||
          mbar_try_wait(&full[j % p.slots], (j / p.slots) & 1);
  }
}


// ---------------------------------------------------------------------------
// Grouped M = 1 GEMV: the tile rows of several weight sets in one launch.
//
// The host balances whole tile rows over the CTAs by bytes (longest first,
// each to the least loaded CTA) and passes every CTA its list of
// (problem, tile row) entries in the launch parameters.  Before the
// dependency wait a CTA builds its item table (entry, 16-row slab, tile
// column) in shared memory and warms its rows in L2, so in a chain of
// launches the next group's weights stream from HBM while this one computes.
// After the wait one thread bulk-copies every row of the CTA and the x of
// each of its problems into shared memory (all requests in flight at once,
// one barrier per row), and the warps walk the items round-robin as their
// rows land.  Item results go to shared memory and each output is summed
// over its tile columns in column order, so the result does not depend on
// which warp took which item.
// ---------------------------------------------------------------------------
constexpr int kGWarps = 16;
constexpr int kGThreads = kGWarps * 32;
constexpr int kMaxGroupCtas = 256;
constexpr size_t kGroupSmemBudget = 110 * 1024;   // two CTAs per SM: this launch and the next

template <int kEntries>
struct GroupParams {
  GemvGroupProblem prob[kMaxGroupProblems];
  int32_t* dev_status;
  int32_t cta_begin[kMaxGroupCtas + 1];   // entries of CTA c: [cta_begin[c], cta_begin[c+1])
  uint32_t entry[kEntries];               // (problem << 24) | tile row, sorted within a CTA
};

struct GEnt {            // one tile row of one problem
  float* y;              // its 32 outputs
  int32_t ibase;         // first item
  int32_t tc;            // tile columns
};
struct GItem {           // one 16-row slab of one tile
  uint32_t tile;         // shared address of the tile
  uint32_t xo;           // x element offset of the tile's 256 columns
  uint32_t eh;           // entry << 1 | slab
  uint32_t xbar;         // barrier of the tile's x
};
struct GCopy {           // one bulk copy into shared memory
  uint64_t src;
  uint32_t dst, bytes;
};

// One tile slab with x held in registers: xv is block g of x for the lanes
// that carry it (g == t: the block goes to MMA columns 0..3, g == t + 4: to
// columns 4..7), xs2 the x sums of the two blocks of this lane's D columns.
QMM_DEV void g1_tile_rx(const G1Tile& d, const uint4 (&xv)[4], bool lo, bool hi, float2 xs2, int t, float& y0,
                        float& y1) {
  uint32_t xa[16], xb[16];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t w[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xa[4 * v + j] = lo ? w[j] : 0u;
      xb[4 * v + j] = hi ? w[j] : 0u;
    }
  }
  float acc[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int w = i >> 2, pi = i & 3;
    const uint32_t a0 = q4_pair_biased(u4_get(d.c[0][0], w), pi);
    const uint32_t a1 = q4_pair_biased(u4_get(d.c[1][0], w), pi);
    const uint32_t a2 = q4_pair_biased(u4_get(d.c[0][1], w), pi);
    const uint32_t a3 = q4_pair_biased(u4_get(d.c[1][1], w), pi);
    mma_bf16_16816(acc[i & 3], a0, a1, a2, a3, xa[i], xb[i]);
  }
  float r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) r[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
  const float s00 = bf16lo_to_f32(d.p[0].x), s01 = bf16lo_to_f32(d.p[0].y);
  const float s10 = bf16lo_to_f32(d.p[1].x), s11 = bf16lo_to_f32(d.p[1].y);
  y0 = fmaf(s00, r[0], fmaf(fmaf(-128.0f, s00, bf16hi_to_f32(d.p[0].x)), xs2.x, y0));
  y0 = fmaf(s01, r[1], fmaf(fmaf(-128.0f, s01, bf16hi_to_f32(d.p[0].y)), xs2.y, y0));
  y1 = fmaf(s10, r[2], fmaf(fmaf(-128.0f, s10, bf16hi_to_f32(d.p[1].x)), xs2.x, y1));
  y1 = fmaf(s11, r[3], fmaf(fmaf(-128.0f, s11, bf16hi_to_f32(d.p[1].y)), xs2.y, y1));
}

template <int kEntries>
__global__ void __launch_bounds__(kGThreads, 2) q4_gemv_group_kernel(const __grid_constant__ GroupParams<kEntries> p) {
  using namespace umma;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = smem_align(sm_raw, 128);
  const int e0 = p.cta_begin[blockIdx.x], e1 = p.cta_begin[blockIdx.x + 1];
  const int ne = e1 - e0;
  // layout (the host's size formula follows it): header, x offsets, barriers
  // (rows, then the x of each problem), copies, entries, items, x behind a
  // zero block, the rows, item results
  int32_t* hdr = reinterpret_cast<int32_t*>(sm);                              // [0] items, [1] x elems, [2] row bytes, [3] problems
  int32_t* xoff = hdr + 4;                                                    // [kMaxGroupProblems] x offset, [.. + 32] x barrier
  uint64_t* bars = reinterpret_cast<uint64_t*>(xoff + 2 * kMaxGroupProblems); // [ne + kMaxGroupProblems]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + ne + kMaxGroupProblems);
  GCopy* copies = reinterpret_cast<GCopy*>(bars + ne + kMaxGroupProblems + 2); // [ne + kMaxGroupProblems]
  GEnt* ents = reinterpret_cast<GEnt*>(copies + ne + kMaxGroupProblems);     // [ne]
  GItem* items = reinterpret_cast<GItem*>(ents + ne);                         // [nitems]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  pdl_launch_dependents();
  // ---- before the wait: only the launch parameters are read ----
  // Warm this CTA's rows in L2.  L2 is where global memory is coherent, so a
  // row that the previous grid writes is still read correctly: the copies
  // into shared memory come after the wait.
  for (int e = (int)threadIdx.x; e < ne; e += kGThreads) {
    const uint32_t en = p.entry[e0 + e];
    const GemvGroupProblem& pr = p.prob[en >> 24];
    const uint32_t row_bytes = (uint32_t)(pr.K / 256) * (uint32_t)kTileBytes;
    bulk_prefetch_l2(pr.tiles + (int64_t)(en & 0xFFFFFFu) * row_bytes, row_bytes);
  }
  if (threadIdx.x == 0) {
    int it = 0, nd = 0, xo = 32, last = -1, rb = 0;
    for (int e = 0; e < ne; ++e) {
      const uint32_t en = p.entry[e0 + e];
      const int pi = (int)(en >> 24);
      const int tc = p.prob[pi].K / 256;
      if (pi != last) {
        xoff[pi] = xo;
        xoff[kMaxGroupProblems + pi] = ne + nd;
        copies[ne + nd] = {reinterpret_cast<uint64_t>(p.prob[pi].X), (uint32_t)xo * 2u, (uint32_t)p.prob[pi].K * 2u};
        mbar_init(&bars[ne + nd], 1);
        ++nd;
        xo += p.prob[pi].K;
        last = pi;
      }
      ents[e].y = p.prob[pi].Y + (int64_t)(en & 0xFFFFFFu) * 32;
      ents[e].ibase = it;
      ents[e].tc = tc;
      it += 2 * tc;
      const uint32_t row_bytes = (uint32_t)tc * (uint32_t)kTileBytes;
      copies[e] = {reinterpret_cast<uint64_t>(p.prob[pi].tiles + (int64_t)(en & 0xFFFFFFu) * row_bytes), (uint32_t)rb,
                   row_bytes};
      mbar_init(&bars[e], 1);
      rb += (int)row_bytes;
    }
    hdr[0] = it;
    hdr[1] = xo;
    hdr[2] = rb;
    hdr[3] = nd;
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int nitems = hdr[0], xelems = hdr[1], ncopies = ne + hdr[3];
  uint8_t* xraw = reinterpret_cast<uint8_t*>(items + nitems);
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(xraw + ((16 - (smem_u32(xraw) & 15)) & 15));   // 32 zeros, then x's
  uint8_t* rows = reinterpret_cast<uint8_t*>(xs + xelems);                     // the CTA's rows (16-byte aligned)
  float* part = reinterpret_cast<float*>(rows + hdr[2]);                       // [nitems][16]
  if ((int)threadIdx.x < ne) {
    const int e = (int)threadIdx.x;   // the host keeps ne <= kGThreads
    const int pi = (int)(p.entry[e0 + e] >> 24);
    const int tc = ents[e].tc;
    const uint32_t row = smem_u32(rows) + copies[e].dst;
    GItem* it = items + ents[e].ibase;
    for (int h = 0; h < 2; ++h)
      for (int c = 0; c < tc; ++c)
        it[h * tc + c] = {row + (uint32_t)c * (uint32_t)kTileBytes, (uint32_t)(xoff[pi] + 256 * c),
                          (uint32_t)(e << 1 | h), (uint32_t)xoff[kMaxGroupProblems + pi]};
  }
  if (threadIdx.x < 4) reinterpret_cast<uint4*>(xs)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();

  // ---- after the wait: tiles, x and y may belong to the previous grid ----
  pdl_wait();
  if (warp == 0) {
    // every copy of the CTA in flight at once, issued by the lanes of one warp
    const uint32_t xbase = smem_u32(xs), rbase = smem_u32(rows);
    for (int c = lane; c < ncopies; c += 32) {
      const GCopy cp = copies[c];
      mbar_arrive_expect_tx(&bars[c], cp.bytes);
      bulk_g2s((c < ne ? rbase : xbase) + cp.dst, reinterpret_cast<const void*>(cp.src), cp.bytes, &bars[c]);
    }
  }

  const bool lo = (g == t), hi = (g == t + 4);
  const bool owner = lo || hi;
  // lanes 5b (b < 4) and 5b - 4 (b >= 4) carry block b of x
  const int src0 = 2 * t < 4 ? 10 * t : 10 * t - 4, src1 = 2 * t + 1 < 4 ? 10 * t + 5 : 10 * t + 1;
  for (int it = warp; it < nitems; it += kGWarps) {
    const GItem im = items[it];
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[im.xbar], 0, abort_flag, p.dev_status) &&
                                     mbar_wait(&bars[im.eh >> 1], 0, abort_flag, p.dev_status)))
      break;
    G1Tile d;
    g1_lds(d, im.tile, 16 * (int)(im.eh & 1) + g, t);
    uint4 xv[4];
    const uint32_t xa = smem_u32(xs + (owner ? im.xo + 32 * g : 0u));
#pragma unroll
    for (int v = 0; v < 4; ++v) xv[v] = lds128(xa + 16u * v);
    float own = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v)
      own += (bf16lo_to_f32(xv[v].x) + bf16hi_to_f32(xv[v].x)) + (bf16lo_to_f32(xv[v].y) + bf16hi_to_f32(xv[v].y)) +
             (bf16lo_to_f32(xv[v].z) + bf16hi_to_f32(xv[v].z)) + (bf16lo_to_f32(xv[v].w) + bf16hi_to_f32(xv[v].w));
    const float2 xs2 = make_float2(__shfl_sync(0xffffffffu, own, src0), __shfl_sync(0xffffffffu, own, src1));
    float y0 = 0.f, y1 = 0.f;
    g1_tile_rx(d, xv, lo, hi, xs2, t, y0, y1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t == 0) {
      part[it * 16 + g] = y0;
      part[it * 16 + g + 8] = y1;
    }
  }
  __syncthreads();
  if (*abort_flag) {
    // copies nobody waited for may still be landing: let them land first
    if (threadIdx.x == 0)
      for (int c = 0; c < ncopies; ++c)
        mbar_drain(&bars[c], 0);
    return;
  }
  // each output: its slab's items summed in tile-column order
  for (int o = threadIdx.x; o < ne * 32; o += kGThreads) {
    const int le = o >> 5, r = o & 31, h = r >> 4, i = r & 15;
    const GEnt en = ents[le];
    const float* pp = part + (en.ibase + h * en.tc) * 16 + i;
    float s = 0.f;
    for (int c = 0; c < en.tc; ++c) s += pp[c * 16];
    en.y[r] = s;
  }
}

}  // namespace

cudaError_t launch_q4_gemv1(const Q4DenseArgs& a, int sms, int32_t* dev_status, cudaStream_t stream) {
  const int TC = a.K / 256;
  const size_t row_bytes = (size_t)TC * kTileBytes;
  int slots = (int)(kRingBudget / row_bytes);
  if (slots > kMaxSlots) slots = kMaxSlots;
  // a multiple of the active consumer pairs (see the kernel's row loop)
  if (slots >= kSWarps / 2) slots -= slots % (kSWarps / 2);
  if (slots >= 3) {
    Gemv1SParams p{};
    p.tiles = a.tiles;
    p.N = a.N;
    p.K = a.K;
    p.X = a.X;
    p.Y = a.Y;
    p.slots = slots;
    p.dev_status = dev_status;
    const int nrows = a.N / 32;
    const int grid = nrows < sms ? nrows : sms;
    const size_t smem = 128 + (size_t)slots * row_bytes + (size_t)a.K * 2 + 64 + (size_t)(a.K / 32) * 4 +
                        (size_t)(kSWarps * 32 + 2) * 4 + 2 * kMaxSlots * 8 + 16 + (size_t)(kSWarps / 2) * 2 * 8 * 2 * 4;
    const cudaError_t e = cudaFuncSetAttribute(q4_gemv1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(q4_gemv1_kernel, dim3(grid), dim3(kSThreads), smem, stream, p);
  }
  Gemv1Params p{};
  p.tiles = a.tiles;
  p.N = a.N;
  p.K = a.K;
  p.X = a.X;
  p.Y = a.Y;
  const int nslabs = a.N / 16;
  // split K across warps while there are too few slab groups to fill the GPU
  int S = 1;
  while (S < kWarps && S * 2 <= TC && (nslabs * S) / kWarps < 4 * sms) S *= 2;
  p.S = S;
  const int groups = (nslabs + kWarps / S - 1) / (kWarps / S);
  const int grid = groups < kCtasPerSm * sms ? groups : kCtasPerSm * sms;
  const size_t smem = (size_t)a.K * 2 + 64 + (size_t)(a.K / 32) * 4 + (size_t)kWarps * 32 * 2 * 4;
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(q4_gemv1_regs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(q4_gemv1_regs_kernel, dim3(grid), dim3(kWarps * 32), smem, stream, p);
}


namespace {

// Balanced assignment of tile rows to CTAs, cached by the group's shapes
// (the pointers change from call to call, the plan does not).
struct GroupPlan {
  std::vector<int> key;                 // grid, then (N, K) per problem
  std::vector<int32_t> cta_begin;       // [grid + 1]
  std::vector<uint32_t> entry;          // (problem << 24) | tile row
  size_t smem = 0;
};

void build_group_plan(const GemvGroupProblem* probs, int n, int grid, GroupPlan& plan) {
  struct Row { int64_t bytes; int pi, tr; };
  std::vector<Row> rows;
  for (int pi = 0; pi < n; ++pi)
    for (int tr = 0; tr < probs[pi].N / 32; ++tr) rows.push_back({(int64_t)(probs[pi].K / 256) * kTileBytes, pi, tr});
  // longest first (stable, so rows of equal size keep problem and row order)
  std::stable_sort(rows.begin(), rows.end(), [](const Row& a, const Row& b) { return a.bytes > b.bytes; });
  using Load = std::pair<int64_t, int>;   // (bytes so far, cta): the least loaded, then the lowest index
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0, c});
  std::vector<std::vector<uint32_t>> per(grid);
  for (const Row& r : rows) {
    Load l = heap.top();
    heap.pop();
    per[l.second].push_back(((uint32_t)r.pi << 24) | (uint32_t)r.tr);
    l.first += r.bytes;
    heap.push(l);
  }
  plan.cta_begin.assign(grid + 1, 0);
  plan.entry.clear();
  plan.smem = 0;
  for (int c = 0; c < grid; ++c) {
    std::sort(per[c].begin(), per[c].end());
    plan.cta_begin[c] = (int32_t)plan.entry.size();
    const int ne = (int)per[c].size();
    int items = 0, last = -1;
    size_t xk = 0, row_bytes = 0;
    for (uint32_t en : per[c]) {
      const int pi = (int)(en >> 24);
      items += 2 * (probs[pi].K / 256);
      row_bytes += (size_t)(probs[pi].K / 256) * kTileBytes;
      if (pi != last) { xk += probs[pi].K; last = pi; }
      plan.entry.push_back(en);
    }
    // must match the kernel's layout: alignment slack, header and x tables,
    // barriers, copies, entries, items, zero block and x, rows, item results
    const size_t smem = 128 + 16 + 8 * (size_t)kMaxGroupProblems + 8 * (size_t)(ne + kMaxGroupProblems + 2) +
                        16 * (size_t)(ne + kMaxGroupProblems) + 16 * (size_t)ne + 16 * (size_t)items + 16 +
                        2 * (32 + xk) + row_bytes + 64 * (size_t)items;
    // one thread per entry builds the item table
    plan.smem = std::max(plan.smem, ne > kGThreads ? SIZE_MAX : smem);
  }
  plan.cta_begin[grid] = (int32_t)plan.entry.size();
}

std::mutex g_plan_mu;
std::vector<GroupPlan> g_plans;   // a few recent shapes, most recent last

template <int kEntries>
cudaError_t launch_group_instance(const GemvGroupProblem* probs, int n, const GroupPlan& plan, int32_t* dev_status,
                                  cudaStream_t stream) {
  static GroupParams<kEntries> p;   // host staging copy; the launch copies it into the parameter space
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n; ++i) p.prob[i] = probs[i];
  p.dev_status = dev_status;
  const int grid = (int)plan.cta_begin.size() - 1;
  std::copy(plan.cta_begin.begin(), plan.cta_begin.end(), p.cta_begin);
  std::copy(plan.entry.begin(), plan.entry.end(), p.entry);
  const cudaError_t e = cudaFuncSetAttribute(q4_gemv_group_kernel<kEntries>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(q4_gemv_group_kernel<kEntries>, dim3(grid), dim3(kGThreads), plan.smem, stream, p);
}

}  // namespace

cudaError_t launch_q4_gemv_group(const GemvGroupProblem* probs, int n, int sms, int32_t* dev_status,
                                 cudaStream_t stream) {
  int rows = 0;
  for (int i = 0; i < n; ++i) rows += probs[i].N / 32;
  const int grid = std::min(std::min(rows, sms), kMaxGroupCtas);
  std::vector<int> key{grid};
  for (int i = 0; i < n; ++i) { key.push_back(probs[i].N); key.push_back(probs[i].K); }
  GroupPlan plan;
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    bool hit = false;
    for (size_t i = 0; i < g_plans.size(); ++i)
      if (g_plans[i].key == key) { plan = g_plans[i]; hit = true; break; }
    if (!hit) {
      plan.key = key;
      build_group_plan(probs, n, grid, plan);
      if (g_plans.size() >= 8) g_plans.erase(g_plans.begin());
      g_plans.push_back(plan);
    }
  }
  if (plan.smem > kGroupSmemBudget) {
    // too much per CTA in one launch: halve the group (a single problem this
    // large runs the single-problem kernel)
    if (n == 1) {
      Q4DenseArgs a{};
      a.tiles = probs[0].tiles;
      a.N = probs[0].N;
      a.K = probs[0].K;
      a.M = 1;
      a.X = probs[0].X;
      a.ldx = probs[0].K;
      a.Y = probs[0].Y;
      a.ldy = probs[0].N;
      return launch_q4_gemv1(a, sms, dev_status, stream);
    }
    const cudaError_t e = launch_q4_gemv_group(probs, n / 2, sms, dev_status, stream);
    if (e != cudaSuccess) return e;
    return launch_q4_gemv_group(probs + n / 2, n - n / 2, sms, dev_status, stream);
  }
  if (rows <= 1024) return launch_group_instance<1024>(probs, n, plan, dev_status, stream);
  return launch_group_instance<kMaxGroupRows>(probs, n, plan, dev_status, stream);
}

}  // namespace qmm
