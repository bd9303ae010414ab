// Exact int8 GEMM for small M (<= 64 rows), streaming form: the weight stream
// of the int8 half at decode and small-batch sizes ("int8 inference",
// "Product kernel (Int8Gemm)"; "The ONNX pack: weights to Q4NX, matmuls to
// our kernels, no VitisAI", "What works today": the M = 16 / 32 projection
// GEMMs and their per-call cost).
//
// One CTA per SM works on one problem: the host gives each problem a number
// of CTAs that evens out the weight bytes per CTA, and each CTA a contiguous
// range of the problem's items, an item being 16 output columns over all of
// K.  A loader thread first fetches the problem's M activation rows, then
// each item's 16 packed weight rows 1024 k at a time into a ring of 16 KB
// slots, each fetch one TMA box (a copy costs the SM's copy engine a fixed
// time whatever its size, so row-sized copies would cap the stream).  Both
// operands are viewed as {64 bytes, rows, k-blocks} and land as [k-block]
// [row][64 bytes], which the MMA fragments read without bank conflicts.
// Eight compute warps in two groups take alternate items (two items in
// flight), the four warps of a group splitting each chunk's K range; each
// widens its codes to f16
// (exact for |code| <= 128) and multiplies them with mma.sync m16n8k16 (fp32
// accumulate): every product is an integer of at most 2^14, so a sum of up
// to 1024 of them is exact in fp32, and the accumulators are drained into
// int32 before a warp's run of steps passes 1024 k.  Where the problem's f16
// activation rows fit in shared memory, they are widened once when the CTA
// starts instead of at every step.  The warps' exact partial sums go to one
// of two shared buffers, and two epilogue warps add them up and apply the
// zero points, bias and output conversion while the compute warps go on
// with the next item.  No CTA waits for another.
#include <algorithm>
#include <mutex>
#include <vector>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kCW = 8;                         // compute warps
constexpr int kGroups = 2;                     // compute groups: group g takes items i0 + g, i0 + g + kGroups, ...
constexpr int kGW = kCW / kGroups;             // warps of a group, splitting each chunk's K
constexpr int kEW = 2;                         // epilogue warps
constexpr int kLoaderWarp = kCW, kEpiWarp0 = kCW + 1;
constexpr int kThreads = 32 * (kCW + 1 + kEW);
constexpr int kItem = 16;                      // output columns per item
constexpr int kChunkKb = 16;                   // 64-byte k-blocks per ring slot (1024 k)
constexpr int kSlotBytes = kChunkKb * kItem * 64;
constexpr int kMaxSlots = 8;
constexpr int kMinSlots = 3;
constexpr int kMaxProb = 16;
constexpr int kMaxCtas = 256;
constexpr size_t kSmemCap = 225 * 1024;

struct alignas(16) StreamProb {
  const int8_t* A;
  int64_t lda;
  int M, K, N;
  uint32_t a_bias;       // XOR that turns an A byte into A' + 128
  const int8_t* B;       // packed [N][Kp]
  int Kp;
  int need_rowsum;
  int a16;               // A widened to f16 once, in shared memory (else int8 A, widened per step)
  Int8Epi epi;
};

struct StreamParams {
  CUtensorMap tmA[kMaxProb];          // A as {64, M, K / 64}, box {64, R, 16}
  CUtensorMap tmB[kMaxProb];          // packed B as {64, N, Kp / 64}, box {64, 16, 16}
  StreamProb prob[kMaxProb];
  int32_t item_begin[kMaxProb + 1];   // items of problem p: [item_begin[p], item_begin[p + 1])
  int32_t cta_begin[kMaxCtas + 1];    // items of CTA c: [cta_begin[c], cta_begin[c + 1]), all of one problem
  uint8_t cta_prob[kMaxCtas];         // the problem of CTA c
  int32_t a_bytes;                    // the A region: the largest of the problems' A layouts
  int32_t slots;                      // ring slots, kMinSlots..kMaxSlots
  int32_t* dev_status;
};

QMM_DEV void bar_compute() { asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory"); }

// Shared memory: A (int8 as [k-block][R][64 bytes], or f16 as [k-block][R]
// [128 bytes] with the 16-byte units of odd rows swapped in pairs), the ring
// [slots][16][16][64],
// the compute warps' partial sums [group][2 items][kGW][R][16] int32, the row sums [R], the CTA's
// problem, then the barriers and the abort flag.
struct Layout {
  uint32_t a, ring, red, rowsum, prob, bars, end;
  static constexpr int kBars = 1 + 2 * kMaxSlots + 4 * kGroups;   // a_full, full[], empty[], red_full[g][2], red_empty[g][2]
};
__host__ __device__ inline Layout stream_layout(int R, int a_bytes, int slots) {
  Layout l;
  l.a = 0;
  l.ring = l.a + (uint32_t)a_bytes;
  l.red = l.ring + (uint32_t)(slots * kSlotBytes);
  l.rowsum = l.red + (uint32_t)(kGroups * 2 * kGW * R * kItem * 4);
  l.prob = l.rowsum + (uint32_t)(R * 4);
  l.bars = l.prob + (uint32_t)sizeof(StreamProb);
  l.end = l.bars + (uint32_t)(Layout::kBars * 8 + 16);
  return l;
}
static_assert(sizeof(StreamProb) % 16 == 0, "keeps the barriers 8-byte aligned");

// One chunk's steps s0..s1 of a warp: B codes from the ring slot, A from
// shared memory (int8 widened here, or f16 widened once), m16n8k16 f16 MMAs
// into the fp32 accumulators.  In a step, lane t of a quad holds k = 16t ..
// 16t + 15 of the 64-k block for both operands: the MMAs' k order is a
// permutation that A and B share, so the sums are unchanged.
template <int MT, int NP, bool A16>
QMM_DEV void chunk_steps(float (&accf)[MT][2][NP][4], int s0, int s1, int kb0, uint32_t bslot, uint32_t a_base,
                         uint32_t a_off0, uint32_t a_off1, uint32_t a_bias) {
  using umma::lds128;
  constexpr uint32_t kA16Kb = MT * 16 * 128, kA8Kb = MT * 16 * 64;
#pragma unroll 2
  for (int st = s0; st < s1; ++st) {
    uint32_t bl[2][4], bh[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const uint4 v = lds128(bslot + (uint32_t)(st * kItem * 64 + nb * 8 * 64));
      biased4_to_f16(v.x ^ 0x80808080u, bl[nb][0], bh[nb][0]);
      biased4_to_f16(v.y ^ 0x80808080u, bl[nb][1], bh[nb][1]);
      biased4_to_f16(v.z ^ 0x80808080u, bl[nb][2], bh[nb][2]);
      biased4_to_f16(v.w ^ 0x80808080u, bl[nb][3], bh[nb][3]);
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t ra[8], rb[8];
      if constexpr (A16) {
        const uint32_t r0 = a_base + (uint32_t)(kb0 + st) * kA16Kb + (uint32_t)(16 * mt * 128), r1 = r0 + 8 * 128;
        const uint4 a0 = lds128(r0 + a_off0), a1 = lds128(r0 + a_off1);
        const uint4 b0 = lds128(r1 + a_off0), b1 = lds128(r1 + a_off1);
        ra[0] = a0.x; ra[1] = a0.y; ra[2] = a0.z; ra[3] = a0.w;
        ra[4] = a1.x; ra[5] = a1.y; ra[6] = a1.z; ra[7] = a1.w;
        rb[0] = b0.x; rb[1] = b0.y; rb[2] = b0.z; rb[3] = b0.w;
        rb[4] = b1.x; rb[5] = b1.y; rb[6] = b1.z; rb[7] = b1.w;
      } else {
        const uint32_t r0 = a_base + (uint32_t)(kb0 + st) * kA8Kb + (uint32_t)(16 * mt * 64);
        const uint4 va = lds128(r0), vb = lds128(r0 + 8 * 64);
        biased4_to_f16(va.x ^ a_bias, ra[0], ra[1]);
        biased4_to_f16(va.y ^ a_bias, ra[2], ra[3]);
        biased4_to_f16(va.z ^ a_bias, ra[4], ra[5]);
        biased4_to_f16(va.w ^ a_bias, ra[6], ra[7]);
        biased4_to_f16(vb.x ^ a_bias, rb[0], rb[1]);
        biased4_to_f16(vb.y ^ a_bias, rb[2], rb[3]);
        biased4_to_f16(vb.z ^ a_bias, rb[4], rb[5]);
        biased4_to_f16(vb.w ^ a_bias, rb[6], rb[7]);
      }
      // consecutive MMAs go to different accumulators
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
          mma_f16_16816(accf[mt][nb][i4 % NP], ra[2 * i4], rb[2 * i4], ra[2 * i4 + 1], rb[2 * i4 + 1], bl[nb][i4],
                        bh[nb][i4]);
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) int8_stream_kernel(const __grid_constant__ StreamParams p) {
  using namespace umma;
  constexpr int R = MT * 16;
  constexpr uint32_t kKbBytes = R * 64;   // one k-block of A in shared memory
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = smem_align(sm_raw, 128);
  const int NS = p.slots;
  const Layout L = stream_layout(R, p.a_bytes, NS);
  uint8_t* sA = sm + L.a;
  uint8_t* ring = sm + L.ring;
  int32_t* red = reinterpret_cast<int32_t*>(sm + L.red);
  int32_t* rowsum = reinterpret_cast<int32_t*>(sm + L.rowsum);
  StreamProb* sq = reinterpret_cast<StreamProb*>(sm + L.prob);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* a_full = bars;                       // the A boxes landed
  uint64_t* full = bars + 1;                     // [slots] a chunk landed
  uint64_t* empty = bars + 1 + kMaxSlots;        // [slots] the compute warps are done with a chunk
  uint64_t* red_full = bars + 1 + 2 * kMaxSlots; // [group][2] an item's partial sums are written
  uint64_t* red_empty = red_full + 2 * kGroups;  // [group][2] the epilogue is done with them
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + Layout::kBars);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int i0 = p.cta_begin[blockIdx.x], i1 = p.cta_begin[blockIdx.x + 1];
  const int pi = p.cta_prob[blockIdx.x];

  pdl_launch_dependents();
  {
    // this CTA's problem into shared memory (read many times, one dynamic
    // index of the parameter space)
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.prob[pi]);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sq);
    for (int x = threadIdx.x; x < (int)(sizeof(StreamProb) / 4); x += kThreads) dst[x] = src[x];
  }
  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGW);   // a chunk is consumed by its item's group
    }
    for (int b = 0; b < 2 * kGroups; ++b) {
      mbar_init(&red_full[b], kGW);
      mbar_init(&red_empty[b], kEW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (i0 >= i1) return;
  const StreamProb& q = *sq;
  const int ib = p.item_begin[pi];
  const int kb_full = q.K / 64;                 // whole k-blocks of A (the TMA part)
  const int na = q.a16 ? 0 : (kb_full + kChunkKb - 1) / kChunkKb;

  if (warp == kLoaderWarp) {
    // ---- loader: the A boxes, then every chunk of every item, in order ----
    {
      // the epilogue's per-column values of this CTA's columns, into L2
      // (one 128-byte line per lane and array)
      const int c0 = (i0 - ib) * kItem, c1 = min(q.N, (i1 - ib) * kItem);
      const int lines = ((c1 - 1) * 4 / 128) - (c0 * 4 / 128) + 1;
      for (int x = lane; x < lines; x += 32) {
        const int64_t off = (int64_t)(c0 * 4 / 128 + x) * 128 / 4;   // first column of the line
        prefetch_l2(q.epi.col_sum + off);
        if (q.epi.s_w) prefetch_l2(q.epi.s_w + off);
        if (q.epi.bias) prefetch_l2(q.epi.bias + off);
      }
    }
    if (lane != 0) return;
    const CUtensorMap* tmA = &p.tmA[pi];
    const CUtensorMap* tmB = &p.tmB[pi];
    tma_prefetch_desc(tmA);
    tma_prefetch_desc(tmB);
    // Warm A in L2 while the previous grid finishes (L2 is where global
    // memory is coherent; the copies come after the wait).  Of the weights
    // only the first chunk: a GPU-wide burst of all of them would queue ahead
    // of A and of every CTA's first chunk.
    for (int j = 0; j < (kb_full + kChunkKb - 1) / kChunkKb; ++j) tma_prefetch_l2_3d(tmA, 0, 0, j * kChunkKb);
    // and only the first chunk of weights (16 KB a CTA)
    tma_prefetch_l2_3d(tmB, 0, (i0 - ib) * kItem, 0);
    pdl_wait();
    // the A boxes go first in this SM's copy queue
    mbar_arrive_expect_tx(a_full, (uint32_t)(na * kChunkKb) * kKbBytes);
    for (int j = 0; j < na; ++j) tma_load_3d(smem_u32(sA + j * kChunkKb * kKbBytes), tmA, a_full, 0, 0, j * kChunkKb);
    int slot = 0, ph = 0, issued = 0;
    bool ok = true;
    for (int i = i0; i < i1 && ok; ++i) {
      const int n0 = (i - ib) * kItem;
      for (int kb = 0; kb < q.Kp / 64; kb += kChunkKb) {
        if (!mbar_wait(&empty[slot], ph ^ 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[slot], (uint32_t)kSlotBytes);
        tma_load_3d(smem_u32(ring + slot * kSlotBytes), tmB, &full[slot], 0, n0, kb);
        ++issued;
        if (++slot == NS) {
          slot = 0;
          ph ^= 1;
        }
      }
    }
    if (!ok) {
      // the copies already issued land before the CTA leaves: the A boxes, and
      // each slot's last issued phase (whether or not it was consumed)
      mbar_drain(a_full, 0);
      for (int s = 0; s < NS && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % NS);   // the last sequence number that used slot s
        mbar_drain(&full[s], (uint32_t)((last / NS) & 1));
      }
    }
    return;
  }

  if (warp >= kEpiWarp0) {
    // ---- epilogue warps: item j's partial sums (buffer j & 1) added up, then
    // zero points, bias and the output conversion; the compute warps go on
    // with the next items meanwhile ----
    pdl_wait();   // bias, scales and column sums may come from the previous grid
    // the problem's fields in registers: the output stores could alias the
    // shared copy as far as the compiler knows, so it would reload them
    const Int8Epi e = q.epi;
    const int qM = q.M, qN = q.N;
    constexpr int kRowStep = kEW * 32 / kItem;
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const int c = et % kItem, r0 = et / kItem;   // this thread: column c, rows r0, r0 + kRowStep, ...
    float sx[R / kRowStep];
#pragma unroll
    for (int k = 0; k < R / kRowStep; ++k) {
      const int m = min(r0 + kRowStep * k, qM - 1);
      sx[k] = e.s_x ? __uint_as_float(ldg32(e.s_x + (e.s_x_stride ? m : 0))) : 1.0f;
    }
    int32_t rs[R / kRowStep];   // row sums, read once the first item's partials (and they) are written
    // the per-column values of item i, loaded two items ahead of their use
    // (under the weight stream even L2 hits take the better part of an item)
    struct Col {
      int32_t cs, bias;
      float sw;
    };
    auto load_col = [&](int i) {
      Col v{0, 0, 1.0f};
      if (i < i1) {
        const int ncol = min((i - ib) * kItem + c, qN - 1);
        v.cs = (int32_t)ldg32(e.col_sum + ncol);
        if (e.bias) v.bias = (int32_t)ldg32(e.bias + ncol);
        if (e.s_w) v.sw = __uint_as_float(ldg32(e.s_w + ncol));
      }
      return v;
    };
    Col c0 = load_col(i0), c1 = load_col(i0 + 1);
    for (int i = i0, j = 0; i < i1; ++i, ++j) {
      const int grp = j % kGroups, jj = j / kGroups;   // the item's group, and its index there
      const int b = grp * 2 + (jj & 1);
      const int n = (i - ib) * kItem + c;
      const Col c2 = load_col(i + 2);
      const int32_t e_cs = c0.cs, e_bias = c0.bias;
      const float e_sw = c0.sw;
      c0 = c1;
      c1 = c2;
      if (!__all_sync(0xffffffffu, mbar_wait(&red_full[b], (uint32_t)((jj >> 1) & 1), abort_flag, p.dev_status)))
        break;
      if (*abort_flag) break;   // the compute warps gave up on this item
      if (j == 0) {
#pragma unroll
        for (int k = 0; k < R / kRowStep; ++k) rs[k] = rowsum[min(r0 + kRowStep * k, R - 1)];
      }
      const uint32_t rb = smem_u32(red) + (uint32_t)((b * kGW * R * kItem + r0 * kItem + c) * 4);
      uint32_t S[R / kRowStep];
#pragma unroll
      for (int k = 0; k < R / kRowStep; ++k) {
        S[k] = 0u;
#pragma unroll
        for (int w = 0; w < kGW; ++w) S[k] += lds32(rb + (uint32_t)((w * R + kRowStep * k) * kItem * 4));
      }
#pragma unroll
      for (int k = 0; k < R / kRowStep; ++k) {
        const int m = r0 + kRowStep * k;
        if (m < qM && n < qN) int8_store_vals(e, m, n, zp_correct((int32_t)S[k], e_cs, rs[k], e), e_bias, sx[k], e_sw);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[b]);
    }
    return;
  }

  // ---- compute warps: each chunk's K split eight ways; item j's partial sums
  // go to buffer j & 1 for the epilogue warps ----
  pdl_wait();   // A may come from the previous grid
  bool a_ok = true;
  if (q.a16) {
    // A from global memory, 16 codes a load, eight loads in flight a thread;
    // widened to f16 (A' exactly) into [k-block][R][128 bytes] with the
    // 16-byte units of odd rows swapped in pairs; rows past M are zeros.
    // Row sums of A' over k < K by shared-memory atomics.
    if (threadIdx.x < R) rowsum[threadIdx.x] = 0;
    bar_compute();
    const int pieces = q.Kp / 16, kr = (q.K + 15) / 16, total = R * pieces;
    const uint32_t to_s8 = q.a_bias ^ 0x80808080u;
    for (int x0 = threadIdx.x; x0 < total; x0 += 8 * kCW * 32) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = x0 + u * kCW * 32, r = x / pieces, c = x - r * pieces;
        v[u] = (x < total && r < q.M && c < kr) ? ldg128(q.A + (int64_t)r * q.lda + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = x0 + u * kCW * 32, r = x / pieces, c = x - r * pieces;
        if (x < total) {
          uint32_t f[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          if (r < q.M && c < kr) {
            biased4_to_f16(v[u].x ^ q.a_bias, f[0], f[1]);
            biased4_to_f16(v[u].y ^ q.a_bias, f[2], f[3]);
            biased4_to_f16(v[u].z ^ q.a_bias, f[4], f[5]);
            biased4_to_f16(v[u].w ^ q.a_bias, f[6], f[7]);
            if (q.need_rowsum) {
              const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
              int acc = 0;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int valid = q.K - (16 * c + 4 * e);
                const uint32_t m = valid >= 4 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : (0xFFFFFFFFu >> (32 - 8 * valid)));
                acc = __dp4a((int)((w4[e] ^ to_s8) & m), 0x01010101, acc);
              }
              atomicAdd(&rowsum[r], acc);
            }
          }
          const uint32_t row = smem_u32(sA) + (uint32_t)((c >> 2) * R * 128 + r * 128);
          const int j = c & 3, sw = r & 1;
          sts128(row + 16u * (uint32_t)((2 * j) ^ sw), make_uint4(f[0], f[1], f[2], f[3]));
          sts128(row + 16u * (uint32_t)((2 * j + 1) ^ sw), make_uint4(f[4], f[5], f[6], f[7]));
        }
      }
    }
    bar_compute();
  } else {
    a_ok = __all_sync(0xffffffffu, mbar_wait(a_full, 0, abort_flag, p.dev_status));
    if (q.K % 64 != 0) {
      // A's partial last k-block is not in the boxes: plain 16-byte loads
      // within roundup(K, 16), written after the boxes (and their zero fill) landed
      if (a_ok) {
        const int kt = kb_full * 64, pieces = (q.K - kt + 15) / 16;
        for (int x = threadIdx.x; x < q.M * pieces; x += kCW * 32) {
          const int r = x / pieces, c = x - r * pieces;
          const uint4 v = ldg128(q.A + (int64_t)r * q.lda + kt + 16 * c);
          sts128(smem_u32(sA + kb_full * kKbBytes + r * 64 + 16 * c), v);
        }
      }
      bar_compute();
    }
    if (a_ok && q.need_rowsum) {
      // row sums of A' over k < K, a warp per row (read after the first item's barrier)
      const uint32_t to_s8 = q.a_bias ^ 0x80808080u;
      for (int r = warp; r < q.M; r += kCW) {
        int acc = 0;
        for (int c = lane; c < q.Kp / 16; c += 32) {
          const uint4 v = lds128(smem_u32(sA + (c >> 2) * kKbBytes + r * 64 + 16 * (c & 3)));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int valid = q.K - (16 * c + 4 * e);
            const uint32_t m = valid >= 4 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : (0xFFFFFFFFu >> (32 - 8 * valid)));
            acc = __dp4a((int)((w4[e] ^ to_s8) & m), 0x01010101, acc);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) rowsum[r] = acc;
      }
    }
  }
  const uint32_t a_bias = q.a_bias;
  const int nkb = q.Kp / 64;
  // fragment addresses: row g (and g + 8), 16 bytes at 16t of each 64-k block
  const uint32_t a_lane = smem_u32(sA) + (uint32_t)(g * 64 + 16 * t);
  // f16 A: row g's 16-byte units 2t and 2t + 1, swapped in pairs on odd rows
  const uint32_t a16_lane = smem_u32(sA) + (uint32_t)(g * 128);
  const uint32_t a16_off0 = 16u * (uint32_t)((2 * t) ^ (g & 1)), a16_off1 = 16u * (uint32_t)((2 * t + 1) ^ (g & 1));
  const uint32_t b_lane = smem_u32(ring) + (uint32_t)(g * 64 + 16 * t);
  const int grp = warp / kGW, wg = warp % kGW;
  const int nch = (nkb + kChunkKb - 1) / kChunkKb;   // chunks per item
  for (int i = i0 + grp, j = 0; i < i1; i += kGroups, ++j) {
    // the item's chunks are numbers (i - i0) * nch + c of the CTA's sequence
    int seq = (i - i0) * nch;
    int slot = seq % NS, ph = (seq / NS) & 1;
    // fp32 accumulators per (row tile, column block, k parity): with one row
    // tile, the k parity doubles the independent MMA chains
    constexpr int NP = MT == 1 ? 2 : 1;
    int acc[MT][2][4];
    float accf[MT][2][NP][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[mt][nb][e] = 0;
#pragma unroll
          for (int pp = 0; pp < NP; ++pp) accf[mt][nb][pp][e] = 0.f;
        }
    int nst = 0;   // steps in the fp32 accumulators since the last drain
    bool ok = a_ok;
    for (int kb0 = 0; kb0 < nkb; kb0 += kChunkKb) {
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&full[slot], (uint32_t)ph, abort_flag, p.dev_status));
      if (ok) {
        const int cs = min(kChunkKb, nkb - kb0);
        const int s0 = wg * cs / kGW, s1 = (wg + 1) * cs / kGW;
        if (nst + (s1 - s0) > 16) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
              for (int pp = 0; pp < NP; ++pp)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  acc[mt][nb][e] += __float2int_rn(accf[mt][nb][pp][e]);
                  accf[mt][nb][pp][e] = 0.f;
                }
          nst = 0;
        }
        nst += s1 - s0;
        const uint32_t bslot = b_lane + (uint32_t)(slot * kSlotBytes);
        if (q.a16)
          chunk_steps<MT, NP, true>(accf, s0, s1, kb0, bslot, a16_lane, a16_off0, a16_off1, a_bias);
        else
          chunk_steps<MT, NP, false>(accf, s0, s1, kb0, bslot, a_lane, 0u, 0u, a_bias);
      }
      // every lane's shared-memory reads of this slot are done
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == NS) {
        slot = 0;
        ph ^= 1;
      }
    }
    // buffer j & 1 is free once the epilogue is done with item j - 2
    const int b = grp * 2 + (j & 1);
    ok = __all_sync(0xffffffffu, mbar_wait(&red_empty[b], (uint32_t)(((j >> 1) & 1) ^ 1), abort_flag, p.dev_status)) && ok;
    const uint32_t rb = smem_u32(red) + (uint32_t)(b * kGW * R * kItem * 4);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        int v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[e] = acc[mt][nb][e];
#pragma unroll
          for (int pp = 0; pp < NP; ++pp) v[e] += __float2int_rn(accf[mt][nb][pp][e]);
        }
        // D fragment: (row g, columns 2t, 2t+1) and (row g + 8, same columns)
        const uint32_t r0 = rb + (uint32_t)(((wg * R + 16 * mt + g) * kItem + 8 * nb + 2 * t) * 4);
        sts64(r0, (uint32_t)v[0], (uint32_t)v[1]);
        sts64(r0 + 8 * kItem * 4, (uint32_t)v[2], (uint32_t)v[3]);
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[b]);
    if (!ok) break;
  }
}

int group_mt(const Int8GemmArgs* probs, int n) {
  int mt = 1;
  for (int i = 0; i < n; ++i) mt = std::max(mt, (probs[i].M + 15) / 16);
  return mt;
}

// k-blocks of int8 A in shared memory: the boxes cover whole 16-block chunks
// of the K / 64 full blocks, and a partial last block sits after them.
int a_blocks(int K) { return std::max((K / 64 + kChunkKb - 1) / kChunkKb * kChunkKb, (K + 63) / 64); }

constexpr int kA16MinSlots = 4;   // f16 A only where it leaves at least this deep a ring

// Shared-memory plan of a group: f16 A per problem where it fits, the A
// region (the largest problem's), the ring depth (0: the group does not fit).
struct GroupPlan {
  int R = 0, a_bytes = 0, slots = 0;
  bool a16[kMaxProb] = {};
};
GroupPlan plan_group(const Int8GemmArgs* probs, int n) {
  GroupPlan g;
  g.R = group_mt(probs, n) * 16;
  for (int i = 0; i < n; ++i) {
    const int b16 = 2 * g.R * (int)probs[i].Kp, b8 = g.R * 64 * a_blocks(probs[i].K);
    g.a16[i] = stream_layout(g.R, b16, kA16MinSlots).end + 128 <= kSmemCap;
    g.a_bytes = std::max(g.a_bytes, g.a16[i] ? b16 : b8);
  }
  for (int s = kMaxSlots; s >= kMinSlots && g.slots == 0; --s)
    if (stream_layout(g.R, g.a_bytes, s).end + 128 <= kSmemCap) g.slots = s;
  return g;
}

template <int MT>
cudaError_t launch_stream_mt(const StreamParams& p, int grid, size_t smem, cudaStream_t stream) {
  const cudaError_t e =
      cudaFuncSetAttribute(int8_stream_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(int8_stream_kernel<MT>, dim3(grid), dim3(kThreads), smem, stream, p);
}

}  // namespace

bool int8_stream_fits(const Int8GemmArgs* probs, int n) {
  if (n < 1 || n > kMaxProb) return false;
  for (int i = 0; i < n; ++i)
    if (probs[i].M > 64 || probs[i].Kp > 65536) return false;
  return plan_group(probs, n).slots > 0;
}

int64_t int8_stream_items(const Int8GemmArgs* probs, int n) {
  int64_t items = 0;
  for (int i = 0; i < n; ++i) items += (probs[i].N + kItem - 1) / kItem;
  return items;
}

cudaError_t launch_int8_stream_group(const Int8GemmArgs* probs, int n, int32_t* dev_status, cudaStream_t stream) {
  if (!int8_stream_fits(probs, n)) return cudaErrorInvalidValue;
  static StreamParams p;   // host staging copy (8 KB); the launch copies it into the parameter space
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  p = StreamParams{};
  const GroupPlan gp = plan_group(probs, n);
  const int R = gp.R, MT = R / 16;
  p.a_bytes = gp.a_bytes;
  p.slots = gp.slots;
  p.dev_status = dev_status;
  int64_t items = 0;
  std::vector<int64_t> ni(n), w(n);
  for (int i = 0; i < n; ++i) {
    const Int8GemmArgs& a = probs[i];
    StreamProb& q = p.prob[i];
    q.A = a.A;
    q.lda = a.lda;
    q.M = a.M;
    q.K = a.K;
    q.N = a.N;
    q.a_bias = a.a_u8 ? 0u : 0x80808080u;
    q.B = a.B;
    q.Kp = (int)a.Kp;
    q.need_rowsum = a.need_rowsum ? 1 : 0;
    q.a16 = gp.a16[i] ? 1 : 0;
    q.epi = a.epi;
    // A's whole 64-byte k-blocks (a partial last one is loaded apart); at
    // least one block keeps the map valid when K < 64 (then no box is issued)
    if (!make_tmap_kblocks(&p.tmA[i], a.A, (uint64_t)a.M, (uint64_t)a.lda, (uint64_t)std::max(a.K / 64, 1), R,
                           kChunkKb) ||
        !make_tmap_kblocks(&p.tmB[i], a.B, (uint64_t)a.N, (uint64_t)a.Kp, (uint64_t)(a.Kp / 64), kItem, kChunkKb))
      return cudaErrorInvalidValue;
    p.item_begin[i] = (int32_t)items;
    ni[i] = (a.N + kItem - 1) / kItem;
    // an item's cost: its weight bytes, a third more where A is widened per step
    w[i] = (int64_t)kItem * a.Kp * (gp.a16[i] ? 3 : 4);
    items += ni[i];
  }
  p.item_begin[n] = (int32_t)items;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int G = std::min(sms, kMaxCtas);
  if (n > G) return cudaErrorInvalidValue;
  // CTAs per problem: start at one each, then keep lowering the largest
  // per-CTA cost (ceil(items / ctas) * item cost) by giving its
  // problem just enough CTAs to drop one item per CTA, while CTAs remain.
  std::vector<int64_t> c(n, 1);
  int64_t left = G - n;
  for (;;) {
    int worst = -1;
    int64_t worst_load = -1;
    for (int i = 0; i < n; ++i) {
      const int64_t load = (ni[i] + c[i] - 1) / c[i] * w[i];
      if (load > worst_load) {
        worst_load = load;
        worst = i;
      }
    }
    const int64_t per = (ni[worst] + c[worst] - 1) / c[worst];
    if (per <= 1) break;
    const int64_t need = (ni[worst] + per - 2) / (per - 1) - c[worst];   // CTAs for per - 1 items each
    if (need > left) break;
    c[worst] += need;
    left -= need;
  }
  // each problem's items in even contiguous ranges over its CTAs
  int cta = 0;
  for (int i = 0; i < n; ++i)
    for (int64_t j = 0; j < c[i]; ++j, ++cta) {
      p.cta_begin[cta] = p.item_begin[i] + (int32_t)(j * ni[i] / c[i]);
      p.cta_prob[cta] = (uint8_t)i;
    }
  p.cta_begin[cta] = (int32_t)items;
  const size_t smem = stream_layout(R, p.a_bytes, p.slots).end + 128;
  switch (MT) {
    case 1: return launch_stream_mt<1>(p, cta, smem, stream);
    case 2: return launch_stream_mt<2>(p, cta, smem, stream);
    case 3: return launch_stream_mt<3>(p, cta, smem, stream);
    default: return launch_stream_mt<4>(p, cta, smem, stream);
  }
}

}  // namespace qmm
