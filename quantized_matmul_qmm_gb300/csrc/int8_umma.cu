// Exact int8 GEMM on the 5th-generation tensor cores (tcgen05) for large M.
//
// The operation is that of "int8 inference", "Product kernel (Int8Gemm)":
// S = sum_k A'B' in int32, then the zero-point correction and the epilogue.
// sm_103a has no tcgen05 integer MMA (ptxas rejects .kind::i8 for it), so the
// contraction runs on kind::f16 with integer-valued operands.  Every code in
// [-128, 127] is exact in f16, and every product, at most 2^14 in magnitude,
// is exact in the fp32 accumulator.  A sum of at most 1024 such products stays
// within 2^24, where fp32 holds every integer.  So the accumulator is drained
// every 1024 K (kChunkK) into int32 registers, and the result is exact.  Two
// TMEM accumulators alternate, so the MMAs of chunk c+1 run while the
// epilogue drains chunk c.
//
// Launches:
//   1. widen: A (uint8/int8) -> A' in f16 with rowSum[m] fused into the same
//      pass (dp4a, then warp shuffles), and packed B' (int8) -> f16.
//   2. the GEMM, on CTA pairs (clusters of two): a pair owns a 256 x 256
//      output tile and issues tcgen05.mma.cta_group::2 (M = 256, N = 256).
//      Each CTA stages its own 128 rows of A and 128 rows of B' (output
//      columns), so per SM the tensor pipe reads 16 KB of operands per 64 K
//      instead of the 24 KB a one-CTA 128 x 256 tile needs, and the pair's L2
//      reads drop by a third.  In each CTA warp 0 issues the TMA loads (both
//      CTAs' loads complete on the even CTA's barrier), warp 1 holds TMEM and,
//      in the even CTA, issues the MMAs; warps 2..9 drain the CTA's own
//      128 x 256 accumulator and run the exact epilogue: zero points, bias,
//      output conversion.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kBM = 128;             // activation rows per CTA (the pair: 256, the MMA M)
constexpr int kBN = 256;             // output columns per tile (MMA N)
constexpr int kBNh = kBN / 2;        // weight rows staged by each CTA of the pair
constexpr int kBK = 64;              // K per stage (one 128-byte swizzle row of f16)
constexpr int kStages = 6;
constexpr int kChunkK = 1024;        // K per exact fp32 chunk
constexpr int kChunkKB = kChunkK / kBK;
static_assert(kChunkK == kPairChunkK, "the W8A16 chunk scales assume 1,024-k chunks");
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBNh * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
// warp 0 TMA producer, warp 1 TMEM owner / MMA issuer, warps 2..9 epilogue.
// Ten warps put three on some SM sub-partitions, which caps the kernel at 168
// registers.
constexpr int kEpiWarp0 = 2;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kTmemCols = 512;       // two 256-column fp32 accumulators
constexpr int kColConstBytes = kEpiWarps * 2 * 128 * 12;   // per warp: two sets of c1 / s_w / Mq, 128 columns
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kColConstBytes + 256;
constexpr int kMinM = 65;            // up to 64 rows the small-M route is used (a pair tile is 256
                                     // rows: from 65 rows on, partly empty tiles still beat the integer MMA)
constexpr uint16_t kBothCtas = 0x3;
constexpr int kMaxDevices = 64;
constexpr int kWidenMaxSmem = 160 * 1024;   // >= 2 rows of the largest padded K (2 x 65792 bytes) + alignment

struct Int8UmmaParams {
  int M, N, K, Kp;
  int tiles_n;                       // number of 256-column tiles
  int ntiles;                        // 256 x 256 tiles
  const int32_t* row_sum;            // [M] (null when zB' == 0)
  Int8Epi epi;
  int32_t* dev_status;
  const float* w8_scales;            // W8A16 and Q8: [N][w8_nb], one per row and 1,024 k
  int w8_nb;
  const float* x_up;                 // Q8: inverse scale of each f16 activation row
};

// W8A16 instance of the kernel: bf16 activations x int8 weights widened to
// bf16 (exact), each 1,024-k accumulator chunk scaled per column by its
// block's weight scale, fp32 output.
constexpr int kW8Out = 100;
// Q8 instance: the same epilogue on f16 weights and f16 activation rows,
// each output row multiplied by its activation row's inverse scale.
constexpr int kQ8Out = 101;
constexpr bool is_chunk_scaled(int out) { return out == kW8Out || out == kQ8Out; }

// Output conversion of one element (fp32 steps with explicit IEEE rounding),
// specialised on the output type; kPerRowMq: requantisation with a per-row
// activation scale, whose multiplier Mq is formed per element.
template <int kOut, bool kPerRowMq>
__device__ __forceinline__ uint32_t epi_convert(const Int8Epi& e, int32_t yb, float sx, float sw, float mq) {
  if constexpr (kOut == QMM_S32) {
    return (uint32_t)yb;
  } else if constexpr (kOut == QMM_F32) {
    return __float_as_uint(__fmul_rn(__fmul_rn(__int2float_rn(yb), sx), sw));
  } else {
    const float m = kPerRowMq ? __fdiv_rn(__fmul_rn(sx, sw), e.s_y) : mq;
    float r = __fmul_rn(__int2float_rn(yb), m);
    r = fminf(fmaxf(r, -1.0e9f), 1.0e9f);
    int q = __float2int_rn(r) + e.zp_y;
    q = (kOut == QMM_S8) ? min(max(q, -128), 127) : min(max(q, 0), 255);
    return (uint32_t)q & 0xFFu;
  }
}

// 32 consecutive columns of one row: converted and stored 16 bytes at a time
// (element-wise at ragged edges or unaligned outputs).  The per-column
// constants are read four at a time (every lane reads the same address).
template <int kOut, bool kPerRowMq>
__device__ __forceinline__ void epi_store32(const Int8UmmaParams& p, int row, int nb, const int32_t* acc,
                                            const uint32_t* c1, const float* sw, const float* mq, uint32_t r1,
                                            float sx, bool vec_ok) {
  const Int8Epi& e = p.epi;
  const bool full = vec_ok && nb + 32 <= p.N;
  constexpr bool kNeedSw = kOut == QMM_F32 || kPerRowMq;
  constexpr bool kNeedMq = (kOut == QMM_S8 || kOut == QMM_U8) && !kPerRowMq;
  constexpr bool kWide = kOut == QMM_S32 || kOut == QMM_F32;
  uint32_t* dst32 = reinterpret_cast<uint32_t*>(e.out) + (int64_t)row * e.ldo + nb;
  uint8_t* dst8 = reinterpret_cast<uint8_t*>(e.out) + (int64_t)row * e.ldo + nb;
  uint32_t w[4];
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 c4 = reinterpret_cast<const uint4*>(c1)[v];
    const float4 w4 = kNeedSw ? reinterpret_cast<const float4*>(sw)[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 m4 = kNeedMq ? reinterpret_cast<const float4*>(mq)[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t cc[4] = {c4.x, c4.y, c4.z, c4.w};
    const float ww[4] = {w4.x, w4.y, w4.z, w4.w}, mm[4] = {m4.x, m4.y, m4.z, m4.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = epi_convert<kOut, kPerRowMq>(e, (int32_t)((uint32_t)acc[4 * v + i] + cc[i] + r1), sx, ww[i], mm[i]);
    if constexpr (kWide) {
      if (full) {
        reinterpret_cast<uint4*>(dst32)[v] = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (nb + 4 * v + i < p.N) dst32[4 * v + i] = o[i];
      }
    } else {
      w[v & 3] = o[0] | (o[1] << 8) | (o[2] << 16) | (o[3] << 24);
      if ((v & 3) == 3) {
        if (full) {
          reinterpret_cast<uint4*>(dst8)[v >> 2] = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (nb + 16 * (v >> 2) + i < p.N) dst8[16 * (v >> 2) + i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
        }
      }
    }
  }
}

// Persistent: pair c (cluster c) walks tiles c, c + #clusters, ...  The stage
// ring and the two TMEM accumulators carry on across tiles, so the epilogue
// of one tile overlaps the MMAs of the next.
template <int kOut, bool kPerRowMq>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
int8_umma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Int8UmmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  // same offsets in both CTAs: the pair MMA addresses the odd CTA's operand
  // tiles through the even CTA's descriptors
  uint8_t* smem = smem_align(smem_raw, 1024);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sConst = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sConst + kColConstBytes);   // used in the even CTA
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;    // [2]
  uint64_t* tempty = tfull + 2;         // [2], used in the even CTA
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();
  const int nkb = p.Kp / kBK;
  const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&tfull[d], 1);
      mbar_init(&tempty[d], 2 * kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  cluster_sync();   // both CTAs' barriers are initialised before any remote use
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs hold their TMEM before the first pair MMA
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the prologue above overlaps the widen grid; its outputs are read below
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;          // k blocks issued so far (all tiles)
      bool ok = true;
      for (int t = pair; t < p.ntiles && ok; t += npairs) {
        // rows past M or N are never stored: a box that would lie wholly
        // outside the tensor is pulled back onto its last row
        const int m0 = min((t / p.tiles_n) * (2 * kBM) + (int)rank * kBM, p.M - 1);
        const int n0 = min((t % p.tiles_n) * kBN + (int)rank * kBNh, p.N - 1);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kStageBytes);
          tma_load_2d_pair(smem_u32(sA + s * kABytes), &tmA, bar, kb * kBK, m0);
          tma_load_2d_pair(smem_u32(sB + s * kBBytes), &tmB, bar, kb * kBK, n0);
        }
      }
      if (ok) {
        // the last stages are released once the MMAs reading them are done,
        // which also means every copy into this CTA has landed
        for (int k = g > kStages ? g - kStages : 0; k < g; ++k)
          if (!mbar_wait(&empty[k % kStages], (k / kStages) & 1, abort_flag, p.dev_status)) break;
      } else {
        // copies already issued land within microseconds
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // The issue loop is kept short (stage and phase counted, descriptors
      // offset from precomputed bases): the tensor pipe queues few MMAs, so
      // this thread's latency per 64-k block is on the critical path.
      constexpr uint32_t idesc = idesc_f16(2 * kBM, kBN, kOut == kW8Out);   // bf16 operands for W8A16 only
      const uint64_t adesc0 = desc_kmajor_sw128(smem_u32(sA)), bdesc0 = desc_kmajor_sw128(smem_u32(sB));
      int s = 0, gc = 0;  // stage; chunks issued (all tiles)
      uint32_t ph = 0;    // phase parity of the full barriers at stage s
      bool ok = true;
      for (int t = pair; t < p.ntiles && ok; t += npairs) {
        for (int c = 0; c < nchunks && ok; ++c, ++gc) {
          const int d = gc & 1, u = gc >> 1;
          if (!mbar_wait(&tempty[d], (u & 1) ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dt = tmem + d * kBN;
          const int nkb_c = min(nkb - c * kChunkKB, kChunkKB);
          for (int kb = 0; kb < nkb_c; ++kb) {
            if (!mbar_wait(&full[s], ph, abort_flag, p.dev_status)) { ok = false; break; }
            tc_fence_after();
            // +32 bytes per 16 K inside the 128-byte swizzle row: +2 in the address field
            const uint64_t ad = adesc0 + (uint64_t)((s * kABytes) >> 4);
            const uint64_t bd = bdesc0 + (uint64_t)((s * kBBytes) >> 4);
            umma_f16_pair(dt, ad, bd, idesc, kb > 0 ? 1u : 0u);
            umma_f16_pair(dt, ad + 2, bd + 2, idesc, 1u);
            umma_f16_pair(dt, ad + 4, bd + 4, idesc, 1u);
            umma_f16_pair(dt, ad + 6, bd + 6, idesc, 1u);
            umma_commit_pair(&empty[s], kBothCtas);
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (ok) umma_commit_pair(&tfull[d], kBothCtas);
        }
      }
      // every MMA has completed before either CTA releases its TMEM
      umma_commit_pair(done, 0x1);
      mbar_wait(done, 0, abort_flag, p.dev_status);
    }
  } else if (is_chunk_scaled(kOut) && warp >= kEpiWarp0) {
    // W8A16 / Q8 epilogue: each 1,024-k chunk of the accumulator, times the
    // weight scale of that chunk's block for each column, is added in fp32.  A
    // warp's 128 column scales are fetched one chunk ahead into shared memory.
    const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
    const int ew = warp - kEpiWarp0;
    float* scs = reinterpret_cast<float*>(sConst) + ew * 768;   // [2][128]
    const uint32_t tempty_even[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
    auto load_scales = [&](int t, int c, int b) {
      const int nbase = (t % p.tiles_n) * kBN + h * 128;
      float sv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int n = nbase + lane + 32 * v;
        sv[v] = n < p.N ? p.w8_scales[(int64_t)n * p.w8_nb + c] : 0.f;
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) scs[b * 128 + lane + 32 * v] = sv[v];
    };
    if (pair < p.ntiles) load_scales(pair, 0, 0);
    __syncwarp();
    float* Yf = reinterpret_cast<float*>(p.epi.out);
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(Yf) & 15) == 0) && (p.epi.ldo % 4 == 0);
    int gc = 0;
    bool ok = true;
    for (int t = pair; t < p.ntiles && ok; t += npairs) {
      const int m0 = (t / p.tiles_n) * (2 * kBM) + (int)rank * kBM, n0 = (t % p.tiles_n) * kBN;
      const int nbase = n0 + h * 128;
      const int row = m0 + 32 * q + lane;
      float acc[128];
      for (int c = 0; c < nchunks; ++c, ++gc) {
        const int d = gc & 1, u = gc >> 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[d], u & 1, abort_flag, p.dev_status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* sc = scs + (gc & 1) * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * kBN + h * 128 + 32 * j), r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = __uint_as_float(r[i]), w = sc[32 * j + i];
            acc[32 * j + i] = (c == 0) ? __fmul_rn(v, w) : fmaf(v, w, acc[32 * j + i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_even[d]);
        // the next chunk's scales: this tile's next block, or the next tile's first
        if (c + 1 < nchunks) load_scales(t, c + 1, (gc + 1) & 1);
        else if (t + npairs < p.ntiles) load_scales(t + npairs, 0, (gc + 1) & 1);
        __syncwarp();
      }
      if (ok && row < p.M) {
        if (kOut == kQ8Out) {
          const float xu = p.x_up[row];   // a power of two: exact
#pragma unroll
          for (int i = 0; i < 128; ++i) acc[i] *= xu;
        }
        float* yrow = Yf + (int64_t)row * p.epi.ldo;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int nb = nbase + 32 * j;
          if (vec_ok && nb + 32 <= p.N) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(yrow + nb)[v] = make_float4(acc[32 * j + 4 * v], acc[32 * j + 4 * v + 1],
                                                                     acc[32 * j + 4 * v + 2], acc[32 * j + 4 * v + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (nb + i < p.N) yrow[nb + i] = acc[32 * j + i];
          }
        }
      }
      __syncwarp();
    }
  } else if (!is_chunk_scaled(kOut) && warp >= kEpiWarp0) {
    // epilogue: warp w reads TMEM lanes 32*(w%4).. and columns h*128..h*128+127
    const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
    const int ew = warp - kEpiWarp0;
    // per-warp column constants of 128 columns (bias - zA' colSum, s_w, Mq),
    // two sets: the tile being drained and the next one, loaded early
    uint32_t* cset = reinterpret_cast<uint32_t*>(sConst) + ew * 768;
    const uint32_t tempty_even[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
    const Int8Epi& e = p.epi;
    constexpr bool kRequant = kOut == QMM_S8 || kOut == QMM_U8;
    const bool per_row_sx = (e.s_x != nullptr && e.s_x_stride != 0);
    const float sx0 = e.s_x ? e.s_x[0] : 1.0f;
    constexpr int esz = (kOut == QMM_S32 || kOut == QMM_F32) ? 4 : 1;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(e.out) & 15) == 0) && (((int64_t)e.ldo * esz) % 16 == 0);
    auto load_consts = [&](int t, int b) {
      const int nbase = (t % p.tiles_n) * kBN + h * 128;
      uint32_t* c1 = cset + b * 384;
      int32_t bi[4], cs[4];
      float wv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {   // all loads first: one memory round trip
        const int n = nbase + lane + 32 * v;
        const bool in = n < p.N;
        bi[v] = (in && e.bias) ? e.bias[n] : 0;
        cs[v] = in ? e.col_sum[n] : 0;
        wv[v] = (in && e.s_w) ? e.s_w[n] : 1.0f;
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int i = lane + 32 * v;
        c1[i] = (uint32_t)bi[v] - e.zAp * (uint32_t)cs[v];
        reinterpret_cast<float*>(c1 + 128)[i] = wv[v];
        reinterpret_cast<float*>(c1 + 256)[i] =
            (kRequant && !kPerRowMq && nbase + i < p.N) ? __fdiv_rn(__fmul_rn(sx0, wv[v]), e.s_y) : 0.0f;
      }
    };
    if (pair < p.ntiles) load_consts(pair, 0);
    __syncwarp();
    int gc = 0, it = 0;
    bool ok = true;
    for (int t = pair; t < p.ntiles && ok; t += npairs, ++it) {
      const int m0 = (t / p.tiles_n) * (2 * kBM) + (int)rank * kBM, n0 = (t % p.tiles_n) * kBN;
      const int nbase = n0 + h * 128;
      const int row = m0 + 32 * q + lane;
      int32_t rsum = 0;
      float sx = sx0;
      int32_t acc[128];
      for (int c = 0; c < nchunks; ++c, ++gc) {
        const int d = gc & 1, u = gc >> 1;
        // warp-uniform: tcgen05.ld below is a whole-warp instruction
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[d], u & 1, abort_flag, p.dev_status))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * kBN + h * 128 + 32 * j), r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int32_t v = __float2int_rn(__uint_as_float(r[i]));
            acc[32 * j + i] = (c == 0) ? v : (int32_t)((uint32_t)acc[32 * j + i] + (uint32_t)v);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_even[d]);
        if (c == 0) {
          // while the remaining chunks run: this row's terms, the next tile's columns
          if (row < p.M) {
            if (p.row_sum) rsum = p.row_sum[row];
            if (per_row_sx) sx = e.s_x[row];
          }
          if (t + npairs < p.ntiles) load_consts(t + npairs, (it + 1) & 1);
        }
      }
      __syncwarp();
      if (ok && row < p.M) {
        const uint32_t r1 = p.row_sum ? (0u - e.zBp * ((uint32_t)rsum - e.Kz)) : 0u;
        const uint32_t* c1 = cset + (it & 1) * 384;
        const float* swc = reinterpret_cast<const float*>(c1 + 128);
        const float* mqc = reinterpret_cast<const float*>(c1 + 256);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          epi_store32<kOut, kPerRowMq>(p, row, nbase + 32 * j, acc + 32 * j, c1 + 32 * j, swc + 32 * j,
                                       mqc + 32 * j, r1, sx, vec_ok);
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  cluster_sync();   // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Widen: A rows (shift, K-tail mask, rowSum) and packed B rows to f16.  A
// persistent grid; each block walks groups of R consecutive rows.  Thread 0
// streams a group into shared memory with one bulk copy per row (2-stage
// ring: the next group lands while this one is converted), then every thread
// converts 8 bytes at a time and writes 16 bytes of f16, coalesced.
constexpr int kWidenThreads = 256;
constexpr int kWidenMaxRows = 8;        // rows per group (R)
constexpr int kWidenGroupBytes = 12288; // target bytes of a group

struct WidenParams {
  const int8_t* A;
  int64_t lda;
  const int8_t* B;
  __half* A16;
  __half* B16;
  int32_t* row_sum;
  int32_t* dev_status;
  int M, K, N, Kp, R;
  bool a_u8;
  bool b_bf16;   // B' as bf16 instead of f16 (the W8A16 instance; M == 0 then)
};

__global__ void __launch_bounds__(kWidenThreads) int8_widen_kernel(const WidenParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[2];
  __shared__ int red[2][kWidenMaxRows][kWidenThreads / 32];
  __shared__ volatile int abort_flag;
  // the GEMM grid may start its prologue; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint8_t* buf = smem_align(smem_raw, 128);
  const int rows = p.M + p.N, R = p.R;
  const int ngroups = (rows + R - 1) / R;
  const int K16 = (p.K + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int grp, int s) {
    uint32_t bytes = 0;
    for (int r = 0; r < R; ++r) {
      const int row = grp * R + r;
      if (row < rows) bytes += row < p.M ? (uint32_t)K16 : (uint32_t)p.Kp;
    }
    fence_proxy_async_smem();   // the generic reads of this buffer precede the copy
    mbar_arrive_expect_tx(&bar[s], bytes);
    for (int r = 0; r < R; ++r) {
      const int row = grp * R + r;
      if (row >= rows) break;
      const uint32_t dst = smem_u32(buf + (size_t)(s * R + r) * p.Kp);
      if (row < p.M) bulk_g2s(dst, p.A + (int64_t)row * p.lda, (uint32_t)K16, &bar[s]);
      else bulk_g2s(dst, p.B + (int64_t)(row - p.M) * p.Kp, (uint32_t)p.Kp, &bar[s]);
    }
  };

  int it = 0;
  if (threadIdx.x == 0 && (int)blockIdx.x < ngroups) issue(blockIdx.x, 0);
  for (int g = blockIdx.x; g < ngroups; g += gridDim.x, ++it) {
    const int s = it & 1;
    // buffer s ^ 1 was released by the barrier that ended the previous group
    if (threadIdx.x == 0 && g + (int)gridDim.x < ngroups) issue(g + gridDim.x, s ^ 1);
    // block-uniform: a wait that gave up in any thread ends the loop for all
    if (__syncthreads_or(!mbar_wait(&bar[s], (it >> 1) & 1, &abort_flag, p.dev_status))) break;
    for (int r = 0; r < R; ++r) {
      const int row = g * R + r;
      if (row >= rows) break;
      const bool is_a = row < p.M;
      const uint8_t* src = buf + (size_t)(s * R + r) * p.Kp;
      __half* dst = is_a ? p.A16 + (int64_t)row * p.Kp : p.B16 + (int64_t)(row - p.M) * p.Kp;
      const int limit = is_a ? K16 : p.Kp;
      const uint32_t xorv = (is_a && p.a_u8) ? 0x80808080u : 0u;
      int sum = 0;
      for (int k = threadIdx.x * 8; k < p.Kp; k += kWidenThreads * 8) {
        uint32_t w[2] = {0u, 0u};
        if (k < limit) {
          const uint2 v = *reinterpret_cast<const uint2*>(src + k);
          w[0] = v.x ^ xorv;
          w[1] = v.y ^ xorv;
          if (is_a && k + 8 > p.K) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int valid = p.K - (k + 4 * q);
              if (valid <= 0) w[q] = 0u;
              else if (valid < 4) w[q] &= (1u << (8 * valid)) - 1u;
            }
          }
        }
        if (p.b_bf16) {
          // every int8 code is exact in bf16 (8 significant bits)
          __nv_bfloat16 h[8];
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int b = 0; b < 4; ++b) h[4 * q + b] = __int2bfloat16_rn((int)(int8_t)(w[q] >> (8 * b)));
          *reinterpret_cast<uint4*>(dst + k) = *reinterpret_cast<const uint4*>(h);
          continue;
        }
        // the codes (exact in f16) through their biased bytes: two byte
        // permutes and two f16x2 subtractions per four codes
        uint4 h;
        sum = __dp4a((int)w[0], 0x01010101, sum);
        sum = __dp4a((int)w[1], 0x01010101, sum);
        biased4_to_f16(w[0] ^ 0x80808080u, h.x, h.y);
        biased4_to_f16(w[1] ^ 0x80808080u, h.z, h.w);
        *reinterpret_cast<uint4*>(dst + k) = h;
      }
      if (is_a) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) red[it & 1][r][warp] = sum;
      }
    }
    __syncthreads();   // buffer s is free; red[it & 1] is complete
    if ((int)threadIdx.x < R && p.row_sum != nullptr) {
      const int row = g * R + threadIdx.x;
      if (row < p.M) {
        int t = 0;
#pragma unroll
        for (int i = 0; i < kWidenThreads / 32; ++i) t += red[it & 1][threadIdx.x][i];
        p.row_sum[row] = t;
      }
    }
  }
  if (abort_flag && threadIdx.x == 0) {
    // the copy issued for the next group lands before the block exits
    const int gn = blockIdx.x + (it + 1) * gridDim.x;
    if (gn < ngroups) mbar_wait(&bar[(it + 1) & 1], ((it + 1) >> 1) & 1, &abort_flag, nullptr,
                                                  100000000ull);
  }
}

struct WsLayout {
  size_t a16, b16, rs, total;
};
WsLayout ws_layout(int64_t M, int64_t K, int64_t N) {
  const int64_t Kp = padded_k(K);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  // A16, the row sums, then B16 last: a call with weights widened beforehand
  // needs the workspace only up to b16
  WsLayout w{};
  w.a16 = 0;
  w.rs = up((size_t)M * Kp * 2);
  w.b16 = w.rs + up((size_t)M * 4);
  w.total = w.b16 + up((size_t)N * Kp * 2);
  return w;
}

using UmmaKernel = void (*)(CUtensorMap, CUtensorMap, Int8UmmaParams);
// One instantiation per output conversion: S32, F32, S8, U8, then S8 and U8
// with a per-row activation scale; last the W8A16 and Q8 instances.
constexpr UmmaKernel kUmmaKernels[8] = {
    int8_umma_kernel<QMM_S32, false>, int8_umma_kernel<QMM_F32, false>, int8_umma_kernel<QMM_S8, false>,
    int8_umma_kernel<QMM_U8, false>,  int8_umma_kernel<QMM_S8, true>,   int8_umma_kernel<QMM_U8, true>,
    int8_umma_kernel<kW8Out, false>,  int8_umma_kernel<kQ8Out, false>};
constexpr int kW8Kernel = 6;
constexpr int kQ8Kernel = 7;

// Clusters of two that fit on the device at once (a GPC with an odd SM count
// leaves one SM over), with the kernel's shared-memory opt-in done: once per
// device, then read from the cache.
cudaError_t resident_pairs(int* pairs) {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) {
    *pairs = n;
    return cudaSuccess;
  }
  for (const auto k : kUmmaKernels) {
    err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  err = cudaFuncSetAttribute(int8_widen_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWidenMaxSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  if (cudaOccupancyMaxActiveClusters(&n, kUmmaKernels[0], &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    int sms = 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    n = sms / 2;
  }
  cache[dev].store(n, std::memory_order_relaxed);
  *pairs = n;
  return cudaSuccess;
}

}  // namespace

bool int8_umma_eligible(int64_t M, int64_t K, int64_t N) {
  (void)K;
  (void)N;
  return M >= kMinM;
}

size_t int8_umma_workspace_bytes(int64_t M, int64_t K, int64_t N, bool b16_given) {
  if (!int8_umma_eligible(M, K, N)) return 0;
  const WsLayout w = ws_layout(M, K, N);
  return b16_given ? w.b16 : w.total;
}

cudaError_t launch_int8_gemm_umma(const Int8GemmArgs& a, void* workspace, int32_t* dev_status,
                                  cudaStream_t stream, const __half* b16) {
  const WsLayout w = ws_layout(a.M, a.K, a.N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* A16 = reinterpret_cast<__half*>(ws + w.a16);
  // weights widened once beforehand (launch_widen_b_int8), or here on every call
  __half* B16 = b16 != nullptr ? const_cast<__half*>(b16) : reinterpret_cast<__half*>(ws + w.b16);
  int32_t* rs = a.need_rowsum ? reinterpret_cast<int32_t*>(ws + w.rs) : nullptr;
  const int Kp = (int)a.Kp;
  WidenParams wp{};
  wp.A = a.A;
  wp.lda = a.lda;
  wp.B = a.B;
  wp.A16 = A16;
  wp.B16 = B16;
  wp.row_sum = rs;
  wp.dev_status = dev_status;
  wp.M = a.M;
  wp.K = a.K;
  wp.N = b16 != nullptr ? 0 : a.N;   // the widen pass takes A's rows, and B's unless they come widened
  wp.Kp = Kp;
  wp.a_u8 = a.a_u8;
  wp.R = std::max(1, std::min(kWidenMaxRows, kWidenGroupBytes / Kp));
  const size_t wsmem = 128 + (size_t)2 * wp.R * Kp;
  const int ngroups = (wp.M + wp.N + wp.R - 1) / wp.R;
  int pairs = 0;
  cudaError_t err = resident_pairs(&pairs);
  if (err != cudaSuccess) return err;
  const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(8, (200u << 10) / wsmem));
  const int wgrid = std::min(ngroups, 2 * pairs * per_sm);
  int8_widen_kernel<<<wgrid, kWidenThreads, wsmem, stream>>>(wp);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, false, A16, (uint64_t)Kp, (uint64_t)a.M, (uint64_t)Kp * 2, kBK, kBM) ||
      !make_tmap_2d(&tmB, false, B16, (uint64_t)Kp, (uint64_t)a.N, (uint64_t)Kp * 2, kBK, kBNh))
    return cudaErrorInvalidValue;
  Int8UmmaParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.Kp = Kp;
  p.tiles_n = (a.N + kBN - 1) / kBN;
  p.ntiles = ((a.M + 2 * kBM - 1) / (2 * kBM)) * p.tiles_n;
  p.row_sum = rs;
  p.epi = a.epi;
  p.dev_status = dev_status;
  if (pairs > p.ntiles) pairs = p.ntiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;   // overlap the widen grid
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int ot = a.epi.out_type;
  const bool per_row_mq = (ot == QMM_S8 || ot == QMM_U8) && a.epi.s_x != nullptr && a.epi.s_x_stride != 0;
  const int which = ot == QMM_S32 ? 0 : ot == QMM_F32 ? 1 : (ot == QMM_S8 ? 2 : 3) + (per_row_mq ? 2 : 0);
  return cudaLaunchKernelEx(&cfg, kUmmaKernels[which], tmA, tmB, p);
}

cudaError_t launch_widen_b_int8(const int8_t* packed, int K, int N, __half* b16, int32_t* dev_status,
                                cudaStream_t stream) {
  WidenParams wp{};
  wp.B = packed;
  wp.B16 = b16;
  wp.dev_status = dev_status;
  wp.M = 0;
  wp.K = K;
  wp.N = N;
  wp.Kp = (int)padded_k(K);
  wp.R = std::max(1, std::min(kWidenMaxRows, kWidenGroupBytes / wp.Kp));
  const size_t wsmem = 128 + (size_t)2 * wp.R * wp.Kp;
  int pairs = 0;
  cudaError_t err = resident_pairs(&pairs);
  if (err != cudaSuccess) return err;
  const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(8, (200u << 10) / wsmem));
  const int wgrid = std::min((N + wp.R - 1) / wp.R, 2 * pairs * per_sm);
  int8_widen_kernel<<<wgrid, kWidenThreads, wsmem, stream>>>(wp);
  return cudaGetLastError();
}

size_t w8_umma_workspace_bytes(int64_t K, int64_t N) { return (size_t)N * padded_k(K) * 2; }

// W8A16 GEMM on the pair kernel: the weight codes are widened to bf16 (exact)
// into the workspace, the bf16 activations are read by TMA in place (rows
// past M and columns past K arrive as zeros), and each 1,024-k accumulator
// chunk is scaled by its block's per-row weight scale in the epilogue.
cudaError_t launch_w8_gemm_umma(const int8_t* codes, const float* scales, int N, int K,
                                const __nv_bfloat16* X, int64_t ldx, int M, float* Y, int64_t ldy,
                                void* workspace, int32_t* dev_status, cudaStream_t stream) {
  const int Kp = (int)padded_k(K);
  __nv_bfloat16* B16 = static_cast<__nv_bfloat16*>(workspace);
  WidenParams wp{};
  wp.B = codes;
  wp.B16 = reinterpret_cast<__half*>(B16);
  wp.dev_status = dev_status;
  wp.M = 0;
  wp.K = K;
  wp.N = N;
  wp.Kp = Kp;
  wp.b_bf16 = true;
  wp.R = std::max(1, std::min(kWidenMaxRows, kWidenGroupBytes / Kp));
  const size_t wsmem = 128 + (size_t)2 * wp.R * Kp;
  const int ngroups = (N + wp.R - 1) / wp.R;
  int pairs = 0;
  cudaError_t err = resident_pairs(&pairs);
  if (err != cudaSuccess) return err;
  const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(8, (200u << 10) / wsmem));
  const int wgrid = std::min(ngroups, 2 * pairs * per_sm);
  int8_widen_kernel<<<wgrid, kWidenThreads, wsmem, stream>>>(wp);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_w16_gemm_umma(B16, false, scales, (K + kChunkK - 1) / kChunkK, N, K, X, ldx, nullptr, M, Y, ldy,
                              dev_status, stream);
}

// The GEMM half of the above on 16-bit weights W16 [N][Kp] (Kp = K rounded
// up to 64, zero columns past K) that an earlier launch in the stream wrote:
// Y = sum over 1,024-k chunks c of scales[n][c] * (X W16^T restricted to c),
// times x_up[m] for f16 operands.  Launched as a programmatic dependent; the
// kernel waits for the previous grid before it reads W16 or X.
cudaError_t launch_w16_gemm_umma(const void* W16, bool f16, const float* scales, int nb, int N, int K,
                                 const void* X, int64_t ldx, const float* x_up, int M, float* Y, int64_t ldy,
                                 int32_t* dev_status, cudaStream_t stream) {
  const int Kp = (int)padded_k(K);
  int pairs = 0;
  cudaError_t err = resident_pairs(&pairs);
  if (err != cudaSuccess) return err;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, true, const_cast<void*>(X), (uint64_t)K, (uint64_t)M, (uint64_t)ldx * 2, kBK, kBM) ||
      !make_tmap_2d(&tmB, true, const_cast<void*>(W16), (uint64_t)Kp, (uint64_t)N, (uint64_t)Kp * 2, kBK, kBNh))
    return cudaErrorInvalidValue;
  Int8UmmaParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.Kp = Kp;
  p.tiles_n = (N + kBN - 1) / kBN;
  p.ntiles = ((M + 2 * kBM - 1) / (2 * kBM)) * p.tiles_n;
  p.epi.out = Y;
  p.epi.ldo = ldy;
  p.dev_status = dev_status;
  p.w8_scales = scales;
  p.w8_nb = nb;
  p.x_up = x_up;
  if (pairs > p.ntiles) pairs = p.ntiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;   // overlap the grid that wrote B16
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kUmmaKernels[f16 ? kQ8Kernel : kW8Kernel], tmA, tmB, p);
}

}  // namespace qmm
