// MUL_MAT_ID on q4_1 tiles: for every (token t, slot i), dst[t][i] = W_e . src1
// with e = ids[t * ld_ids + i] ("Zaya 8B Q4NX on the AMD NPU", "The bugs that
// were the work": the ids are a strided view, and the down projection reads a
// per-slot src1 row).  Weights are 32x256 q4_1 tiles, w = q * scale + min
// ("NPU engine: full ELFs, no xclbin", "Q4NX chunks").
//
// One CTA owns 128 weight rows of one expert and every (token, slot) pair
// routed to that expert, up to 64 pairs per pass.  Each weight is read from
// HBM once per pass and used for all of the pass's pairs: the grouped
// dispatch the pages credit for the MoE speed-up.
//
// Routing.  A one-CTA router writes per-expert offsets and the grouped
// (token, slot) list into the caller's workspace.  For decode-sized calls
// (T * n_used no more than one pair per thread) each CTA instead scans the
// ids itself, in pair order.
//
// Activations.  With a full workspace, a copy kernel first packs the rows of
// src1 in expert order, so that every CTA's B operand is a dense block that
// TMA loads whole.  With only the routing tables (the no-allocation entry
// point) or after the in-CTA scan, a loader warp gathers the rows itself with
// cp.async.
//
// The contraction runs on the 5th-generation tensor cores with the weights as
// the M = 128 side and the pairs as N (16..64).  The dequantised weights go
// from registers straight into TMEM, which tcgen05.mma reads as its A
// operand, so they never pass through shared memory; only the raw tiles and
// the gathered activations do.  Roles (224 threads):
//   warp 6     weight producer: TMA of whole tile columns (the 4 tiles of the
//              CTA's rows, codes and pairs as two boxes each) into a 3-stage
//              ring, 128-byte swizzle.
//   warps 0-3  transform, one weight row per lane (TMEM lane = row): read the
//              row's codes and pairs, w = bf16(q * s + m) with one rounding,
//              tcgen05.st of 128 k at a time into one of two TMEM A buffers.
//              After the last stage they drain the fp32 accumulator into Y.
//   warp 4     activation loader: TMA of the packed rows, or a cp.async
//              gather, into the 128-byte-swizzle K-major layout (3-stage
//              ring).
//   warp 5     TMEM owner; lane 0 issues tcgen05.mma (kind::f16, bf16).
// Every wait is bounded; a timeout sets the caller's status word and the CTA
// leaves cleanly.
#include <cuda_bf16.h>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kThreads = 224;
constexpr int kRows = 128;                          // weight rows per CTA (MMA M)
constexpr int kTok = 64;                            // pairs per pass (largest MMA N)
constexpr int kKC = 128;                            // K per MMA / activation stage
constexpr int kRawStages = 3;                       // weight ring, one tile column (256 k) per stage
constexpr int kBStages = 3;
constexpr int kAStages = 2;
constexpr int kCodeBox = 4096;                      // 32 code rows x 128 B
constexpr int kPairBox = 1024;                      // 8 pair rows x 128 B
constexpr int kRawBytes = 4 * (kCodeBox + kPairBox);   // 4 tile rows: codes [4][4 KB], then pairs [4][1 KB]
constexpr int kBAtomBytes = kTok * 128;             // 64 rows x 64 k bf16, 128-byte swizzle
constexpr int kBBytes = 2 * kBAtomBytes;            // 128 k per stage
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColD = 0;                       // accumulator: columns [0, 64)
constexpr uint32_t kColA = 64;                      // A buffer s: columns [64 + 64 s, 128 + 64 s)
constexpr int kLoaderLag = 2;                       // activation stages in flight before signalling
constexpr size_t kSmemBytes = 1024 + (size_t)kBStages * kBBytes + (size_t)kRawStages * kRawBytes + 256;
constexpr int kScanMaxPairs = kThreads;             // in-CTA scan: one id per thread
constexpr int kXBox = 16;                           // packed activations: TMA box rows

// Routing and activation source of one launch.
enum MoeMode { kScanGather = 0, kTableGather = 1, kTablePacked = 2 };

// mbarrier block after the two rings
constexpr int kBarWFull = 0;
constexpr int kBarWEmpty = kBarWFull + kRawStages;
constexpr int kBarAFull = kBarWEmpty + kRawStages;
constexpr int kBarAEmpty = kBarAFull + kAStages;
constexpr int kBarBFull = kBarAEmpty + kAStages;
constexpr int kBarBEmpty = kBarBFull + kBStages;
constexpr int kBarDFull = kBarBEmpty + kBStages;
constexpr int kBarDone = kBarDFull + 1;
constexpr int kNumBars = kBarDone + 1;
static_assert(kNumBars * 8 + 8 <= 256, "barrier block");

struct MoeParams {
  int64_t tiles_per_expert;
  int N, K;
  const __nv_bfloat16* X;
  int64_t ldx_token, ldx_slot;
  const int32_t* ids;
  int64_t ld_ids;
  int n_used, T, n_expert;
  float* Y;
  int64_t ldy_token, ldy_slot;
  const int32_t* offsets;   // router mode only
  const int32_t* pairs;     // router mode only
  int32_t* dev_status;
};

// q * s + m in bf16 from a (128 + q) pair: the subtraction is exact, the fma
// rounds once.
__device__ __forceinline__ uint32_t dequant2(uint32_t q2_biased, uint32_t s2, uint32_t m2) {
  __nv_bfloat162 q = *reinterpret_cast<__nv_bfloat162*>(&q2_biased);
  const uint32_t c128 = 0x43004300u;
  q = __hsub2(q, *reinterpret_cast<const __nv_bfloat162*>(&c128));
  const __nv_bfloat162 w =
      __hfma2(q, *reinterpret_cast<__nv_bfloat162*>(&s2), *reinterpret_cast<__nv_bfloat162*>(&m2));
  return *reinterpret_cast<const uint32_t*>(&w);
}

// Exclusive prefix of `v` over the CTA; `total` gets the sum.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int s = wsum[w];
    before += (w < warp) ? s : 0;
    total += s;
  }
  __syncthreads();
  return before + incl - v;
}

__device__ __forceinline__ void pair_offsets(const MoeParams& p, int pr, int64_t& xo, int64_t& yo) {
  const int tok = pr / p.n_used, slot = pr % p.n_used;
  xo = (int64_t)tok * p.ldx_token + (int64_t)slot * p.ldx_slot;
  yo = (int64_t)tok * p.ldy_token + (int64_t)slot * p.ldy_slot;
}

// One weight stage: the CTA's (up to) 4 tiles of tile column tc.
__device__ __forceinline__ bool produce_weights(const CUtensorMap* tmC, const CUtensorMap* tmP, const MoeParams& p,
                                                int e, int n0, int tc, int gws, uint32_t raw0, uint64_t* w_full,
                                                uint64_t* w_empty, volatile int* abort_flag) {
  const int slot = gws % kRawStages;
  if (!mbar_wait(&w_empty[slot], ((gws / kRawStages) & 1) ^ 1, abort_flag, p.dev_status)) return false;
  const int TC = p.K / 256;
  int live = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) live += (n0 + 32 * q < p.N) ? 1 : 0;
  mbar_arrive_expect_tx(&w_full[slot], (uint32_t)live * (kCodeBox + kPairBox));
  const uint32_t sb = raw0 + slot * kRawBytes;
  for (int q = 0; q < live; ++q) {
    const int tile = (int)((int64_t)e * p.tiles_per_expert + (int64_t)((n0 >> 5) + q) * TC + tc);
    tma_load_3d(sb + q * kCodeBox, tmC, &w_full[slot], 0, 0, tile);
    tma_load_3d(sb + 4 * kCodeBox + q * kPairBox, tmP, &w_full[slot], 0, 32, tile);
  }
  return true;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 2)
q4_moe_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
              const __grid_constant__ CUtensorMap tmX, const MoeParams p) {
  constexpr bool kScan = kMode == kScanGather;
  constexpr bool kPacked = kMode == kTablePacked;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int64_t xoff[kTok], yoff[kTok];
  __shared__ int wsum[kThreads / 32];
  uint8_t* smem = smem_align(smem_raw, 1024);
  const uint32_t sB0 = smem_u32(smem);                              // [kBStages][2 atoms]
  const uint32_t raw0 = sB0 + kBStages * kBBytes;                   // [kRawStages][codes | pairs]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBStages * kBBytes + kRawStages * kRawBytes);
  uint64_t* w_full = bars + kBarWFull;     // TMA bytes
  uint64_t* w_empty = bars + kBarWEmpty;   // 4 transform-warp arrivals
  uint64_t* a_full = bars + kBarAFull;     // 4 transform-warp arrivals
  uint64_t* a_empty = bars + kBarAEmpty;   // MMA commit
  uint64_t* b_full = bars + kBarBFull;     // loader arrival (with TMA bytes when packed)
  uint64_t* b_empty = bars + kBarBEmpty;   // MMA commit
  uint64_t* d_full = bars + kBarDFull;     // once per pass, MMA commit
  uint64_t* done = bars + kBarDone;        // teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y, n0 = blockIdx.x * kRows;
  const int nks = p.K / kKC;     // MMA stages per pass
  const int TC = p.K / 256;      // weight stages per pass
  const int npairs = p.T * p.n_used;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 4);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(d_full, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // When most experts receive pairs, the first weight stages are fetched
  // before the routing is known: they do not depend on it.
  const bool early = npairs >= p.n_expert;
  int w_issued = 0;   // weight stages of pass 0 already issued (producer lane only)
  if (warp == 6 && lane == 0 && early) {
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmP);
    for (; w_issued < kRawStages && w_issued < TC; ++w_issued)
      produce_weights(&tmC, &tmP, p, e, n0, w_issued, w_issued, raw0, w_full, w_empty, abort_flag);
  }

  // ---- this expert's pairs ----
  uint32_t mask = 0;
  int first = 0, total = 0, rank0 = 0;
  if (kScan) {
    first = threadIdx.x;   // one pair per thread (npairs <= kThreads)
    if (first < npairs) {
      const int id = p.ids[(int64_t)(first / p.n_used) * p.ld_ids + (first % p.n_used)];
      if (id == e) mask = 1u;
      if ((id < 0 || id >= p.n_expert) && blockIdx.x == 0 && blockIdx.y == 0)
        set_status(p.dev_status, QMM_ERR_BAD_EXPERT_ID);
    }
    rank0 = cta_exclusive_scan(__popc(mask), wsum, total);
  } else {
    first = p.offsets[e];
    total = p.offsets[e + 1] - first;
  }
  if (total == 0) {
    // no TMA write may land after the CTA has left
    if (warp == 6 && lane == 0)
      for (int s = 0; s < w_issued; ++s) mbar_wait(&w_full[s], 0, abort_flag, p.dev_status);
    return;
  }

  if (warp == 5) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  int pass = 0;
  for (int pass0 = 0; pass0 < total; pass0 += kTok, ++pass) {
    const int nt = min(kTok, total - pass0);
    const int ncol = (nt + 15) & ~15;
    if (kScan) {
      uint32_t m = mask;
      int rk = rank0;
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        if (rk >= pass0 && rk < pass0 + kTok) pair_offsets(p, first + j, xoff[rk - pass0], yoff[rk - pass0]);
        ++rk;
      }
    } else {
      for (int c = threadIdx.x; c < nt; c += kThreads)
        pair_offsets(p, p.pairs[first + pass0 + c], xoff[c], yoff[c]);
    }
    __syncthreads();

    if (warp < 4) {
      // ---- transform: raw tiles -> bf16 weights in TMEM ----
      const int n = n0 + 32 * warp + lane;
      const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
      for (int tc = 0; tc < TC && ok; ++tc) {
        const int gws = pass * TC + tc, slot = gws % kRawStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&w_full[slot], (gws / kRawStages) & 1, abort_flag, p.dev_status))) {
          ok = false;
          break;
        }
        const uint32_t cb = raw0 + slot * kRawBytes + warp * kCodeBox + lane * 128;
        uint4 cw[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) cw[b] = lds128(cb + 16 * (b ^ (lane & 7)));
        const uint32_t pb = raw0 + slot * kRawBytes + 4 * kCodeBox + warp * kPairBox + (lane >> 2) * 128;
        const uint4 pr0 = lds128(pb + 16 * ((2 * (lane & 3)) ^ ((lane >> 2) & 7)));
        const uint4 pr1 = lds128(pb + 16 * ((2 * (lane & 3) + 1) ^ ((lane >> 2) & 7)));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int gs = pass * nks + 2 * tc + h, as = gs % kAStages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&a_empty[as], ((gs / kAStages) & 1) ^ 1, abort_flag, p.dev_status))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const int b = 4 * h + 2 * hh + bb;
              const uint32_t pair = u4_get(b < 4 ? pr0 : pr1, b & 3);
              const uint32_t s2 = __byte_perm(pair, 0, 0x1010), m2 = __byte_perm(pair, 0, 0x3232);
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const uint32_t word = u4_get(cw[b], t);
#pragma unroll
                for (int i = 0; i < 4; ++i) v[16 * bb + 4 * t + i] = dequant2(q4_pair_biased(word, i), s2, m2);
              }
            }
            tmem_st32(trow + kColA + 64 * as + 32 * hh, v);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[as]);
        }
        // Every lane has consumed its loads of this raw slot (the values went
        // into TMEM above), so the producer may refill it.
        __syncwarp();
        if (lane == 0) mbar_arrive(&w_empty[slot]);
      }
      // ---- epilogue: fp32 accumulator -> Y (lane = weight row, column = pair) ----
      if (ok && __all_sync(0xffffffffu, mbar_wait(d_full, pass & 1, abort_flag, p.dev_status))) {
        tc_fence_after();
        const bool live = n < p.N;
        for (int c0 = 0; c0 < ncol; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(trow + kColD + c0, v);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < nt) p.Y[yoff[c0 + i] + n] = __uint_as_float(v[i]);
          }
        }
        tc_fence_before();
      } else {
        ok = false;
      }
    } else if (warp == 4) {
      // ---- activation loader ----
      if (kPacked) {
        if (lane == 0) {
          if (pass == 0) tma_prefetch_desc(&tmX);
          const int row0 = first + pass0;
          for (int ks = 0; ks < nks && ok; ++ks) {
            const int gs = pass * nks + ks, bs = gs % kBStages;
            if (!mbar_wait(&b_empty[bs], ((gs / kBStages) & 1) ^ 1, abort_flag, p.dev_status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&b_full[bs], (uint32_t)(2 * ncol * 128));
            const uint32_t sb = sB0 + bs * kBBytes;
#pragma unroll
            for (int at = 0; at < 2; ++at)
              for (int c0 = 0; c0 < ncol; c0 += kXBox)
                tma_load_2d_u32(sb + at * kBAtomBytes + (c0 >> 3) * 1024, &tmX, &b_full[bs], ks * kKC + 64 * at,
                                row0 + c0);
          }
        }
        __syncwarp();
      } else {
        for (int ks = 0; ks < nks + kLoaderLag && ok; ++ks) {
          if (ks < nks) {
            const int gs = pass * nks + ks, bs = gs % kBStages;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&b_empty[bs], ((gs / kBStages) & 1) ^ 1, abort_flag, p.dev_status))) {
              ok = false;
              break;
            }
            const uint32_t sb = sB0 + bs * kBBytes;
            for (int i = lane; i < ncol * 16; i += 32) {
              const int c = i >> 4, ch = i & 15;
              const bool valid = c < nt;
              const __nv_bfloat16* src = valid ? p.X + xoff[c] + (int64_t)ks * kKC + 8 * ch : p.X;
              const uint32_t dst = sb + (ch >> 3) * kBAtomBytes + (c >> 3) * 1024 + (c & 7) * 128 +
                                   (uint32_t)(((ch & 7) ^ (c & 7)) << 4);
              cp_async16_zfill(dst, src, valid ? 16u : 0u);
            }
          }
          cp_async_commit();
          if (ks >= kLoaderLag) {
            cp_async_wait<kLoaderLag>();
            fence_proxy_async_smem();   // generic-proxy writes -> tcgen05 reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_full[(pass * nks + ks - kLoaderLag) % kBStages]);
          }
        }
      }
    } else if (warp == 5) {
      // ---- MMA issuer ----
      if (lane == 0) {
        const uint32_t idesc = idesc_f16(kRows, ncol, true);
        for (int ks = 0; ks < nks && ok; ++ks) {
          const int gs = pass * nks + ks, as = gs % kAStages, bs = gs % kBStages;
          if (!mbar_wait(&a_full[as], (gs / kAStages) & 1, abort_flag, p.dev_status) ||
              !mbar_wait(&b_full[bs], (gs / kBStages) & 1, abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = sB0 + bs * kBBytes;
#pragma unroll
          for (int j = 0; j < kKC / 16; ++j)
            umma_f16_ta(tmem + kColD, tmem + kColA + 64 * as + 8 * j,
                        desc_kmajor_sw128(sb + (j >> 2) * kBAtomBytes + 32 * (j & 3)), idesc,
                        (ks > 0 || j > 0) ? 1u : 0u);
          umma_commit(&a_empty[as]);
          umma_commit(&b_empty[bs]);
        }
        if (ok) umma_commit(d_full);
      }
      __syncwarp();
    } else {
      // ---- weight producer ----
      if (lane == 0) {
        if (pass > 0 || !early) {
          tma_prefetch_desc(&tmC);
          tma_prefetch_desc(&tmP);
        }
        for (int tc = (pass == 0 ? w_issued : 0); tc < TC && ok; ++tc)
          ok = produce_weights(&tmC, &tmP, p, e, n0, tc, pass * TC + tc, raw0, w_full, w_empty, abort_flag);
      }
      __syncwarp();
    }
    __syncthreads();   // accumulator drained; routing slots and rings free for the next pass
  }

  // ---- teardown ----
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 6 && lane == 0 && *abort_flag) {
    // a stage the transform never consumed may still be in flight
    const int last = pass * TC;
    for (int g = last > kRawStages ? last - kRawStages : 0; g < last; ++g)
      mbar_wait(&w_full[g % kRawStages], (g / kRawStages) & 1, abort_flag, nullptr, 100000000ull) ||
          mbar_try_wait(&w_full[g % kRawStages], (g / kRawStages) & 1);
  }
  if (kPacked && warp == 4 && lane == 0 && *abort_flag) {
    // activation loads of the last stages may still be in flight
    const int last = pass * nks;
    for (int g = last > kBStages ? last - kBStages : 0; g < last; ++g)
      mbar_wait(&b_full[g % kBStages], (g / kBStages) & 1, abort_flag, nullptr, 100000000ull) ||
          mbar_try_wait(&b_full[g % kBStages], (g / kBStages) & 1);
  }
  if (warp == 5) {
    if (lane == 0) {
      umma_commit(done);   // every MMA of this CTA has completed before TMEM is freed
      mbar_wait(done, 0, abort_flag, nullptr, 100000000ull) || mbar_try_wait(done, 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

// Rows r of the packed activations are the pairs in expert order:
// Xp[r][:] = src1 of pairs[r].  Eight rows per CTA, 16 bytes per thread and row.
constexpr int kPermRows = 8;
__global__ void __launch_bounds__(256)
moe_permute_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx_token, int64_t ldx_slot, int n_used,
                   const int32_t* __restrict__ offsets, int n_expert, const int32_t* __restrict__ pairs, int K,
                   __nv_bfloat16* __restrict__ Xp) {
  const int total = offsets[n_expert];
  const int chunks = K / 8;
#pragma unroll
  for (int i = 0; i < kPermRows; ++i) {
    const int r = blockIdx.x * kPermRows + i;
    if (r >= total) break;
    const int pr = pairs[r];
    const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)(pr / n_used) * ldx_token +
                                                      (int64_t)(pr % n_used) * ldx_slot);
    uint4* dst = reinterpret_cast<uint4*>(Xp + (int64_t)r * K);
    for (int c = threadIdx.x; c < chunks; c += 256) dst[c] = ldg128(src + c);
  }
}

template <int kMode>
cudaError_t launch_grouped(const CUtensorMap& tmC, const CUtensorMap& tmP, const CUtensorMap& tmX,
                           const MoeParams& p, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(q4_moe_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)((p.N + kRows - 1) / kRows), (unsigned)p.n_expert);
  q4_moe_kernel<kMode><<<grid, kThreads, kSmemBytes, stream>>>(tmC, tmP, tmX, p);
  return cudaGetLastError();
}

}  // namespace

size_t q4_moe_table_bytes(int64_t n_expert, int64_t n_used, int64_t T) {
  const size_t off = ((size_t)(n_expert + 1) * 4 + 255) / 256 * 256;
  return off + ((size_t)(T * n_used) * 4 + 255) / 256 * 256;
}

size_t q4_moe_workspace_bytes(int64_t n_expert, int64_t n_used, int64_t T, int64_t K) {
  return q4_moe_table_bytes(n_expert, n_used, T) + (size_t)(T * n_used) * (size_t)K * 2;
}

cudaError_t launch_q4_moe(const Q4MoEArgs& a, cudaStream_t stream) {
  MoeParams p{};
  p.tiles_per_expert = (int64_t)(a.N / 32) * (a.K / 256);
  p.N = a.N;
  p.K = a.K;
  p.X = a.X;
  p.ldx_token = a.ldx_token;
  p.ldx_slot = a.ldx_slot;
  p.ids = a.ids;
  p.ld_ids = a.ld_ids;
  p.n_used = a.n_used;
  p.T = a.T;
  p.n_expert = a.n_expert;
  p.Y = a.Y;
  p.ldy_token = a.ldy_token;
  p.ldy_slot = a.ldy_slot;
  p.dev_status = a.dev_status;
  const uint64_t n_tiles = (uint64_t)a.n_expert * (uint64_t)p.tiles_per_expert;
  if (n_tiles > (uint64_t)INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tmC, tmP, tmX;
  if (!make_tmap_q4_tiles(&tmC, a.tiles, n_tiles, 32) || !make_tmap_q4_tiles(&tmP, a.tiles, n_tiles, 8))
    return cudaErrorInvalidValue;
  const int npairs = a.T * a.n_used;
  if (npairs <= kScanMaxPairs) return launch_grouped<kScanGather>(tmC, tmP, tmC, p, stream);
  const size_t smem = (size_t)a.n_expert * 2 * sizeof(int);
  moe_route_kernel<<<1, 1024, smem, stream>>>(a.ids, a.ld_ids, a.n_used, a.T, a.n_expert, a.offsets,
                                              a.pairs, a.dev_status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  p.offsets = a.offsets;
  p.pairs = a.pairs;
  if (a.xperm == nullptr) return launch_grouped<kTableGather>(tmC, tmP, tmC, p, stream);
  moe_permute_kernel<<<(unsigned)((npairs + kPermRows - 1) / kPermRows), 256, 0, stream>>>(
      a.X, a.ldx_token, a.ldx_slot, a.n_used, a.offsets, a.n_expert, a.pairs, a.K, a.xperm);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (!make_tmap_2d(&tmX, true, a.xperm, (uint64_t)a.K, (uint64_t)npairs, (uint64_t)a.K * 2, 64, kXBox))
    return cudaErrorInvalidValue;
  return launch_grouped<kTablePacked>(tmC, tmP, tmX, p, stream);
}

}  // namespace qmm
