// q4 GEMMs on the 5th-generation tensor cores: the prefill GEMM and
// MUL_MAT_ID.  Weights are 32x256 q4_1 tiles, w = q * scale + min ("NPU
// engine: full ELFs, no xclbin", "Q4NX chunks"; "Zaya 8B Q4NX on the AMD NPU",
// round 26).
//
// MUL_MAT_ID: for every (token t, slot i), dst[t][i] = W_e . src1 with
// e = ids[t * ld_ids + i] ("Zaya 8B Q4NX on the AMD NPU", "The bugs that were
// the work": the ids are a strided view, and the down projection reads a
// per-slot src1 row).  The prefill GEMM is the same kernel with one "expert"
// and the M rows of X in order; the pages' lesson for prefill (round 25o) is
// to reuse each dequantised weight across many activation columns.
//
// Work is cut into units of 128 weight rows of one expert; a unit's jobs are
// its expert's (token, slot) pairs, up to kTok (64, or 128 for a large dense
// M) per job.  Each weight is read from HBM once per job and used for all of
// the job's pairs: the grouped dispatch the pages credit for the MoE
// speed-up.  The grid is persistent (two CTAs per SM for MUL_MAT_ID, one for
// the dense GEMM); every role walks the CTA's units in the same order, and
// the pipelines run on across unit boundaries, so the next unit's weights
// stream in while the current one finishes.  The fp32 accumulator is double
// buffered in TMEM, so a job's epilogue overlaps the next job's MMAs.
//
// Routing.  A routing grid writes per-expert offsets and the grouped
// (token, slot) list into the caller's workspace, in pair order inside each
// expert.
//
// Activations.  With a full workspace, a packing grid (the routing grid's
// programmatic dependent) copies the rows of src1 in expert order, so that
// every job's B operand is a dense block that TMA loads whole.  With only the
// routing tables (the no-allocation entry point) a loader warp gathers the
// rows with cp.async.  The grouped kernel is launched as the last grid's
// programmatic dependent, so it starts while that grid still runs.
//
// Operands are f16: each weight is formed once as f16(q * s + m) (one
// rounding, 2^-11 relative), and each activation row is stored in f16 after a
// power-of-two scale that makes the conversion exact and overflow-free; the
// epilogue multiplies every output column back by its row's inverse scale.
// The activation rows are converted by the grid before this one (the packing
// grid, or for the dense GEMM a conversion grid); in the gather mode the
// loader converts each gathered stage in place in shared memory.
//
// The contraction runs on the 5th-generation tensor cores with the weights as
// the M = 128 side and the pairs as N (16..kTok).  The dequantised weights go
// from registers straight into TMEM, which tcgen05.mma reads as its A
// operand, so they never pass through shared memory; only the raw tiles and
// the activations do.  TMEM: two accumulators of kTok columns, then two or
// four A buffers of 64 columns (128 k).  Roles, in warp order:
//   transform  four or eight warps; warp (q, h) owns TMEM lane quarter q (one
//              weight row per lane) and, with eight, 64-k half h of every
//              128-k stage: it reads the rows' codes and pairs, forms
//              w = f16(q * s + m) with one rounding, and stores the stage into
//              an A buffer (tcgen05.st).  With four, they also drain each
//              job's accumulator into Y.
//   epilogue   (one CTA per SM) four warps draining accumulators into Y.
//   loader     TMA of the packed rows (or of X for the dense GEMM), or a
//              cp.async gather, into the 128-byte-swizzle K-major layout.
//   MMA        TMEM owner; lane 0 issues tcgen05.mma (kind::f16, f16 operands).
//   producer   TMA of whole tile columns: one box for the unit's 4 tiles'
//              codes, one for their pairs, 128-byte swizzle.
// Every wait is bounded; a timeout sets the caller's status word and the CTA
// leaves cleanly.
#include <cuda_bf16.h>

#include <algorithm>

#include "f16_operands.cuh"
#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kRows = 128;                          // weight rows per unit (MMA M)
constexpr int kKC = 128;                            // K per MMA / activation stage
constexpr int kRawStagesMax = 4;                    // weight ring, one tile column (256 k) per stage
constexpr int kBStagesMax = 4;
constexpr int kAStagesMax = 4;
constexpr int kCodeBox = 4096;                      // 32 code rows x 128 B
constexpr int kPairBox = 1024;                      // 8 pair rows x 128 B
constexpr int kRawBytes = 4 * (kCodeBox + kPairBox);   // 4 tile rows: codes [4][4 KB], then pairs [4][1 KB]
constexpr int kLoaderLag = 2;                       // gathered activation stages in flight before signalling

// Sizes that follow from the largest job width kTok (the MMA's N): two fp32
// accumulators of kTok columns, then two A buffers of 64 columns in TMEM;
// activation stages of kTok rows x 128 k.
// Two CTA layouts.  Two CTAs per SM (MUL_MAT_ID: small jobs, so two units
// in flight per SM hide each other's fill and drain): four transform warps
// that also drain the accumulator, two A buffers, TMEM 256 columns.  One CTA
// per SM (dense prefill): eight transform warps, four epilogue warps, four A
// buffers, TMEM 512 columns, deeper rings.  kTok is the widest job (MMA N).
template <int kTok, int kCtas>
struct Lay {
  static constexpr int kXW = kCtas == 2 ? 4 : 8;           // transform warps
  static constexpr bool kSepEpi = kCtas == 1;              // epilogue warps of their own
  static constexpr int kWarps = kXW + (kSepEpi ? 4 : 0) + 3;
  // TMEM A buffers of 64 columns (128 k); a 192-token job's two accumulators
  // leave room for two
  static constexpr int kAStages = (kCtas == 2 || kTok > 128) ? 2 : 4;
  static constexpr int kRawStages = kCtas == 2 ? 3 : (kTok == 64 ? 4 : 3);
  static constexpr int kBStages = (kCtas == 2 || kTok > 128) ? 3 : 4;   // activation ring depth
  static constexpr int kBAtomBytes = kTok * 128;           // kTok rows x 64 k f16, 128-byte swizzle
  static constexpr int kBBytes = 2 * kBAtomBytes;          // 128 k per stage
  static constexpr uint32_t kColA = 2 * kTok;              // after the two accumulators
  static constexpr uint32_t kTmemCols = kCtas == 2 ? 256 : 512;
  static constexpr size_t kSmemBytes = 1024 + (size_t)kBStages * kBBytes + (size_t)kRawStages * kRawBytes + 256;
  static_assert(kColA + 64 * kAStages <= kTmemCols, "TMEM budget");
};

// Activation source of one launch: MUL_MAT_ID with the routing tables only
// (gather), MUL_MAT_ID with packed rows, or a dense GEMM (one "expert", all
// M rows of X in order).
enum MoeMode { kTableGather = 0, kTablePacked = 1, kDense = 2 };

// mbarrier block after the two rings
constexpr int kBarWFull = 0;
constexpr int kBarWEmpty = kBarWFull + kRawStagesMax;
constexpr int kBarAFull = kBarWEmpty + kRawStagesMax;
constexpr int kBarAEmpty = kBarAFull + kAStagesMax;
constexpr int kBarBFull = kBarAEmpty + kAStagesMax;
constexpr int kBarBEmpty = kBarBFull + kBStagesMax;
constexpr int kBarDFull = kBarBEmpty + kBStagesMax;
constexpr int kBarDEmpty = kBarDFull + 2;
constexpr int kBarDone = kBarDEmpty + 2;
constexpr int kNumBars = kBarDone + 1;
static_assert(kNumBars * 8 + 8 <= 256, "barrier block");

struct MoeParams {
  int64_t tiles_per_expert;
  int N, K;
  const __nv_bfloat16* X;   // gather mode: the bf16 src1 rows
  int64_t ldx_token, ldx_slot;
  int n_used, n_expert, npairs;
  int n_units, nrb;         // units = sets x experts x 128-row blocks, unit u = (set * E + e) * nrb + row block
  int units_per_set;        // experts x row blocks (MUL_MAT_ID); the dense GEMM has one set
  float* Y;
  float* Y2;                // second weight set's output (the gate/up pair), else null
  int64_t ldy_token, ldy_slot;
  const int32_t* offsets;   // [n_expert + 1]; null for the dense GEMM
  const int32_t* pairs;     // grouped (token, slot) ids
  int dense_rows;           // dense GEMM: M
  int dense_chunks;         // dense GEMM: token chunks of kTok per row block; unit u = rb * chunks + chunk
  const float* xup;         // inverse activation-row scales: per token (dense) or per grouped rank
  int32_t* dev_status;
};

__device__ __forceinline__ void pair_offsets(const MoeParams& p, int pr, int64_t& xo, int64_t& yo) {
  const int tok = pr / p.n_used, slot = pr % p.n_used;
  xo = (int64_t)tok * p.ldx_token + (int64_t)slot * p.ldx_slot;
  yo = (int64_t)tok * p.ldy_token + (int64_t)slot * p.ldy_slot;
}

// The CTA's jobs, in the same order for every role: units blockIdx.x,
// blockIdx.x + gridDim.x, ...; each unit's pairs in passes of up to kTok.
// Units without pairs are skipped.
// Weight set, expert and first weight row of unit u.
__device__ __forceinline__ void unit_rows(const MoeParams& p, int u, int& set, int& e, int& n0) {
  if (p.offsets == nullptr) {   // dense: u = row block * chunks + token chunk
    set = 0;
    e = 0;
    n0 = (u / p.dense_chunks) * kRows;
  } else {                      // MUL_MAT_ID: u = (set * experts + expert) * row blocks + row block
    set = u >= p.units_per_set ? 1 : 0;
    const int us = u - set * p.units_per_set;
    e = us / p.nrb;
    n0 = (us - e * p.nrb) * kRows;
  }
}

template <int kTok>
struct Jobs {
  int u, set, e, n0, first, total, pass0;
  __device__ Jobs() : u((int)blockIdx.x - (int)gridDim.x), set(0), e(0), n0(0), first(0), total(0), pass0(0) {}
  __device__ bool next(const MoeParams& p) {
    pass0 += kTok;
    while (pass0 >= total) {
      u += gridDim.x;
      if (u >= p.n_units) return false;
      unit_rows(p, u, set, e, n0);
      if (p.offsets == nullptr) {   // one job: this unit's chunk of rows of X
        first = 0;
        pass0 = (u % p.dense_chunks) * kTok;
        total = min(p.dense_rows, pass0 + kTok);
      } else {
        first = p.offsets[e];
        total = p.offsets[e + 1] - first;
        pass0 = 0;
      }
    }
    return true;
  }
  __device__ int nt() const { return min(kTok, total - pass0); }
  __device__ int ncol() const { return (nt() + 15) & ~15; }
};

// One weight stage: the unit's (up to) 4 tiles of tile column tc.
template <int kRawStages>
__device__ __forceinline__ bool produce_weights(const CUtensorMap* tmC, const CUtensorMap* tmP, const MoeParams& p,
                                                int e, int n0, int tc, int gws, uint32_t raw0, uint64_t* w_full,
                                                uint64_t* w_empty, volatile int* abort_flag) {
  const int slot = gws % kRawStages;
  if (!mbar_wait(&w_empty[slot], ((gws / kRawStages) & 1) ^ 1, abort_flag, p.dev_status)) return false;
  // one box of the unit's 4 tile rows for the codes, one for the pairs; tile
  // rows past the expert's last (a partial unit) load junk that no one stores
  mbar_arrive_expect_tx(&w_full[slot], (uint32_t)(4 * (kCodeBox + kPairBox)));
  const uint32_t sb = raw0 + slot * kRawBytes;
  const int trow = (int)((int64_t)e * (p.N / 32) + (n0 >> 5));
  tma_load_4d(sb, tmC, &w_full[slot], 0, 0, tc, trow);
  tma_load_4d(sb + 4 * kCodeBox, tmP, &w_full[slot], 0, 32, tc, trow);
  return true;
}

// kN accumulator columns (one TMEM load) of one lane's weight row n into Y,
// each times its column's inverse activation scale.  The scales are read four
// at a time (every lane reads the same address); dense rows of Y are
// consecutive tokens, so the output pointer steps by ldy.
template <int kN, int kMode>
__device__ __forceinline__ void epilogue_store(const MoeParams& p, const uint32_t (&v)[kN], int c0, int nt, bool live,
                                               float* ycol0, const int64_t* yoff_q, const float* ysc_q) {
  float sc[kN];
#pragma unroll
  for (int j = 0; j < kN / 4; ++j) {
    const float4 f = *reinterpret_cast<const float4*>(ysc_q + c0 + 4 * j);
    sc[4 * j] = f.x;
    sc[4 * j + 1] = f.y;
    sc[4 * j + 2] = f.z;
    sc[4 * j + 3] = f.w;
  }
  if (!live) return;
  if (kMode == kDense) {
    float* yp = ycol0 + (int64_t)c0 * p.ldy_token;
#pragma unroll
    for (int i = 0; i < kN; ++i) {
      if (c0 + i < nt) *yp = __uint_as_float(v[i]) * sc[i];
      yp += p.ldy_token;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kN / 2; ++j) {
      const longlong2 o = *reinterpret_cast<const longlong2*>(yoff_q + c0 + 2 * j);
      if (c0 + 2 * j < nt) ycol0[o.x] = __uint_as_float(v[2 * j]) * sc[2 * j];
      if (c0 + 2 * j + 1 < nt) ycol0[o.y] = __uint_as_float(v[2 * j + 1]) * sc[2 * j + 1];
    }
  }
}

// Drain job `jb`'s accumulator (buffer njobs & 1) for TMEM lane quarter q into
// Y: lane = weight row, column = pair.  Returns false after an abort.
template <int kMode, int kTok>
__device__ __forceinline__ bool epilogue_job(const MoeParams& p, const Jobs<kTok>& jb, int q, int lane, uint32_t tmem,
                                             int njobs, uint64_t* d_full, uint64_t* d_empty, int64_t* yoff_q,
                                             float* ysc_q, volatile int* abort_flag) {
  const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
  const int n = jb.n0 + 32 * q + lane;
  const int nt = jb.nt(), ncol = jb.ncol();
  // column c is token pass0 + c (dense) or grouped rank first + pass0 + c
  const int r0 = kMode == kDense ? jb.pass0 : jb.first + jb.pass0;
  for (int c = lane; c < nt; c += 32) {
    if (kMode != kDense) {
      int64_t xo;
      pair_offsets(p, p.pairs[jb.first + jb.pass0 + c], xo, yoff_q[c]);
    }
    ysc_q[c] = p.xup[r0 + c];
  }
  __syncwarp();
  const int db = njobs & 1;
  if (!__all_sync(0xffffffffu, mbar_wait(&d_full[db], (njobs >> 1) & 1, abort_flag, p.dev_status))) return false;
  tc_fence_after();
  const bool live = n < p.N;
  float* ycol0 = (jb.set ? p.Y2 : p.Y) + n + (kMode == kDense ? (int64_t)jb.pass0 * p.ldy_token : 0);
  const uint32_t tacc = trow + (uint32_t)(kTok * db);
  int c0 = 0;
  for (; c0 + 32 <= ncol; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tacc + c0, v);
    tmem_wait_ld();
    epilogue_store<32, kMode>(p, v, c0, nt, live, ycol0, yoff_q, ysc_q);
  }
  if (c0 < ncol) {   // ncol is a multiple of 16
    uint32_t v[16];
    tmem_ld16(tacc + c0, v);
    tmem_wait_ld();
    epilogue_store<16, kMode>(p, v, c0, nt, live, ycol0, yoff_q, ysc_q);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&d_empty[db]);
  return true;
}

template <int kMode, int kTok, int kCtas>
__global__ void __launch_bounds__(32 * Lay<kTok, kCtas>::kWarps, kCtas)
q4_tc_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
             const __grid_constant__ CUtensorMap tmC2, const __grid_constant__ CUtensorMap tmP2,
             const __grid_constant__ CUtensorMap tmX, const MoeParams p) {
  constexpr bool kPacked = kMode != kTableGather;   // activations by TMA
  using L = Lay<kTok, kCtas>;
  constexpr int kXW = L::kXW;
  constexpr int kRawStages = L::kRawStages;
  constexpr int kAStages = L::kAStages;
  constexpr int kBStages = L::kBStages;
  constexpr int kBAtomBytes = L::kBAtomBytes;
  constexpr int kBBytes = L::kBBytes;
  constexpr uint32_t kColA = L::kColA;
  constexpr uint32_t kTmemCols = L::kTmemCols;
  // warps 0 .. kXW-1 transform (kXW / 4 per TMEM lane quarter), then (one CTA
  // per SM) four epilogue warps, then the activation loader, the MMA issuer
  // and the weight producer
  constexpr int kHalves = kXW / 4;
  constexpr int kWEpi = kXW, kWLoad = kXW + (L::kSepEpi ? 4 : 0), kWMma = kWLoad + 1, kWProd = kWLoad + 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int64_t xoff[kMode == kTableGather ? kTok : 1];   // gather mode: the loader's rows of the current job
  __shared__ __align__(16) int64_t yoff[4][kTok];   // each epilogue warp's output rows of its current job
  __shared__ __align__(16) float ysc[4][kTok];      // and their inverse activation scales
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
  uint64_t* d_full = bars + kBarDFull;     // [2] per job, MMA commit
  uint64_t* d_empty = bars + kBarDEmpty;   // [2] per job, 4 epilogue-warp arrivals
  uint64_t* done = bars + kBarDone;        // teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nks = p.K / kKC;     // MMA stages per job
  const int TC = p.K / 256;      // weight stages per job

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], kXW);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], kXW);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&d_full[j], 1);
      mbar_init(&d_empty[j], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The first unit's first weight stages do not depend on the routing: when
  // most experts receive pairs they are fetched while the routing or packing
  // grid may still run.  (The routing grid is an ordinary stream-ordered
  // launch, so whatever wrote the tiles before it has completed.)
  int set_first, e_first, n0_first;
  unit_rows(p, (int)blockIdx.x, set_first, e_first, n0_first);
  const int pre = p.npairs >= p.n_expert ? min(kRawStages, TC) : 0;
  if (warp == kWProd && lane == 0) {
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmP);
    if (p.Y2 != nullptr) {
      tma_prefetch_desc(&tmC2);
      tma_prefetch_desc(&tmP2);
    }
    for (int tc = 0; tc < pre; ++tc)
      produce_weights<kRawStages>(set_first ? &tmC2 : &tmC, set_first ? &tmP2 : &tmP, p, e_first, n0_first, tc, tc,
                                  raw0, w_full, w_empty, abort_flag);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // When the first unit has no pairs, its prefetched stages are consumed and dropped.
  const bool first_empty = p.offsets != nullptr && p.offsets[e_first + 1] == p.offsets[e_first];

  bool ok = true;
  int njobs = 0;
  if (warp < kXW) {
    // ---- transform: raw tiles -> f16 weights in TMEM; then the epilogue ----
    // Warp (q, hw): TMEM lane quarter q (its 32 weight rows), and of each
    // 128-k stage the 64-k half hw when two warps share a quarter.
    const int q = warp & 3, hw = warp >> 2;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    float wmax = 0.0f;   // largest |m| + 15|s| of the blocks this thread formed
    int gws = 0, gs = 0;
    if (first_empty) {
      for (; gws < pre && ok; ++gws) {
        ok = __all_sync(0xffffffffu, mbar_wait(&w_full[gws], 0, abort_flag, p.dev_status));
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&w_empty[gws]);
      }
    }
    Jobs<kTok> jb;
    while (ok && jb.next(p)) {
      const int n = jb.n0 + 32 * q + lane;
      for (int tc = 0; tc < TC && ok; ++tc, ++gws) {
        const int slot = gws % kRawStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&w_full[slot], (gws / kRawStages) & 1, abort_flag, p.dev_status))) {
          ok = false;
          break;
        }
        const uint32_t cb = raw0 + slot * kRawBytes + q * kCodeBox + lane * 128;
        uint4 cw[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
          if (kHalves == 1 || ((b >> 1) & 1) == hw) cw[b] = lds128(cb + 16 * (b ^ (lane & 7)));
        const uint32_t pb = raw0 + slot * kRawBytes + 4 * kCodeBox + q * kPairBox + (lane >> 2) * 128;
        const uint4 pr0 = lds128(pb + 16 * ((2 * (lane & 3)) ^ ((lane >> 2) & 7)));
        const uint4 pr1 = lds128(pb + 16 * ((2 * (lane & 3) + 1) ^ ((lane >> 2) & 7)));
#pragma unroll
        for (int h = 0; h < 2; ++h, ++gs) {
          const int as = gs % kAStages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&a_empty[as], ((gs / kAStages) & 1) ^ 1, abort_flag, p.dev_status))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (kHalves == 2 && hh != hw) continue;
            uint32_t v[32];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const int b = 4 * h + 2 * hh + bb;
              uint32_t s2, m2;
              q4_pair_to_f16(u4_get(b < 4 ? pr0 : pr1, b & 3), s2, m2, wmax);
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const uint32_t word = u4_get(cw[b], t);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  v[16 * bb + 4 * t + i] = dequant2_f16(q4_pair_biased_f16(word, i), s2, m2);
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
      if (!L::kSepEpi && ok) {
        ok = epilogue_job<kMode, kTok>(p, jb, q, lane, tmem, njobs, d_full, d_empty, yoff[q], ysc[q], abort_flag);
        ++njobs;
      }
    }
    // a weight beyond f16's range would have become infinite
    if (__any_sync(0xffffffffu, wmax > kF16Max) && lane == 0) set_status(p.dev_status, QMM_ERR_RANGE);
  } else if (L::kSepEpi && warp < kWEpi + 4) {
    // ---- epilogue: fp32 accumulator -> Y (lane = weight row, column = pair) ----
    const int q = warp & 3;
    Jobs<kTok> jb;
    while (ok && jb.next(p)) {
      ok = epilogue_job<kMode, kTok>(p, jb, q, lane, tmem, njobs, d_full, d_empty, yoff[q], ysc[q], abort_flag);
      ++njobs;
    }
  } else if (warp == kWLoad) {
    // ---- activation loader ----
    int gs = 0;
    Jobs<kTok> jb;
    if (kPacked) {
      if (lane == 0) {
        tma_prefetch_desc(&tmX);
        while (ok && jb.next(p)) {
          const int row0 = jb.first + jb.pass0;
          for (int ks = 0; ks < nks; ++ks, ++gs) {
            const int bs = gs % kBStages;
            if (!mbar_wait(&b_empty[bs], ((gs / kBStages) & 1) ^ 1, abort_flag, p.dev_status)) {
              ok = false;
              break;
            }
            // whole kTok-row boxes (rows past the job's pairs are junk columns)
            mbar_arrive_expect_tx(&b_full[bs], (uint32_t)(2 * kBAtomBytes));
            const uint32_t sb = sB0 + bs * kBBytes;
            tma_load_2d_u32(sb, &tmX, &b_full[bs], ks * kKC, row0);
            tma_load_2d_u32(sb + kBAtomBytes, &tmX, &b_full[bs], ks * kKC + 64, row0);
          }
        }
      }
      __syncwarp();
    } else {
      // The rows are gathered in bf16 with cp.async and converted to f16 in
      // place once they have landed (both are 16-bit, so the swizzled
      // positions do not change).  Each lane converts the chunks it copied.
      int signalled = 0;   // stages whose b_full has been raised
      int st_r0[kBStagesMax] = {}, st_nt[kBStagesMax] = {};   // grouped rank of column 0 and width, per stage
      auto convert_stage = [&](int g) {
        const int bs = g % kBStages;
        const int r0 = st_r0[bs], nt = st_nt[bs];
        const uint32_t sb = sB0 + bs * kBBytes;
        for (int i = lane; i < nt * 16; i += 32) {
          const int c = i >> 4, ch = i & 15;
          const uint32_t dst = sb + (ch >> 3) * kBAtomBytes + (c >> 3) * 1024 + (c & 7) * 128 +
                               (uint32_t)(((ch & 7) ^ (c & 7)) << 4);
          // the inverse of a power of two in fp32's normal range
          const float down = __uint_as_float((254u << 23) - __float_as_uint(p.xup[r0 + c]));
          sts128(dst, bf16x8_to_f16x8_scaled(lds128(dst), down));
        }
      };
      while (ok && jb.next(p)) {
        const int nt = jb.nt(), ncol = jb.ncol();
        __syncwarp();   // the previous job's copies have read xoff
        for (int c = lane; c < nt; c += 32) {
          int64_t yo;
          pair_offsets(p, p.pairs[jb.first + jb.pass0 + c], xoff[c], yo);
        }
        __syncwarp();
        for (int ks = 0; ks < nks; ++ks, ++gs) {
          const int bs = gs % kBStages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&b_empty[bs], ((gs / kBStages) & 1) ^ 1, abort_flag, p.dev_status))) {
            ok = false;
            break;
          }
          st_r0[bs] = jb.first + jb.pass0;
          st_nt[bs] = nt;
          const uint32_t sb = sB0 + bs * kBBytes;
          for (int i = lane; i < ncol * 16; i += 32) {
            const int c = i >> 4, ch = i & 15;
            const bool valid = c < nt;
            const __nv_bfloat16* src = valid ? p.X + xoff[c] + (int64_t)ks * kKC + 8 * ch : p.X;
            const uint32_t dst = sb + (ch >> 3) * kBAtomBytes + (c >> 3) * 1024 + (c & 7) * 128 +
                                 (uint32_t)(((ch & 7) ^ (c & 7)) << 4);
            cp_async16_zfill(dst, src, valid ? 16u : 0u);
          }
          cp_async_commit();
          if (gs + 1 - signalled > kLoaderLag) {
            cp_async_wait<kLoaderLag>();
            convert_stage(signalled);
            fence_proxy_async_smem();   // generic-proxy writes -> tcgen05 reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_full[signalled % kBStages]);
            ++signalled;
          }
        }
      }
      cp_async_wait<0>();
      if (ok)
        for (int g = signalled; g < gs; ++g) convert_stage(g);
      fence_proxy_async_smem();
      __syncwarp();
      for (; signalled < gs; ++signalled)
        if (lane == 0) mbar_arrive(&b_full[signalled % kBStages]);
    }
  } else if (warp == kWMma) {
    // ---- MMA issuer ----
    // The tensor pipe queues few MMAs and this thread shares its SM
    // sub-partition with busy transform and epilogue warps, so the issue loop
    // is kept short: stages and phases are counted, and every descriptor is a
    // precomputed base plus a constant.
    if (lane == 0) {
      const uint64_t bdesc0 = desc_kmajor_sw128(sB0);
      const uint32_t acol0 = tmem + kColA;
      int as = 0, bs = 0;
      uint32_t aph = 0, bph = 0;
      Jobs<kTok> jb;
      while (ok && jb.next(p)) {
        const int db = njobs & 1;
        const uint32_t idesc = idesc_f16(kRows, jb.ncol(), false);   // f16 A and B
        const uint32_t dt = tmem + (uint32_t)(kTok * db);
        if (!mbar_wait(&d_empty[db], ((njobs >> 1) & 1) ^ 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          if (!(mbar_try_wait(&a_full[as], aph) || mbar_wait(&a_full[as], aph, abort_flag, p.dev_status)) ||
              !(mbar_try_wait(&b_full[bs], bph) || mbar_wait(&b_full[bs], bph, abort_flag, p.dev_status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t at = acol0 + 64u * (uint32_t)as;
          // +32 bytes per 16 k inside a 128-byte swizzle row (+2 in the address
          // field); the second 64 k of the stage is the next atom
          const uint64_t bd = bdesc0 + (uint64_t)((bs * kBBytes) >> 4);
#pragma unroll
          for (int j = 0; j < kKC / 16; ++j)
            umma_f16_ta(dt, at + 8u * (uint32_t)j, bd + (uint64_t)((j >> 2) * (kBAtomBytes >> 4) + 2 * (j & 3)),
                        idesc, (ks > 0 || j > 0) ? 1u : 0u);
          umma_commit(&a_empty[as]);
          umma_commit(&b_empty[bs]);
          if (++as == kAStages) {
            as = 0;
            aph ^= 1u;
          }
          if (++bs == kBStages) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&d_full[db]);
        ++njobs;
      }
    }
    __syncwarp();
  } else {
    // ---- weight producer ----
    if (lane == 0) {
      int gws = pre;
      Jobs<kTok> jb;
      bool first = true;
      while (ok && jb.next(p)) {
        // the first unit's first stages were issued before the routing wait
        const int tc0 = (first && !first_empty) ? pre : 0;   // the first job is then the first unit's pass 0
        first = false;
        for (int tc = tc0; tc < TC && ok; ++tc, ++gws)
          ok = produce_weights<kRawStages>(jb.set ? &tmC2 : &tmC, jb.set ? &tmP2 : &tmP, p, jb.e, jb.n0, tc, gws, raw0,
                                           w_full, w_empty, abort_flag);
      }
    }
    __syncwarp();
  }

  // ---- teardown ----
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && lane == 0 && (warp == kWLoad || warp == kWProd)) {
    // TMA writes of stages nobody consumed may still be in flight
    uint64_t* full = warp == kWProd ? w_full : b_full;
    const int n = warp == kWProd ? kRawStages : kBStages;
    for (int s = 0; s < n; ++s)
      for (int ph = 0; ph < 2; ++ph)
        mbar_wait(&full[s], ph, abort_flag, nullptr, 50000000ull) || mbar_try_wait(&full[s], ph);
  }
  if (warp == kWMma) {
    if (lane == 0) {
      umma_commit(done);   // every MMA of this CTA has completed before TMEM is freed
      mbar_wait(done, 0, abort_flag, nullptr, 100000000ull) || mbar_try_wait(done, 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Routing: expert offsets and the grouped pair list.  Block b owns pairs
// [b*PB, (b+1)*PB), PB a multiple of 256.  Every block counts all ids (the
// expert offsets) and the ids before its range (each expert's base rank
// there).  It then ranks its pairs in rounds of 256, in pair order: inside a
// warp, lanes with the same expert are ordered by match_any; across the eight
// warps of a round, by per-warp expert counts in shared memory.  So the
// grouped list is deterministic.
constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads)
moe_route_kernel(const int32_t* __restrict__ ids, int64_t ld_ids, int n_used, int T, int n_expert, int PB,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ pairs, int32_t* dev_status) {
  extern __shared__ int rsm[];
  int* off = rsm;                    // [n_expert + 1]: histogram, then exclusive offsets
  int* before = rsm + n_expert + 1;  // [n_expert]: pairs of each expert before the current round
  int* cnt = before + n_expert;      // [kRouteWarps][n_expert]: this round's counts per warp
  __shared__ int wsum[kRouteWarps];
  // the packing grid (or the grouped kernel) may start; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int npairs = T * n_used;
  const int p0 = blockIdx.x * PB;
  for (int e = tid; e <= n_expert; e += kRouteThreads) off[e] = 0;
  for (int e = tid; e < n_expert; e += kRouteThreads) before[e] = 0;
  __syncthreads();
  bool bad = false;
  // eight independent loads in flight per thread, then the shared-memory counts
  for (int base = 0; base < npairs; base += 8 * kRouteThreads) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int pr = base + u * kRouteThreads + tid;
      ev[u] = pr < npairs ? ids[(int64_t)(pr / n_used) * ld_ids + (pr % n_used)] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int pr = base + u * kRouteThreads + tid;
      if (pr >= npairs) continue;
      const int e = ev[u];
      if (e < 0 || e >= n_expert) {
        bad = true;
        continue;
      }
      atomicAdd(&off[e], 1);
      if (pr < p0) atomicAdd(&before[e], 1);
    }
  }
  if (bad && blockIdx.x == 0) set_status(dev_status, QMM_ERR_BAD_EXPERT_ID);
  __syncthreads();
  // exclusive scan of off[0 .. n_expert) in place; off[n_expert] = total
  {
    const int per = (n_expert + kRouteThreads - 1) / kRouteThreads;
    const int lo = min(tid * per, n_expert), hi = min(lo + per, n_expert);
    int seg = 0;
    for (int e = lo; e < hi; ++e) seg += off[e];
    int incl = seg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      wbase += (w < warp) ? wsum[w] : 0;
      total += wsum[w];
    }
    int runv = wbase + incl - seg;
    __syncthreads();   // every thread has read its segment before any is overwritten
    for (int e = lo; e < hi; ++e) {
      const int c = off[e];
      off[e] = runv;
      runv += c;
    }
    if (tid == 0) off[n_expert] = total;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e <= n_expert; e += kRouteThreads) offsets[e] = off[e];
  // rank this block's pairs, 256 per round, in pair order
  const int p_end = min(p0 + PB, npairs);
  for (int r0 = p0; r0 < p_end; r0 += kRouteThreads) {
    for (int i = tid; i < kRouteWarps * n_expert; i += kRouteThreads) cnt[i] = 0;
    __syncthreads();
    const int pr = r0 + tid;
    int e = -1;
    if (pr < p_end) {
      e = ids[(int64_t)(pr / n_used) * ld_ids + (pr % n_used)];
      if (e < 0 || e >= n_expert) e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int local = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && local == 0) cnt[warp * n_expert + e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int rank = off[e] + before[e] + local;
      for (int w = 0; w < warp; ++w) rank += cnt[w * n_expert + e];
      pairs[rank] = pr;
    }
    __syncthreads();
    // this round's pairs come before the next round's
    for (int x = tid; x < n_expert; x += kRouteThreads) {
      int sum = 0;
      for (int w = 0; w < kRouteWarps; ++w) sum += cnt[w * n_expert + x];
      before[x] += sum;
    }
    __syncthreads();
  }
}

// Activation packing: the src1 row of every grouped pair, as f16 operands at
// its rank, so that each job's B operand is one dense block, and the row's
// inverse scale up[rank].  With Xp null (the gather mode) only the scales are
// written.  One warp per row; rows of up to 2,048 elements stay in registers
// between the max and the conversion, longer ones are read twice.
__global__ void __launch_bounds__(kRouteThreads)
moe_pack_kernel(const int32_t* __restrict__ pairs, const int32_t* __restrict__ offsets, int n_expert, int n_used,
                const __nv_bfloat16* __restrict__ X, int64_t ldx_token, int64_t ldx_slot, int K,
                __half* __restrict__ Xp, float* __restrict__ up) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the pair list comes from the routing grid
  const int lane = threadIdx.x & 31;
  const int total = offsets[n_expert];
  const int chunks = K / 8;
  const int nw = (int)gridDim.x * kRouteWarps;
  for (int r = (int)blockIdx.x * kRouteWarps + ((int)threadIdx.x >> 5); r < total; r += nw) {
    const int pr = pairs[r];
    const int t = pr / n_used, i = pr - t * n_used;
    const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)t * ldx_token + (int64_t)i * ldx_slot);
    uint4 v[8];
    uint32_t am = 0;
    for (int c0 = 0; c0 < chunks; c0 += 8 * 32) {
      uint4 w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        w[u] = c < chunks ? ldg128(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        am = bf16x2_absmax_bits(am, w[u].x);
        am = bf16x2_absmax_bits(am, w[u].y);
        am = bf16x2_absmax_bits(am, w[u].z);
        am = bf16x2_absmax_bits(am, w[u].w);
        if (c0 == 0) v[u] = w[u];
      }
    }
    float down, u_r;
    f16_row_scale(__reduce_max_sync(0xffffffffu, bf16x2_absmax_fold(am)), down, u_r);
    if (lane == 0) up[r] = u_r;
    if (Xp == nullptr) continue;
    uint4* dst = reinterpret_cast<uint4*>(Xp + (int64_t)r * K);
    for (int c0 = 0; c0 < chunks; c0 += 8 * 32) {
      if (c0 > 0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < chunks) v[u] = ldg128(src + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) dst[c] = bf16x8_to_f16x8_scaled(v[u], down);
      }
    }
  }
}

template <int kMode, int kTok, int kCtas>
cudaError_t launch_tc(const CUtensorMap& tmC, const CUtensorMap& tmP, const CUtensorMap& tmC2, const CUtensorMap& tmP2,
                      const CUtensorMap& tmX, const MoeParams& p, cudaStream_t stream) {
  using L = Lay<kTok, kCtas>;
  auto kern = q4_tc_kernel<kMode, kTok, kCtas>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kSmemBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)min(p.n_units, kCtas * sms));   // persistent
  cfg.blockDim = dim3(32 * L::kWarps);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;   // overlap the packing or conversion grid
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmC, tmP, tmC2, tmP2, tmX, p);
}

}  // namespace

size_t q4_moe_table_bytes(int64_t n_expert, int64_t n_used, int64_t T) {
  const size_t off = ((size_t)(n_expert + 1) * 4 + 255) / 256 * 256;
  return off + 2 * (((size_t)(T * n_used) * 4 + 255) / 256 * 256);   // pair ids, then row scales
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
  p.n_used = a.n_used;
  p.n_expert = a.n_expert;
  p.npairs = a.T * a.n_used;
  p.nrb = (a.N + kRows - 1) / kRows;
  p.units_per_set = a.n_expert * p.nrb;
  p.n_units = (a.tiles2 != nullptr ? 2 : 1) * p.units_per_set;
  p.Y = a.Y;
  p.Y2 = a.tiles2 != nullptr ? a.Y2 : nullptr;
  p.ldy_token = a.ldy_token;
  p.ldy_slot = a.ldy_slot;
  p.offsets = a.offsets;
  p.pairs = a.pairs;
  p.xup = a.xup;
  p.dev_status = a.dev_status;
  const uint64_t n_tiles = (uint64_t)a.n_expert * (uint64_t)p.tiles_per_expert;
  if (n_tiles > (uint64_t)INT32_MAX || 2 * (int64_t)a.n_expert * p.nrb > INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tmC, tmP, tmC2, tmP2, tmX;
  const uint64_t tile_rows = (uint64_t)a.n_expert * (uint64_t)(a.N / 32);
  if (!make_tmap_q4_tiles(&tmC, a.tiles, (uint64_t)(a.K / 256), tile_rows, 32) ||
      !make_tmap_q4_tiles(&tmP, a.tiles, (uint64_t)(a.K / 256), tile_rows, 8))
    return cudaErrorInvalidValue;
  tmC2 = tmC;
  tmP2 = tmP;
  if (a.tiles2 != nullptr && (!make_tmap_q4_tiles(&tmC2, a.tiles2, (uint64_t)(a.K / 256), tile_rows, 32) ||
                              !make_tmap_q4_tiles(&tmP2, a.tiles2, (uint64_t)(a.K / 256), tile_rows, 8)))
    return cudaErrorInvalidValue;
  const int npairs = a.T * a.n_used;
  // 256 pairs per routing block, more when the batch is large enough that
  // every block recounting all ids would cost more
  int PB = kRouteThreads;
  while ((int64_t)npairs * ((npairs + PB - 1) / PB) > (int64_t)16 << 20) PB *= 2;
  const int nblk = (npairs + PB - 1) / PB;
  const size_t rsmem = (size_t)((2 + kRouteWarps) * a.n_expert + 1) * sizeof(int);
  if (rsmem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)rsmem);
    if (e != cudaSuccess) return e;
  }
  moe_route_kernel<<<nblk, kRouteThreads, rsmem, stream>>>(a.ids, a.ld_ids, a.n_used, a.T, a.n_expert, PB,
                                                           a.offsets, a.pairs, a.dev_status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  {
    // packed rows and their scales, or (gather mode) the scales alone
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int pgrid = std::max(1, std::min((npairs + kRouteWarps - 1) / kRouteWarps, 8 * sms));
    err = launch_pdl(moe_pack_kernel, dim3(pgrid), dim3(kRouteThreads), 0, stream, (const int32_t*)a.pairs,
                     (const int32_t*)a.offsets, a.n_expert, a.n_used, a.X, a.ldx_token, a.ldx_slot, a.K, a.xperm,
                     a.xup);
    if (err != cudaSuccess) return err;
  }
  if (a.xperm == nullptr) return launch_tc<kTableGather, 64, 2>(tmC, tmP, tmC2, tmP2, tmC, p, stream);
  if (!make_tmap_2d(&tmX, true, a.xperm, (uint64_t)a.K, (uint64_t)npairs, (uint64_t)a.K * 2, 64, 64))
    return cudaErrorInvalidValue;
  return launch_tc<kTablePacked, 64, 2>(tmC, tmP, tmC2, tmP2, tmX, p, stream);
}

bool q4_umma_eligible(int64_t M, int64_t N, int64_t K) {
  (void)N;
  (void)K;
  return M >= 17;   // M <= 16 runs the decode GEMV kernels
}

cudaError_t launch_q4_gemm_umma(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream) {
  __half* Xh = static_cast<__half*>(a.act16);   // the activations as scaled f16 rows [M][K]
  MoeParams p{};
  p.tiles_per_expert = (int64_t)(a.N / 32) * (a.K / 256);
  p.N = a.N;
  p.K = a.K;
  p.X = a.X;
  p.ldx_token = a.ldx;
  p.n_used = 1;
  p.n_expert = 1;
  p.npairs = a.M;
  p.nrb = (a.N + kRows - 1) / kRows;
  p.n_units = p.nrb;
  p.units_per_set = p.nrb;
  p.Y = a.Y;
  p.ldy_token = a.ldy;
  p.dense_rows = a.M;
  p.xup = reinterpret_cast<const float*>(static_cast<const char*>(a.act16) + act_f16_scale_offset(a.M, a.K));
  p.dev_status = dev_status;
  if (p.tiles_per_expert > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tmC, tmP, tmX;
  if (!make_tmap_q4_tiles(&tmC, a.tiles, (uint64_t)(a.K / 256), (uint64_t)(a.N / 32), 32) ||
      !make_tmap_q4_tiles(&tmP, a.tiles, (uint64_t)(a.K / 256), (uint64_t)(a.N / 32), 8))
    return cudaErrorInvalidValue;
  // Token chunk per job (the MMA's N): 64 for small M.  Otherwise 192 when
  // that takes fewer chunks than 128 and the units still cover every SM
  // (wider MMAs amortise their issue, and each weight is dequantised fewer
  // times); small N keeps 128 for more units.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int c192 = (a.M + 191) / 192, c128 = (a.M + 127) / 128;
  const int tok = a.M <= 64 ? 64 : (a.M > 128 && c192 < c128 && (int64_t)p.nrb * c192 >= sms ? 192 : 128);
  if (!make_tmap_2d(&tmX, true, Xh, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 64, (uint32_t)tok))
    return cudaErrorInvalidValue;
  p.dense_chunks = (a.M + tok - 1) / tok;
  if ((int64_t)p.nrb * p.dense_chunks > INT32_MAX) return cudaErrorInvalidValue;
  p.n_units = p.nrb * p.dense_chunks;
  const cudaError_t err = launch_act_to_f16(a.X, a.ldx, a.M, a.K, a.act16, stream);
  if (err != cudaSuccess) return err;
  if (tok == 64) return launch_tc<kDense, 64, 1>(tmC, tmP, tmC, tmP, tmX, p, stream);
  if (tok == 192) return launch_tc<kDense, 192, 1>(tmC, tmP, tmC, tmP, tmX, p, stream);
  return launch_tc<kDense, 128, 1>(tmC, tmP, tmC, tmP, tmX, p, stream);
}

}  // namespace qmm
