// 4-bit GEMM at prefill sizes on the 5th-generation tensor cores.
//
// Y[m][n] = sum_k X[m][k] * w[n][k], with w = q * scale + min from 32x256 q4_1
// tiles ("NPU engine: full ELFs, no xclbin", "Q4NX chunks"; "Zaya 8B Q4NX on
// the AMD NPU", round 26).  The pages' lesson for prefill (round 25o): reuse
// each dequantised weight across many activation columns.  Here each weight
// is dequantised once per 256 tokens, straight into shared memory, and never
// exists in expanded form in HBM.
//
// One CTA computes a 128 (weight rows) x 256 (tokens) tile.  The MMA's M side
// is the weights (the A operand, written by the transform warps in the
// 128-byte-swizzle K-major layout).  Its N side is X (the B operand, loaded
// by TMA).  The accumulator is fp32 in TMEM.
//   warp 0     TMA producer for X tiles (4-stage ring)
//   warp 1     TMEM owner and MMA issuer (tcgen05.mma kind::f16, bf16)
//   warps 2-5  transform: each owns one 32-row tile row; lane = row.  Code
//              words and (scale, min) pairs are prefetched four stages ahead
//              in registers, and each weight is formed as bf16(q*s + min)
//              with one fma.rn.bf16x2 (one rounding).  Then these warps
//              drain TMEM and store Y.
#include <cuda_bf16.h>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kBW = 128;            // weight rows per tile (MMA M)
constexpr int kBT = 256;            // tokens per tile (MMA N)
constexpr int kBK = 64;             // K per stage
constexpr int kStages = 4;
constexpr int kWBytes = kBW * kBK * 2;   // 16 KB
constexpr int kXBytes = kBT * kBK * 2;   // 32 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * (kWBytes + kXBytes) + 256;
constexpr int kPrefetch = 4;        // stages of raw weights in flight per transform thread
constexpr int kMinM = 17;           // M <= 16 runs the decode GEMV kernel

struct Q4UmmaParams {
  const uint8_t* tiles;
  int N, K, M;
  float* Y;
  int64_t ldy;
  int32_t* dev_status;
};

struct RawStage {
  uint4 w[2];   // code words 0..3 of blocks 2s and 2s+1 (32 contiguous bytes of the row)
  uint2 p;      // (scale, min) pairs of blocks 2s, 2s+1
};

__device__ __forceinline__ void load_raw(RawStage& r, const uint8_t* row_tile0, const uint8_t* pair_tile0,
                                         int kb, bool valid) {
  if (!valid) {
    r.w[0] = make_uint4(0u, 0u, 0u, 0u);
    r.w[1] = make_uint4(0u, 0u, 0u, 0u);
    r.p = make_uint2(0u, 0u);
    return;
  }
  const int tc = kb >> 2, s4 = kb & 3;
  const uint8_t* base = row_tile0 + (int64_t)tc * kTileBytes + 32 * s4;
  r.w[0] = ldg128(base);
  r.w[1] = ldg128(base + 16);
  r.p = *reinterpret_cast<const uint2*>(pair_tile0 + (int64_t)tc * kTileBytes + 8 * s4);
}

__device__ __forceinline__ uint32_t bf16x2_sub_fma(uint32_t q2, uint32_t s2, uint32_t m2) {
  // (128+q) - 128 = q exactly, then q*s + m with a single rounding
  __nv_bfloat162 q = *reinterpret_cast<__nv_bfloat162*>(&q2);
  const uint32_t c128 = 0x43004300u;
  q = __hsub2(q, *reinterpret_cast<const __nv_bfloat162*>(&c128));
  const __nv_bfloat162 w = __hfma2(q, *reinterpret_cast<__nv_bfloat162*>(&s2), *reinterpret_cast<__nv_bfloat162*>(&m2));
  return *reinterpret_cast<const uint32_t*>(&w);
}

// Dequantise one stage (64 k of one row) into the swizzled A tile.
__device__ __forceinline__ void write_stage(uint8_t* tile, int row, const RawStage& r) {
  const uint32_t rowoff = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
  for (int bl = 0; bl < 2; ++bl) {
    const uint32_t pair = bl ? r.p.y : r.p.x;
    const uint32_t s2 = __byte_perm(pair, 0, 0x1010);
    const uint32_t m2 = __byte_perm(pair, 0, 0x3232);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t word = u4_get(r.w[bl], t);
      uint4 o;
      o.x = bf16x2_sub_fma(q4_pair_biased(word, 0), s2, m2);
      o.y = bf16x2_sub_fma(q4_pair_biased(word, 1), s2, m2);
      o.z = bf16x2_sub_fma(q4_pair_biased(word, 2), s2, m2);
      o.w = bf16x2_sub_fma(q4_pair_biased(word, 3), s2, m2);
      const int c = 4 * bl + t;    // 16-byte chunk = k 8c .. 8c+7 of the stage
      *reinterpret_cast<uint4*>(tile + rowoff + (uint32_t)(((c ^ (row & 7)) & 7) << 4)) = o;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
q4_umma_kernel(const __grid_constant__ CUtensorMap tmX, const Q4UmmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  uint8_t* sW = smem;
  uint8_t* sX = smem + kStages * kWBytes;
  uint64_t* xfull = reinterpret_cast<uint64_t*>(smem + kStages * (kWBytes + kXBytes));
  uint64_t* wfull = xfull + kStages;
  uint64_t* empty = wfull + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* done = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBW, m0 = blockIdx.y * kBT;
  const int nkb = p.K / kBK;
  const int TC = p.K / 256;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&wfull[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag, p.dev_status)) break;
        mbar_arrive_expect_tx(&xfull[s], kXBytes);
        tma_load_2d(sX + s * kXBytes, &tmX, &xfull[s], kb * kBK, m0);
        issued = kb + 1;
      }
      if (*abort_flag)
        for (int kb = issued > kStages ? issued - kStages : 0; kb < issued; ++kb)
          mbar_wait(&xfull[kb % kStages], (kb / kStages) & 1, abort_flag, nullptr, 100000000ull) ||
              mbar_try_wait(&xfull[kb % kStages], (kb / kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kBW, kBT, true);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1;
        if (!mbar_wait(&xfull[s], ph, abort_flag, p.dev_status) ||
            !mbar_wait(&wfull[s], ph, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w_addr = smem_u32(sW + s * kWBytes);
        const uint32_t x_addr = smem_u32(sX + s * kXBytes);
#pragma unroll
        for (int j = 0; j < kBK / 16; ++j)
          umma_f16(tmem, desc_kmajor_sw128(w_addr + 32 * j), desc_kmajor_sw128(x_addr + 32 * j), idesc,
                   (kb > 0 || j > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
      }
      if (ok) umma_commit(tfull);
      umma_commit(done);
      mbar_wait(done, 0, abort_flag, p.dev_status);
    }
  } else {
    // transform warps 2..5 -> tile row tw, row = lane; then epilogue on TMEM quadrant warp%4
    const int tw = warp - 2;
    const int row = 32 * tw + lane;                 // row inside the 128-row tile
    const int n = n0 + row;
    const bool valid = n < p.N;
    const int tr = (valid ? n : 0) / 32;
    const uint8_t* row_tile0 = p.tiles + (int64_t)tr * TC * kTileBytes + (n & 31) * 128;
    const uint8_t* pair_tile0 = p.tiles + (int64_t)tr * TC * kTileBytes + 4096 + (n & 31) * 32;
    RawStage ring[kPrefetch];
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) load_raw(ring[i], row_tile0, pair_tile0, i, valid && i < nkb);
    bool ok = true;
    for (int kb0 = 0; kb0 < nkb && ok; kb0 += kPrefetch) {
#pragma unroll
      for (int i = 0; i < kPrefetch; ++i) {
        const int kb = kb0 + i;
        if (kb < nkb && ok) {
          const int s = kb % kStages;
          if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag, p.dev_status)) {
            ok = false;
          } else {
            write_stage(sW + s * kWBytes, row, ring[i]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[s]);
            load_raw(ring[i], row_tile0, pair_tile0, kb + kPrefetch, valid && kb + kPrefetch < nkb);
          }
        }
      }
    }
    // epilogue: this warp reads TMEM lanes 32*(warp%4)..; its rows are n0 + 32*(warp%4) + lane
    const int q = warp & 3;
    const int nrow = n0 + 32 * q + lane;
    ok = __all_sync(0xffffffffu, ok);
    // warp-uniform: tcgen05.ld below is a whole-warp instruction
    if (ok && __all_sync(0xffffffffu, mbar_wait(tfull, 0, abort_flag, p.dev_status))) {
      tc_fence_after();
#pragma unroll 1
      for (int j = 0; j < kBT / 32; ++j) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * j), r);
        tmem_wait_ld();
        if (nrow < p.N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int m = m0 + 32 * j + i;
            if (m < p.M) p.Y[(int64_t)m * p.ldy + nrow] = __uint_as_float(r[i]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool q4_umma_eligible(int64_t M, int64_t N, int64_t K) {
  (void)N;
  (void)K;
  return M >= kMinM;
}

cudaError_t launch_q4_gemm_umma(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream) {
  CUtensorMap tmX;
  if (!make_tmap_2d(&tmX, true, const_cast<__nv_bfloat16*>(a.X), (uint64_t)a.K, (uint64_t)a.M,
                    (uint64_t)a.ldx * 2, kBK, kBT))
    return cudaErrorInvalidValue;
  Q4UmmaParams p{};
  p.tiles = a.tiles;
  p.N = a.N;
  p.K = a.K;
  p.M = a.M;
  p.Y = a.Y;
  p.ldy = a.ldy;
  p.dev_status = dev_status;
  cudaError_t err =
      cudaFuncSetAttribute(q4_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)((a.N + kBW - 1) / kBW), (unsigned)((a.M + kBT - 1) / kBT));
  q4_umma_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmX, p);
  return cudaGetLastError();
}

}  // namespace qmm
