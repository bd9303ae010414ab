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
//   2. the GEMM: one CTA per 128 x 256 output tile.  Warp 0 issues TMA loads
//      of both f16 operands into a 4-stage mbarrier ring (128-byte swizzle).
//      Warp 1 owns TMEM and issues tcgen05.mma.  Warps 2..9 drain the
//      accumulator and run the exact epilogue: zero points, bias, output
//      conversion.
#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kBM = 128;             // activation rows per tile (MMA M)
constexpr int kBN = 256;             // weight rows per tile (MMA N)
constexpr int kBK = 64;              // K per stage (one 128-byte swizzle row of f16)
constexpr int kStages = 4;
constexpr int kChunkK = 1024;        // K per exact fp32 chunk
constexpr int kChunkKB = kChunkK / kBK;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
// warp 0 TMA producer, warp 1 MMA issuer, warps 2..9 epilogue.  Ten warps put
// three on some SM sub-partitions, which caps the kernel at 168 registers.
constexpr int kEpiWarp0 = 2;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kTmemCols = 512;       // two 256-column fp32 accumulators
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 8 * 128 * 12 + 256;
constexpr int kMinM = 256;           // below this the legacy-MMA route is used

struct Int8UmmaParams {
  int M, N, K, Kp;
  int tiles_n;                       // number of 256-column tiles
  int ntiles;
  const int32_t* row_sum;            // [M] (null when zB' == 0)
  Int8Epi epi;
  int32_t* dev_status;
};

constexpr int kColConstBytes = kEpiWarps * 128 * 12;   // per-warp c1 / s_w / Mq of 128 columns

// Output conversion of one element (fp32 steps with explicit IEEE rounding).
__device__ __forceinline__ uint32_t epi_convert(const Int8Epi& e, int32_t yb, float sx, float sw, float mq,
                                                bool per_row_mq) {
  const int ot = e.out_type;
  if (ot == QMM_S32) return (uint32_t)yb;
  if (ot == QMM_F32) return __float_as_uint(__fmul_rn(__fmul_rn(__int2float_rn(yb), sx), sw));
  const float m = per_row_mq ? __fdiv_rn(__fmul_rn(sx, sw), e.s_y) : mq;
  float r = __fmul_rn(__int2float_rn(yb), m);
  r = fminf(fmaxf(r, -1.0e9f), 1.0e9f);
  int q = __float2int_rn(r) + e.zp_y;
  q = (ot == QMM_S8) ? min(max(q, -128), 127) : min(max(q, 0), 255);
  return (uint32_t)q & 0xFFu;
}

// 32 consecutive columns of one row: converted and stored 16 bytes at a time
// (element-wise at ragged edges or unaligned outputs).
__device__ __forceinline__ void epi_store32(const Int8UmmaParams& p, int row, int nb, const int32_t* acc,
                                            const uint32_t* c1, const float* sw, const float* mq, uint32_t r1,
                                            float sx, bool per_row_mq, bool vec_ok) {
  const Int8Epi& e = p.epi;
  const bool full = vec_ok && nb + 32 <= p.N;
  if (e.out_type == QMM_S32 || e.out_type == QMM_F32) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(e.out) + (int64_t)row * e.ldo + nb;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = 4 * v + i;
        o[i] = epi_convert(e, (int32_t)((uint32_t)acc[c] + c1[c] + r1), sx, sw[c], mq[c], per_row_mq);
      }
      if (full) {
        reinterpret_cast<uint4*>(dst)[v] = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (nb + 4 * v + i < p.N) dst[4 * v + i] = o[i];
      }
    }
  } else {
    uint8_t* dst = reinterpret_cast<uint8_t*>(e.out) + (int64_t)row * e.ldo + nb;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int c = 16 * v + 4 * wi + b;
          word |= epi_convert(e, (int32_t)((uint32_t)acc[c] + c1[c] + r1), sx, sw[c], mq[c], per_row_mq)
                  << (8 * b);
        }
        w[wi] = word;
      }
      if (full) {
        reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (nb + 16 * v + i < p.N) dst[16 * v + i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
      }
    }
  }
}

// Persistent: each CTA walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// The stage ring and the two TMEM accumulators carry on across tiles, so the
// epilogue of one tile overlaps the MMAs of the next.
__global__ void __launch_bounds__(kThreads, 1)
int8_umma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Int8UmmaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sConst = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sConst + kColConstBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;    // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = p.Kp / kBK;
  const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&tfull[d], 1);
      mbar_init(&tempty[d], kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
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
      int g = 0;          // k blocks issued so far (all tiles)
      bool ok = true;
      for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
        const int m0 = (t / p.tiles_n) * kBM, n0 = (t % p.tiles_n) * kBN;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(sA + s * kABytes, &tmA, &full[s], kb * kBK, m0);
          tma_load_2d(sB + s * kBBytes, &tmB, &full[s], kb * kBK, n0);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA leaves
        for (int k = g > kStages ? g - kStages : 0; k < g; ++k)
          mbar_try_wait(&full[k % kStages], (k / kStages) & 1) ||
              mbar_wait(&full[k % kStages], (k / kStages) & 1, abort_flag, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kBM, kBN, false);
      int g = 0, gc = 0;  // k blocks consumed, chunks issued (all tiles)
      bool ok = true;
      for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
        for (int c = 0; c < nchunks && ok; ++c, ++gc) {
          const int d = gc & 1, u = gc >> 1;
          if (!mbar_wait(&tempty[d], (u & 1) ^ 1, abort_flag, p.dev_status)) { ok = false; break; }
          tc_fence_after();
          const int kend = min(nkb, (c + 1) * kChunkKB);
          for (int kb = c * kChunkKB; kb < kend; ++kb, ++g) {
            const int s = g % kStages;
            if (!mbar_wait(&full[s], (g / kStages) & 1, abort_flag, p.dev_status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * kABytes);
            const uint32_t b_addr = smem_u32(sB + s * kBBytes);
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
              umma_f16(tmem + d * 256, desc_kmajor_sw128(a_addr + 32 * j), desc_kmajor_sw128(b_addr + 32 * j),
                       idesc, (kb > c * kChunkKB || j > 0) ? 1u : 0u);
            umma_commit(&empty[s]);
          }
          if (ok) umma_commit(&tfull[d]);
        }
      }
      // every MMA has completed before TMEM is released
      umma_commit(done);
      mbar_wait(done, 0, abort_flag, p.dev_status);
    }
  } else if (warp >= kEpiWarp0) {
    // epilogue: warp w reads TMEM lanes 32*(w%4).. and columns h*128..h*128+127
    const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
    const int ew = warp - kEpiWarp0;
    uint32_t* c1 = reinterpret_cast<uint32_t*>(sConst) + ew * 384;
    float* swc = reinterpret_cast<float*>(c1 + 128);
    float* mqc = reinterpret_cast<float*>(c1 + 256);
    const Int8Epi& e = p.epi;
    const bool requant = (e.out_type == QMM_S8 || e.out_type == QMM_U8);
    const bool per_row_sx = (e.s_x != nullptr && e.s_x_stride != 0);
    const float sx0 = e.s_x ? e.s_x[0] : 1.0f;
    const int esz = (e.out_type == QMM_S32 || e.out_type == QMM_F32) ? 4 : 1;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(e.out) & 15) == 0) && (((int64_t)e.ldo * esz) % 16 == 0);
    int gc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
      const int m0 = (t / p.tiles_n) * kBM, n0 = (t % p.tiles_n) * kBN;
      const int nbase = n0 + h * 128;
      // per-column constants of this warp's 128 columns: bias - zA' colSum, s_w, Mq
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int i = lane + 32 * v, n = nbase + i;
        uint32_t cc = 0u;
        float w = 1.0f, m = 0.0f;
        if (n < p.N) {
          cc = (uint32_t)(e.bias ? e.bias[n] : 0) - e.zAp * (uint32_t)e.col_sum[n];
          w = e.s_w ? e.s_w[n] : 1.0f;
          if (requant && !per_row_sx) m = __fdiv_rn(__fmul_rn(sx0, w), e.s_y);
        }
        c1[i] = cc;
        swc[i] = w;
        mqc[i] = m;
      }
      __syncwarp();
      const int row = m0 + 32 * q + lane;
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
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * 256 + h * 128 + 32 * j), r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int32_t v = __float2int_rn(__uint_as_float(r[i]));
            acc[32 * j + i] = (c == 0) ? v : (int32_t)((uint32_t)acc[32 * j + i] + (uint32_t)v);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[d]);
      }
      if (ok && row < p.M) {
        const uint32_t r1 = p.row_sum ? (0u - e.zBp * ((uint32_t)p.row_sum[row] - e.Kz)) : 0u;
        const float sx = per_row_sx ? e.s_x[row] : sx0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          epi_store32(p, row, nbase + 32 * j, acc + 32 * j, c1 + 32 * j, swc + 32 * j, mqc + 32 * j, r1, sx,
                      requant && per_row_sx, vec_ok);
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One block per row: A rows (shift, K-tail mask, rowSum) or packed B rows.
__global__ void __launch_bounds__(128) int8_widen_kernel(const int8_t* __restrict__ A, int64_t lda, bool a_u8,
                                                         int M, int K, const int8_t* __restrict__ B, int N,
                                                         int Kp, __half* __restrict__ A16,
                                                         __half* __restrict__ B16,
                                                         int32_t* __restrict__ row_sum) {
  __shared__ int red[4];
  const int row = blockIdx.x;
  const bool is_a = row < M;
  const int8_t* src = is_a ? A + (int64_t)row * lda : B + (int64_t)(row - M) * Kp;
  __half* dst = is_a ? A16 + (int64_t)row * Kp : B16 + (int64_t)(row - M) * Kp;
  const int K16 = (K + 15) & ~15;
  const int limit = is_a ? K16 : Kp;
  const uint32_t xorv = (is_a && a_u8) ? 0x80808080u : 0u;
  int sum = 0;
  for (int k = threadIdx.x * 16; k < Kp; k += blockDim.x * 16) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (k < limit) {
      const uint4 v = ldg128(src + k);
      w[0] = v.x ^ xorv; w[1] = v.y ^ xorv; w[2] = v.z ^ xorv; w[3] = v.w ^ xorv;
      if (is_a && k + 16 > K) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int valid = K - (k + 4 * q);
          if (valid <= 0) w[q] = 0u;
          else if (valid < 4) w[q] &= (1u << (8 * valid)) - 1u;
        }
      }
    }
    __half h[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      sum = __dp4a((int)w[q], 0x01010101, sum);
#pragma unroll
      for (int b = 0; b < 4; ++b) h[4 * q + b] = __int2half_rn((int)(int8_t)(w[q] >> (8 * b)));
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst + k);
    d4[0] = *reinterpret_cast<const uint4*>(&h[0]);
    d4[1] = *reinterpret_cast<const uint4*>(&h[8]);
  }
  if (is_a && row_sum != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) row_sum[row] = red[0] + red[1] + red[2] + red[3];
  }
}

struct WsLayout {
  size_t a16, b16, rs, total;
};
WsLayout ws_layout(int64_t M, int64_t K, int64_t N) {
  const int64_t Kp = padded_k(K);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  WsLayout w{};
  w.a16 = 0;
  w.b16 = up((size_t)M * Kp * 2);
  w.rs = w.b16 + up((size_t)N * Kp * 2);
  w.total = w.rs + up((size_t)M * 4);
  return w;
}

}  // namespace

bool int8_umma_eligible(int64_t M, int64_t K, int64_t N) {
  (void)K;
  (void)N;
  return M >= kMinM;
}

size_t int8_umma_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  return int8_umma_eligible(M, K, N) ? ws_layout(M, K, N).total : 0;
}

cudaError_t launch_int8_gemm_umma(const Int8GemmArgs& a, void* workspace, int32_t* dev_status,
                                  cudaStream_t stream) {
  const WsLayout w = ws_layout(a.M, a.K, a.N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* A16 = reinterpret_cast<__half*>(ws + w.a16);
  __half* B16 = reinterpret_cast<__half*>(ws + w.b16);
  int32_t* rs = a.need_rowsum ? reinterpret_cast<int32_t*>(ws + w.rs) : nullptr;
  const int Kp = (int)a.Kp;
  int8_widen_kernel<<<a.M + a.N, 128, 0, stream>>>(a.A, a.lda, a.a_u8, a.M, a.K, a.B, a.N, Kp, A16, B16, rs);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, false, A16, (uint64_t)Kp, (uint64_t)a.M, (uint64_t)Kp * 2, kBK, kBM) ||
      !make_tmap_2d(&tmB, false, B16, (uint64_t)Kp, (uint64_t)a.N, (uint64_t)Kp * 2, kBK, kBN))
    return cudaErrorInvalidValue;
  Int8UmmaParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.Kp = Kp;
  p.tiles_n = (a.N + kBN - 1) / kBN;
  p.ntiles = ((a.M + kBM - 1) / kBM) * p.tiles_n;
  p.row_sum = rs;
  p.epi = a.epi;
  p.dev_status = dev_status;
  err = cudaFuncSetAttribute(int8_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const int grid = p.ntiles < sms ? p.ntiles : sms;
  int8_umma_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

}  // namespace qmm
