// MUL_MAT_ID on q4_1 tiles: for every (token t, slot i), dst[t][i] = W_e . src1
// with e = ids[t * ld_ids + i] ("Zaya 8B Q4NX on the AMD NPU", "The bugs that
// were the work": the ids are a strided view, and the down projection reads a
// per-slot src1 row).  Weights are 32x256 q4_1 tiles, w = q * scale + min
// ("NPU engine: full ELFs, no xclbin", "Q4NX chunks").
//
// One CTA owns 128 weight rows of one expert and every (token, slot) pair
// routed to that expert, up to 64 pairs per pass.  Each weight is read from
// HBM once per pass and used for all of the pass's pairs, which is the
// grouped dispatch the pages credit for the MoE speed-up.
//
//   * Routing.  When T * n_used is small the CTA scans the ids itself: every
//     thread marks the hits in its own run of pairs in a bit mask, and a CTA
//     prefix sum gives each hit its rank, so the pairs of an expert keep pair
//     order.  Larger batches run a one-CTA router first, which writes per-expert
//     offsets and pair lists into the caller's workspace.
//   * Staging.  cp.async moves half a tile column (128 K) per stage: the code
//     bytes of the CTA's 128 rows, their (scale, min) pairs, and the 64
//     gathered activation rows.  Both land in shared memory with an XOR
//     swizzle on 16-byte units, so the fragment reads below are free of bank
//     conflicts.  Four stages are in flight.
//   * Math.  Each warp owns 16 weight rows.  ldmatrix hands every lane the code
//     word of its MMA rows; a lop3 turns two codes into (128 + q) bf16 pairs,
//     and q * scale + min is formed in bf16 with one rounding (sub, then fma).
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate) multiplies them with eight
//     pairs' activations per column group.  The k order inside each MMA is a
//     permutation of the block's 32 columns, the same on both operands.
//
// The work is bound by the weight stream (one pass reads 0.625 bytes per
// weight and does 2 * pairs flops per weight), so the legacy MMA is enough:
// the tensor pipe is not the limit at these pair counts.
#include <cuda_bf16.h>

#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kThreads = 256;                 // 8 warps x 16 weight rows
constexpr int kRows = 128;                    // weight rows per CTA
constexpr int kTok = 64;                      // pairs per pass (8 MMA column groups)
constexpr int kKC = 128;                      // K per stage: half a tile column
constexpr int kStages = 4;
constexpr int kCodeBytes = kRows * 64;        // 8 KB: 4 blocks x 16 B per row
constexpr int kPairBytes = kRows * 16;        // 2 KB: 4 (scale, min) pairs per row
constexpr int kXBytes = kTok * kKC * 2;       // 16 KB
constexpr int kStageBytes = kCodeBytes + kPairBytes + kXBytes;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes;
constexpr int kScanMaxPairs = 32 * kThreads;  // one 32-bit hit mask per thread

struct MoeParams {
  const uint8_t* tiles;
  int64_t expert_bytes;
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// src_bytes = 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

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

// Weight part of one stage: codes of blocks 4h..4h+3 of tile column tc for
// the CTA's 128 rows, and their (scale, min) pairs.  Code unit j of row r
// goes to 16-byte slot j ^ ((r >> 1) & 3): the 8 rows of an ldmatrix phase
// then cover all 32 banks.
__device__ __forceinline__ void load_weights(const MoeParams& p, const uint8_t* etiles, int n0, int ks,
                                             uint32_t sbase) {
  const int TC = p.K / 256;
  const int tc = ks >> 1, h = ks & 1;
  for (int i = threadIdx.x; i < kRows * 5; i += kThreads) {
    if (i < kRows * 4) {
      const int r = i >> 2, j = i & 3;
      const int n = n0 + r;
      if (n < p.N) {
        const uint8_t* src = etiles + ((int64_t)(n >> 5) * TC + tc) * kTileBytes + (n & 31) * 128 + 64 * h + 16 * j;
        cp_async16(sbase + r * 64 + 16 * (j ^ ((r >> 1) & 3)), src);
      }
    } else {
      const int r = i - kRows * 4;
      const int n = n0 + r;
      if (n < p.N) {
        const uint8_t* src = etiles + ((int64_t)(n >> 5) * TC + tc) * kTileBytes + 4096 + (n & 31) * 32 + 16 * h;
        cp_async16(sbase + kCodeBytes + r * 16, src);
      }
    }
  }
}

// Activation part of one stage: 16-byte unit u (8 columns) of pair column c
// goes to slot u ^ (c & 7).  Columns past the pass's pair count are zero.
__device__ __forceinline__ void load_x(const MoeParams& p, const int64_t* xoff, int nt, int ncol, int ks,
                                       uint32_t sbase) {
  const uint32_t sx = sbase + kCodeBytes + kPairBytes;
  for (int i = threadIdx.x; i < ncol * 16; i += kThreads) {
    const int c = i >> 4, u = i & 15;
    const bool valid = c < nt;
    const __nv_bfloat16* src = valid ? p.X + xoff[c] + (int64_t)ks * kKC + 8 * u : p.X;
    cp_async16_zfill(sx + c * 256 + 16 * (u ^ (c & 7)), src, valid ? 16 : 0);
  }
}

template <int kNG>
__device__ __forceinline__ void compute_stage(uint32_t sbase, int warp, int lane, int ngroups,
                                              float (&acc)[kNG][4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t sc = sbase, sp = sbase + kCodeBytes, sx = sbase + kCodeBytes + kPairBytes;
  // ldmatrix: lanes 8i..8i+7 address the rows of matrix i.  Matrix i of the
  // first load is (row half i & 1, block i >> 1); the second covers blocks 2, 3.
  const int rr = 16 * warp + 8 * ((lane >> 3) & 1) + (lane & 7);
  const int jm = lane >> 4;
  const int sw = (rr >> 1) & 3;
  uint32_t cw[8];
  ldmatrix_x4(sc + rr * 64 + 16 * (jm ^ sw), cw[0], cw[1], cw[2], cw[3]);
  ldmatrix_x4(sc + rr * 64 + 16 * ((jm + 2) ^ sw), cw[4], cw[5], cw[6], cw[7]);
  const uint4 pa = lds128(sp + (16 * warp + g) * 16);
  const uint4 pb = lds128(sp + (16 * warp + 8 + g) * 16);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t wA = cw[2 * j], wB = cw[2 * j + 1];
    const uint32_t pA = u4_get(pa, j), pB = u4_get(pb, j);
    const uint32_t sA = __byte_perm(pA, 0, 0x1010), mA = __byte_perm(pA, 0, 0x3232);
    const uint32_t sB = __byte_perm(pB, 0, 0x1010), mB = __byte_perm(pB, 0, 0x3232);
    const uint32_t a0 = dequant2(q4_pair_biased(wA, 0), sA, mA);
    const uint32_t a1 = dequant2(q4_pair_biased(wB, 0), sB, mB);
    const uint32_t a2 = dequant2(q4_pair_biased(wA, 1), sA, mA);
    const uint32_t a3 = dequant2(q4_pair_biased(wB, 1), sB, mB);
    const uint32_t a4 = dequant2(q4_pair_biased(wA, 2), sA, mA);
    const uint32_t a5 = dequant2(q4_pair_biased(wB, 2), sB, mB);
    const uint32_t a6 = dequant2(q4_pair_biased(wA, 3), sA, mA);
    const uint32_t a7 = dequant2(q4_pair_biased(wB, 3), sB, mB);
    const uint32_t xcol = sx + g * 256 + 16 * ((4 * j + t) ^ g);
#pragma unroll
    for (int ng = 0; ng < kNG; ++ng) {
      if (ng < ngroups) {
        const uint4 xv = lds128(xcol + ng * 8 * 256);
        mma_bf16_16816(acc[ng], a0, a1, a2, a3, xv.x, xv.y);
        mma_bf16_16816(acc[ng], a4, a5, a6, a7, xv.z, xv.w);
      }
    }
  }
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

// Weights of stages 0 .. kStages-2 into buffers 0 .. kStages-2, one commit
// group per stage (empty groups past the last stage keep the count fixed).
__device__ __forceinline__ void issue_weight_prologue(const MoeParams& p, const uint8_t* etiles, int n0,
                                                      int nks, uint32_t sbase0) {
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nks) load_weights(p, etiles, n0, s, sbase0 + s * kStageBytes);
    cp_async_commit();
  }
}

template <bool kScan>
__global__ void __launch_bounds__(kThreads, 2) q4_moe_kernel(const MoeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int64_t xoff[kTok], yoff[kTok];
  __shared__ int wsum[kThreads / 32];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.y;
  const int n0 = blockIdx.x * kRows;
  const int nks = p.K / kKC;
  const uint8_t* etiles = p.tiles + (int64_t)e * p.expert_bytes;
  const uint32_t sbase0 = smem_addr(smem);
  const bool rows_live = n0 + 16 * warp < p.N;

  // When most experts receive pairs, the weights of the first stages are
  // fetched before the routing is known: they do not depend on it.
  const int npairs = p.T * p.n_used;
  const bool early = npairs >= p.n_expert;
  if (early) issue_weight_prologue(p, etiles, n0, nks, sbase0);

  // ---- this expert's pairs ----
  uint32_t mask = 0;
  int first = 0, total = 0, rank0 = 0;
  if (kScan) {
    const int per = (npairs + kThreads - 1) / kThreads;   // <= 32
    first = threadIdx.x * per;
    int id[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int pr = first + j;
      id[j] = -1;
      if (j < per && pr < npairs) id[j] = p.ids[(int64_t)(pr / p.n_used) * p.ld_ids + (pr % p.n_used)];
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int pr = first + j;
      if (j < per && pr < npairs) {
        if (id[j] == e) mask |= 1u << j;
        bad |= (id[j] < 0 || id[j] >= p.n_expert);
      }
    }
    if (bad && blockIdx.x == 0 && blockIdx.y == 0) set_status(p.dev_status, QMM_ERR_BAD_EXPERT_ID);
    rank0 = cta_exclusive_scan(__popc(mask), wsum, total);
  } else {
    first = p.offsets[e];
    total = p.offsets[e + 1] - first;
  }
  if (total == 0) {
    cp_async_wait<0>();   // no copy may land after the CTA has left
    return;
  }

  for (int pass0 = 0; pass0 < total; pass0 += kTok) {
    const int nt = min(kTok, total - pass0);
    const int ngroups = (nt + 7) >> 3;
    if (pass0 > 0 || !early) issue_weight_prologue(p, etiles, n0, nks, sbase0);
    if (kScan) {
      uint32_t m = mask;
      int r = rank0;
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        if (r >= pass0 && r < pass0 + kTok) pair_offsets(p, first + j, xoff[r - pass0], yoff[r - pass0]);
        ++r;
      }
    } else {
      for (int c = threadIdx.x; c < nt; c += kThreads)
        pair_offsets(p, p.pairs[first + pass0 + c], xoff[c], yoff[c]);
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < nks) load_x(p, xoff, nt, 8 * ngroups, s, sbase0 + s * kStageBytes);
      cp_async_commit();
    }

    float acc[8][4];
#pragma unroll
    for (int ng = 0; ng < 8; ++ng)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[ng][c] = 0.f;

    for (int ks = 0; ks < nks; ++ks) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      const int kn = ks + kStages - 1;
      if (kn < nks) {
        const uint32_t sb = sbase0 + (kn % kStages) * kStageBytes;
        load_weights(p, etiles, n0, kn, sb);
        load_x(p, xoff, nt, 8 * ngroups, kn, sb);
      }
      cp_async_commit();
      if (rows_live) compute_stage<8>(sbase0 + (ks % kStages) * kStageBytes, warp, lane, ngroups, acc);
    }
    cp_async_wait<0>();

    if (rows_live) {
      const int g = lane >> 2, t = lane & 3;
      const int nrow = n0 + 16 * warp + g;
#pragma unroll
      for (int ng = 0; ng < 8; ++ng) {
        if (ng < ngroups) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = 8 * ng + 2 * t + (c & 1);
            if (col < nt) p.Y[yoff[col] + nrow + 8 * (c >> 1)] = acc[ng][c];
          }
        }
      }
    }
    __syncthreads();   // xoff / yoff and the stage buffers are reused by the next pass
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

template <bool kScan>
cudaError_t launch_grouped(const MoeParams& p, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(q4_moe_kernel<kScan>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)((p.N + kRows - 1) / kRows), (unsigned)p.n_expert);
  q4_moe_kernel<kScan><<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t q4_moe_workspace_bytes(int64_t n_expert, int64_t n_used, int64_t T) {
  const size_t off = ((size_t)(n_expert + 1) * 4 + 255) / 256 * 256;
  return off + (size_t)(T * n_used) * 4;
}

cudaError_t launch_q4_moe(const Q4MoEArgs& a, cudaStream_t stream) {
  MoeParams p{};
  p.tiles = a.tiles;
  p.expert_bytes = (int64_t)(a.N / 32) * (a.K / 256) * kTileBytes;
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
  if ((int64_t)a.T * a.n_used <= kScanMaxPairs) return launch_grouped<true>(p, stream);
  const size_t smem = (size_t)a.n_expert * 2 * sizeof(int);
  moe_route_kernel<<<1, 1024, smem, stream>>>(a.ids, a.ld_ids, a.n_used, a.T, a.n_expert, a.offsets,
                                              a.pairs, a.dev_status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  p.offsets = a.offsets;
  p.pairs = a.pairs;
  return launch_grouped<false>(p, stream);
}

}  // namespace qmm
