// W8A16: int8 weights with a scale for every 1,024 weights of a row, bf16
// activations ("llama.cpp-xdna -- CPU, iGPU and XDNA1 NPU on AMD Ryzen
// APUs", sections "The NPU worker" and "Running": in the GGML_XDNA_NPU_W8
// mode each 1,024-weight block of a row is int8 with its own scale, and the
// scale multiplies that block's partial sum).
//
// Pack: per (row n, block b of 1,024 k), packB's rule: s = fl(amax / 127),
// q = clamp(rint_even(fl(w / s)), -127, 127), 0 where s == 0.  Codes are
// [N][Kp] (Kp = K rounded up to 64, zero padding), scales [N][ceil(K/1024)].
//
// Decode GEMV for one token over many rows: the streaming ring kernel
// (w8_gemv_ring_kernel, below).  Otherwise (M <= 16, or few rows): a warp
// streams 32/G rows at once with G lanes per row, G sized so that every lane
// has about eight 16-byte groups of its row (a K = 1024 row is 1 KB: four
// rows per warp, 4 KB in flight per warp).  Each lane converts its codes
// exactly with a byte permute and one add (the int-to-float unit runs at a
// quarter of the fma rate) and multiplies them with x read through the
// read-only cache, even and odd columns as the two lanes of packed f32x2
// fmas.  Sixteen codes never straddle a 1,024 block, so
// each group's partial sum is scaled by its own block's scale.
#include <cuda_bf16.h>

#include <algorithm>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kW8Block = 1024;
constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads)
pack_w8_kernel(const float* __restrict__ W, int64_t ldw, int K, int Kp, int8_t* __restrict__ codes,
               float* __restrict__ scales, int nb) {
  __shared__ float red[kPackThreads / 32];
  const int n = blockIdx.x;
  const float* row = W + (int64_t)n * ldw;
  int8_t* out = codes + (int64_t)n * Kp;
  for (int b = 0; b < nb; ++b) {
    const int k0 = b * kW8Block, k1 = min(K, k0 + kW8Block);
    float a = 0.f;
    for (int k = k0 + (int)threadIdx.x; k < k1; k += kPackThreads) a = fmaxf(a, fabsf(row[k]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kPackThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) scales[(int64_t)n * nb + b] = s;
    for (int k = k0 + (int)threadIdx.x; k < k1; k += kPackThreads) {
      int q = 0;
      if (s > 0.f) q = min(max(__float2int_rn(__fdiv_rn(row[k], s)), -127), 127);
      out[k] = (int8_t)q;
    }
  }
  for (int k = K + (int)threadIdx.x; k < Kp; k += kPackThreads) out[k] = 0;
}

constexpr int kGvWarps = 8;
constexpr int kGvSteps = 8;   // 16-byte code groups in flight per lane

// 16 int8 codes as fp32 (exact), without the int-to-float unit.
__device__ __forceinline__ void codes16_to_f32(const uint4 v, float (&c)[16]) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[4 * i + j] = s8_byte_to_f32(w[i], j);
}

// A warp works on 32 / G rows at once, G lanes per row (G a power of two
// chosen so that a lane has about kGvSteps groups of its row): each load
// instruction of the warp reads G consecutive 16-byte groups of every one of
// its rows, and kGvSteps such loads are in flight before any is used.
template <int kM>
__global__ void __launch_bounds__(kGvWarps * 32)
w8_gemv_kernel(const int8_t* __restrict__ codes, const float* __restrict__ scales, int N, int K, int Kp, int nb,
               const __nv_bfloat16* __restrict__ X, int64_t ldx, float* __restrict__ Y, int64_t ldy, int M, int G) {
  const int lane = threadIdx.x & 31;
  const int R = 32 / G, sub = lane / G, sl = lane % G;
  const int warp_g = (int)blockIdx.x * kGvWarps + ((int)threadIdx.x >> 5);
  const int nwarps = (int)gridDim.x * kGvWarps;
  const int ngroups = Kp / 16;                       // 16-code groups of a row
  for (int n0 = warp_g * R; n0 < N; n0 += nwarps * R) {
    const int n = n0 + sub;
    const bool live = n < N;
    const uint4* row = reinterpret_cast<const uint4*>(codes + (int64_t)(live ? n : 0) * Kp);
    const float* srow = scales + (int64_t)(live ? n : 0) * nb;
    float acc[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) acc[m] = 0.f;
    for (int g0 = 0; g0 < ngroups; g0 += G * kGvSteps) {
      uint4 v[kGvSteps];
#pragma unroll
      for (int u = 0; u < kGvSteps; ++u) {
        const int g = g0 + G * u + sl;
        v[u] = (live && g < ngroups) ? ldg128_stream(row + g) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kGvSteps; ++u) {
        const int g = g0 + G * u + sl;
        if (!live || g >= ngroups) continue;
        const int k0 = 16 * g;
        if (k0 >= K) continue;   // padding codes are zero; x past K is not read
        float c[16];
        codes16_to_f32(v[u], c);
        const float s = __ldg(srow + k0 / kW8Block);
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          if (m >= M) break;
          const __nv_bfloat16* xr = X + (int64_t)m * ldx + k0;
          float part = 0.f;
          if (k0 + 16 <= K) {
            const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(xr));
            const uint4 x1 = __ldg(reinterpret_cast<const uint4*>(xr) + 1);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            // even and odd columns as the two lanes of packed f32x2 fmas
            uint64_t pp = f2_mul(f2_pack(c[0], c[1]), f2_pack(bf16lo_to_f32(xw[0]), bf16hi_to_f32(xw[0])));
#pragma unroll
            for (int i = 1; i < 8; ++i)
              pp = f2_fma(f2_pack(c[2 * i], c[2 * i + 1]), f2_pack(bf16lo_to_f32(xw[i]), bf16hi_to_f32(xw[i])), pp);
            float pe, po;
            f2_unpack(pp, pe, po);
            part = pe + po;
          } else {
            for (int i = 0; k0 + i < K; ++i) part = fmaf(c[i], __bfloat162float(xr[i]), part);
          }
          acc[m] = fmaf(part, s, acc[m]);
        }
      }
    }
    // sum over the G lanes of each row (G is a power of two: the xor partners
    // stay inside the row's lane group)
#pragma unroll
    for (int m = 0; m < kM; ++m) {
      if (m >= M) break;
      float a = acc[m];
      for (int o = G >> 1; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (sl == 0 && live) Y[(int64_t)m * ldy + n] = a;
    }
  }
}

// ---------------------------------------------------------------------------
// Streaming decode GEMV for one token over many rows.  One producer thread
// brings 32-row items of whole rows into a ring in shared memory, one TMA box
// per item, seen as {128 bytes, 32 rows, Kp / 128 k-blocks} with the 128-byte
// swizzle: the box lands as [k-block][row][128 bytes] with 16-byte unit u of
// row r at u ^ (r & 7), so the eight rows a quarter-warp reads sit in eight
// different bank groups.  Each consumer warp owns one ring slot and takes the
// items of that slot in order.  Lane (r, h) of a warp works on rows r and
// r + 16 over half h of the k-blocks, so every x value read from shared
// memory serves two rows; the halves are added with one shuffle.
// ---------------------------------------------------------------------------
constexpr int kW8RItemRows = 32;
constexpr int kW8RMaxWarps = 12;              // consumer warps = ring slots
constexpr size_t kW8RSmemCap = 227 * 1024;
constexpr int kW8RMaxKp = 2048;               // at most 3 scale blocks per lane

struct W8RingParams {
  CUtensorMap tm;                             // the codes as {128 bytes, rows, k-blocks}
  const int8_t* codes;
  const float* scales;
  int N, K, Kp, nb;
  const __nv_bfloat16* X;
  float* Y;
  int32_t* dev_status;
};

// 4 codes of a word (already XORed with 0x80808080) as two f32 pairs, exact.
__device__ __forceinline__ void w8_word_pairs(uint32_t w, uint64_t& p01, uint64_t& p23) {
  const uint64_t nbias = f2_pack(-8388736.0f, -8388736.0f);   // -(2^23 + 128)
  p01 = f2_add(f2_pack(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u)),
                       __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541u))), nbias);
  p23 = f2_add(f2_pack(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542u)),
                       __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543u))), nbias);
}

// 16 codes of one row times x (16 f32 in four 16-byte vectors) into the pair
// accumulator acc (even and odd k in its two halves).
__device__ __forceinline__ uint64_t w8_dot16(const uint4 c, const uint4 (&x)[4], uint64_t acc) {
  const uint32_t w[4] = {c.x ^ 0x80808080u, c.y ^ 0x80808080u, c.z ^ 0x80808080u, c.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint64_t p01, p23;
    w8_word_pairs(w[i], p01, p23);
    acc = f2_fma(p01, f2_pack(__uint_as_float(x[i].x), __uint_as_float(x[i].y)), acc);
    acc = f2_fma(p23, f2_pack(__uint_as_float(x[i].z), __uint_as_float(x[i].w)), acc);
  }
  return acc;
}

__device__ __forceinline__ float f2_sum(uint64_t v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return lo + hi;
}

__global__ void __launch_bounds__(32 * (kW8RMaxWarps + 1), 1) w8_gemv_ring_kernel(const __grid_constant__ W8RingParams p) {
  using namespace umma;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = smem_align(sm_raw, 1024);
  const int W = (int)blockDim.x / 32 - 1;                 // consumer warps, one ring slot each
  const uint32_t slot_bytes = (uint32_t)kW8RItemRows * (uint32_t)p.Kp;
  uint8_t* ring = sm;                                      // [W][Kp / 128][32][128], swizzled
  float* xs = reinterpret_cast<float*>(ring + (size_t)W * slot_bytes);   // [Kp], zeros past K
  uint64_t* full = reinterpret_cast<uint64_t*>(xs + p.Kp);
  uint64_t* empty = full + kW8RMaxWarps;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kW8RMaxWarps);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int items = (p.N + kW8RItemRows - 1) / kW8RItemRows;
  const int my_items = (int)blockIdx.x < items ? (items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int nkb = p.Kp / 128;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.tm);
    for (int s = 0; s < W; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();


  if (warp == W) {
    // ---- producer: items blockIdx.x, blockIdx.x + gridDim.x, ... ----
    if (lane == 0) {
      // the first two items into L2 while the previous grid finishes (the
      // copies into shared memory only start after the wait)
      for (int j = 0; j < my_items && j < 2; ++j) {
        const int row0 = ((int)blockIdx.x + j * (int)gridDim.x) * kW8RItemRows;
        const int rows = min(kW8RItemRows, p.N - row0);
        bulk_prefetch_l2(p.codes + (int64_t)row0 * p.Kp, (uint32_t)rows * (uint32_t)p.Kp);
      }
      pdl_wait();
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < my_items; ++j) {
        const int s = j % W;
        if (!mbar_wait(&empty[s], (uint32_t)(((j / W) & 1) ^ 1), abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        const int row0 = ((int)blockIdx.x + j * (int)gridDim.x) * kW8RItemRows;
        mbar_arrive_expect_tx(&full[s], slot_bytes);
        tma_load_3d(smem_u32(ring) + (uint32_t)s * slot_bytes, &p.tm, &full[s], 0, row0, 0);
        ++issued;
      }
      if (!ok) {
        // the items already issued land before the CTA leaves: each slot's
        // last issued phase, whether or not it was consumed
        for (int s = 0; s < W && s < issued; ++s) {
          const int last = issued - 1 - ((issued - 1 - s) % W);
          mbar_drain(&full[s], (uint32_t)((last / W) & 1));
        }
      }
    }
    return;
  }

  // ---- consumers: x as f32 into shared memory, then the items of this
  // warp's slot ----
  pdl_wait();   // x and y may belong to the previous grid
  for (int k = threadIdx.x; k < p.Kp; k += W * 32) xs[k] = k < p.K ? __bfloat162float(p.X[k]) : 0.f;
  asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
  const int r = lane & 15, h = lane >> 4;
  const int kb0 = h ? (nkb + 1) / 2 : 0, kb1 = h ? nkb : (nkb + 1) / 2;   // this lane's k-blocks
  const int b0 = (kb0 * 128) >> 10;                                       // its first scale block
  const uint32_t xsa = smem_u32(xs);
  for (int j = warp; j < my_items; j += W) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[warp], (uint32_t)((j / W) & 1), abort_flag, p.dev_status)))
      break;
    const int n0 = ((int)blockIdx.x + j * (int)gridDim.x) * kW8RItemRows + r, n1 = n0 + 16;
    // the scales of (at most) three blocks from b0 for both rows, read ahead
    float sA[3], sB[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int b = b0 + q;
      sA[q] = (n0 < p.N && b < p.nb) ? __ldg(p.scales + (int64_t)n0 * p.nb + b) : 0.f;
      sB[q] = (n1 < p.N && b < p.nb) ? __ldg(p.scales + (int64_t)n1 * p.nb + b) : 0.f;
    }
    const uint32_t rowA = smem_u32(ring) + (uint32_t)warp * slot_bytes + (uint32_t)r * 128u;
    const uint32_t rowB = rowA + 16u * 128u;
    float yA = 0.f, yB = 0.f;
    uint64_t accA = 0ull, accB = 0ull;   // pair sums of the current scale block
    int q = 0;                           // current block, relative to b0
    for (int kb = kb0; kb < kb1; ++kb) {
      const int bq = ((kb * 128) >> 10) - b0;
      if (bq != q) {   // a new scale block: close the previous one
        yA = fmaf(f2_sum(accA), q == 0 ? sA[0] : (q == 1 ? sA[1] : sA[2]), yA);
        yB = fmaf(f2_sum(accB), q == 0 ? sB[0] : (q == 1 ? sB[1] : sB[2]), yB);
        accA = 0ull;
        accB = 0ull;
        q = bq;
      }
      const uint32_t off = (uint32_t)kb * (uint32_t)(kW8RItemRows * 128);
#pragma unroll 4
      for (int u = 0; u < 8; ++u) {
        const uint32_t sw = (uint32_t)((u ^ (r & 7)) << 4);
        const uint4 cA = lds128(rowA + off + sw);
        const uint4 cB = lds128(rowB + off + sw);
        const uint32_t xa = xsa + (uint32_t)(kb * 128 + 16 * u) * 4u;
        const uint4 xv[4] = {lds128(xa), lds128(xa + 16u), lds128(xa + 32u), lds128(xa + 48u)};
        accA = w8_dot16(cA, xv, accA);
        accB = w8_dot16(cB, xv, accB);
      }
    }
    if (kb1 > kb0) {
      yA = fmaf(f2_sum(accA), q == 0 ? sA[0] : (q == 1 ? sA[1] : sA[2]), yA);
      yB = fmaf(f2_sum(accB), q == 0 ? sB[0] : (q == 1 ? sB[1] : sB[2]), yB);
    }
    // every lane's reads of this slot are done
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[warp]);
    yA += __shfl_xor_sync(0xffffffffu, yA, 16);
    yB += __shfl_xor_sync(0xffffffffu, yB, 16);
    if (h == 0) {
      if (n0 < p.N) p.Y[n0] = yA;
      if (n1 < p.N) p.Y[n1] = yB;
    }
  }
}

}  // namespace

int64_t w8_padded_k(int64_t K) { return (K + 63) / 64 * 64; }
int64_t w8_blocks(int64_t K) { return (K + kW8Block - 1) / kW8Block; }

cudaError_t launch_pack_w8(const float* W, int N, int K, int64_t ldw, int8_t* codes, float* scales,
                           cudaStream_t stream) {
  pack_w8_kernel<<<N, kPackThreads, 0, stream>>>(W, ldw, K, (int)w8_padded_k(K), codes, scales, (int)w8_blocks(K));
  return cudaGetLastError();
}

cudaError_t launch_w8_gemv(const int8_t* codes, const float* scales, int N, int K, const __nv_bfloat16* X,
                           int64_t ldx, int M, float* Y, int64_t ldy, int32_t* dev_status, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int Kp = (int)w8_padded_k(K), nb = (int)w8_blocks(K);
  if (M == 1 && Kp % 128 == 0 && Kp <= kW8RMaxKp && N / kW8RItemRows >= 2 * sms) {
    // one token over many rows: the streaming ring kernel, with at least
    // three 32-row items in flight per SM
    const size_t slot_bytes = (size_t)kW8RItemRows * Kp;
    const size_t fixed = 1024 + (size_t)Kp * 4 + 2 * kW8RMaxWarps * 8 + 16;
    const int W = (int)std::min<size_t>((kW8RSmemCap - fixed) / slot_bytes, kW8RMaxWarps);
    if (W >= 3) {
      W8RingParams p{};
      if (!make_tmap_kblocks128_sw(&p.tm, codes, (uint64_t)N, (uint64_t)Kp, (uint64_t)(Kp / 128), kW8RItemRows,
                                   (uint32_t)(Kp / 128)))
        return cudaErrorInvalidValue;
      p.codes = codes;
      p.scales = scales;
      p.N = N;
      p.K = K;
      p.Kp = Kp;
      p.nb = nb;
      p.X = X;
      p.Y = Y;
      p.dev_status = dev_status;
      const size_t smem = fixed + (size_t)W * slot_bytes;
      const cudaError_t e =
          cudaFuncSetAttribute(w8_gemv_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_pdl(w8_gemv_ring_kernel, dim3((unsigned)sms), dim3(32 * (W + 1)), smem, stream, p);
    }
  }
  // lanes per row: about kGvSteps groups each, at least 4 lanes, at most 32
  int G = 32;
  while (G > 4 && G * kGvSteps > Kp / 16) G >>= 1;
  const int R = 32 / G;
  const int rows_per_block = kGvWarps * R;
  const int grid = std::max(1, std::min((N + rows_per_block - 1) / rows_per_block, 8 * sms));
  if (M <= 1)
    w8_gemv_kernel<1><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  else if (M <= 4)
    w8_gemv_kernel<4><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  else
    w8_gemv_kernel<16><<<grid, kGvWarps * 32, 0, stream>>>(codes, scales, N, K, Kp, nb, X, ldx, Y, ldy, M, G);
  return cudaGetLastError();
}

}  // namespace qmm
