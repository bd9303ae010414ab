// Exact int8 GEMM for small M (<= 64 rows): the weight-streaming regime of
// the int8 half ("int8 inference", "Product kernel (Int8Gemm)"; "The ONNX
// pack: weights to Q4NX, matmuls to our kernels, no VitisAI", "What works
// today": the M = 16 / 32 projection GEMMs).
//
// Integer route.  On this GPU the legacy integer MMA (m16n8k32 s8) and dp4a
// both run near 158 TOPS, while the f16 MMA (m16n8k16, fp32 accumulation)
// runs near 600 TFLOPS.  So the codes are widened to f16, which is exact for
// |A'|, |B'| <= 128, and multiplied there: every product is an integer of at
// most 2^14, a sum of up to 1024 of them is an integer below 2^24 and hence
// exact in fp32, and the accumulators are drained into int32 every 1024 k.
//
// Work split.  A cluster of 8 CTAs owns 64 output columns; CTA r takes the
// r-th eighth of K in whole 64-k steps.  It stages its slice of A' as f16 in
// shared memory (all 64 columns reuse it) together with the slice's partial
// row sums, and each of its 8 warps streams the slice of 8 weight columns
// straight from HBM, 16 bytes per lane and step.  Inside a step, lane t of a
// quad holds bytes 16t..16t+15 of a row, and the MMA's logical k order is a
// permutation of those bytes that A and B share, so the sum is unchanged.
// The partial S and row sums are exact integers: each warp stores its 8
// columns' partials into the CTA of the cluster that owns those columns
// (distributed shared memory, one slot per source CTA), and after one
// cluster barrier every CTA adds its 8 slots and applies the zero-point
// correction, bias and output conversion to its own 8 columns.
#include <mutex>
#include <vector>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

constexpr int kCluster = 8;        // K slices of one column block
constexpr int kWarps = 8;          // one 8-column n-block per warp
constexpr int kCols = 8 * kWarps;  // columns of a cluster
constexpr int kStepsInFlight = 8;  // 64-k steps of weights loaded ahead per warp
constexpr size_t kSmemBudget = 160 * 1024;

struct SmallParams {
  const int8_t* A;
  int64_t lda;
  int M, K, N;
  uint32_t a_xor;        // 0x80808080 for uint8 A (A' = A - 128 is A with the top bit flipped), else 0
  const int8_t* B;       // packed [N][Kp]
  int64_t Kp;
  int need_rowsum;
  Int8Epi epi;
};

// Several problems in one launch: problem i owns clusters
// [cluster_begin[i], cluster_begin[i + 1]), one per 64 output columns.
constexpr int kMaxGroup = 16;
struct SmallGroup {
  SmallParams prob[kMaxGroup];
  int32_t cluster_begin[kMaxGroup + 1];
  int32_t nprob;
};
constexpr size_t kParamSlot = (sizeof(SmallParams) + 15) / 16 * 16;   // the problem's copy in shared memory

// Four int8 codes (A' or B', two's complement) as two f16x2 pairs, exactly:
// byte b + 128 becomes the low mantissa byte of 1024 (f16 0x6400), and
// 1024 + 128 is subtracted.
QMM_DEV void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140u);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342u);
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));   // 1152 = 0x6480
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// Stores into shared memory of any CTA of the cluster (cluster address).
QMM_DEV void st_dsmem_v2(uint32_t cluster_addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(cluster_addr), "r"(a), "r"(b) : "memory");
}
QMM_DEV void st_dsmem(uint32_t cluster_addr, uint32_t a) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(a) : "memory");
}

template <int MT>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWarps * 32)
    int8_small_kernel(const __grid_constant__ SmallGroup gp) {
  using namespace umma;
  extern __shared__ __align__(16) uint8_t sm_all[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int rank = (int)cluster_ctarank();
  // this cluster's problem and column block; the problem's parameters are
  // copied into shared memory once (they are read throughout)
  const int cl = (int)(blockIdx.x / kCluster);
  int pi = 0;
  while (pi + 1 < gp.nprob && gp.cluster_begin[pi + 1] <= cl) ++pi;
  SmallParams* ps = reinterpret_cast<SmallParams*>(sm_all);
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&gp.prob[pi]);
    uint32_t* dst = reinterpret_cast<uint32_t*>(ps);
    for (int i = threadIdx.x; i < (int)(sizeof(SmallParams) / 4); i += kWarps * 32) dst[i] = src[i];
  }
  __syncthreads();
  const SmallParams& p = *ps;
  uint8_t* sm = sm_all + kParamSlot;
  const int n0 = (cl - gp.cluster_begin[pi]) * kCols;
  const int S64 = (int)(p.Kp / 64);
  const int s0 = rank * S64 / kCluster, s1 = (rank + 1) * S64 / kCluster;
  const int nsteps = s1 - s0, klen = nsteps * 64;
  const int SA = klen + 8;                                          // f16 row stride (16-byte pad)
  // The accumulators sit at the same offsets in every CTA of the cluster (the
  // slices, and so the staged A', may differ in length by one step).
  int32_t* xfer = reinterpret_cast<int32_t*>(sm);                   // [kCluster][MT*16][8]: each CTA's partial S of this CTA's columns
  int32_t* rs_x = xfer + kCluster * MT * 16 * 8;                    // [kCluster][MT*16]: each CTA's partial row sums
  int32_t* rsum = rs_x + kCluster * MT * 16;                        // [MT*16]: row sums over this slice
  __half* As = reinterpret_cast<__half*>(rsum + MT * 16);           // [MT*16][SA]

  umma::pdl_launch_dependents();
  for (int i = threadIdx.x; i < MT * 16; i += kWarps * 32) rsum[i] = 0;
  // this warp's weights: column n0 + 8 warp + g, bytes 16t.. of each step;
  // warm them in L2 while the previous grid finishes (only the loads into
  // registers must follow the dependency wait)
  const int ncol = n0 + 8 * warp + g;
  const bool col_ok = ncol < p.N;
  const int8_t* brow = p.B + (int64_t)(col_ok ? ncol : 0) * p.Kp + (int64_t)s0 * 64 + 16 * t;
  if (t == 0 && col_ok && klen > 0) bulk_prefetch_l2(brow, (uint32_t)klen);
  umma::pdl_wait();   // A and the weights may come from the previous grid

  uint4 breg[kStepsInFlight];
#pragma unroll
  for (int j = 0; j < kStepsInFlight; ++j)
    breg[j] = (j < nsteps && col_ok) ? ldg128_stream(brow + 64 * j) : make_uint4(0u, 0u, 0u, 0u);

  // A' slice as f16 (zeros past M and K) and its partial row sums
  __syncthreads();   // rsum zeroed
  const int kq = klen / 16;
  for (int c = threadIdx.x; c < MT * 16 * kq; c += kWarps * 32) {
    const int row = c / kq, kl = (c - row * kq) * 16;
    const int k = s0 * 64 + kl;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (row < p.M && k < p.K) {
      const int8_t* src = p.A + (int64_t)row * p.lda + k;
      if (k + 16 <= p.K) {
        w = ldg128(src);
      } else {
        uint32_t b[4] = {0u, 0u, 0u, 0u};
        for (int e = 0; k + e < p.K; ++e) b[e >> 2] |= (uint32_t)(uint8_t)src[e] << (8 * (e & 3));
        w = make_uint4(b[0], b[1], b[2], b[3]);
      }
      // A' as int8: u8 codes move down by 128, int8 codes stay; bytes past K stay 0
      const uint32_t x = p.a_xor;
      const int valid = min(16, p.K - k);
      uint32_t m[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = valid - 4 * q;
        m[q] = v >= 4 ? 0xFFFFFFFFu : (v <= 0 ? 0u : (0xFFFFFFFFu >> (32 - 8 * v)));
      }
      w.x = (w.x ^ x) & m[0];
      w.y = (w.y ^ x) & m[1];
      w.z = (w.z ^ x) & m[2];
      w.w = (w.w ^ x) & m[3];
      if (p.need_rowsum) {
        int s = __dp4a((int)w.x, 0x01010101, 0);
        s = __dp4a((int)w.y, 0x01010101, s);
        s = __dp4a((int)w.z, 0x01010101, s);
        s = __dp4a((int)w.w, 0x01010101, s);
        atomicAdd(&rsum[row], s);
      }
    }
    uint32_t f[8];
    s8x4_to_f16x4(w.x, f[0], f[1]);
    s8x4_to_f16x4(w.y, f[2], f[3]);
    s8x4_to_f16x4(w.z, f[4], f[5]);
    s8x4_to_f16x4(w.w, f[6], f[7]);
    const uint32_t dst = smem_u32(As + row * SA + kl);
    sts128(dst, make_uint4(f[0], f[1], f[2], f[3]));
    sts128(dst + 16, make_uint4(f[4], f[5], f[6], f[7]));
  }
  __syncthreads();

  // S partial: fp32 chunks of at most 1024 k (16 steps), drained into int32
  int acc[MT][4];
  float accf[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) { acc[mt][e] = 0; accf[mt][e] = 0.f; }
  for (int j0 = 0; j0 < nsteps; j0 += kStepsInFlight) {
#pragma unroll
    for (int j = 0; j < kStepsInFlight; ++j) {
      if (j0 + j < nsteps) {
        const uint4 bw = breg[j];
        uint32_t bl[4], bh[4];
        s8x4_to_f16x4(bw.x, bl[0], bh[0]);
        s8x4_to_f16x4(bw.y, bl[1], bh[1]);
        s8x4_to_f16x4(bw.z, bl[2], bh[2]);
        s8x4_to_f16x4(bw.w, bl[3], bh[3]);
        const int kl = (j0 + j) * 64 + 16 * t;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t r0 = smem_u32(As + (mt * 16 + g) * SA + kl);
          const uint32_t r1 = smem_u32(As + (mt * 16 + g + 8) * SA + kl);
          const uint4 a00 = lds128(r0), a01 = lds128(r0 + 16);
          const uint4 a10 = lds128(r1), a11 = lds128(r1 + 16);
          const uint32_t ra[8] = {a00.x, a00.y, a00.z, a00.w, a01.x, a01.y, a01.z, a01.w};
          const uint32_t rb[8] = {a10.x, a10.y, a10.z, a10.w, a11.x, a11.y, a11.z, a11.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mma_f16_16816(accf[mt], ra[2 * i], rb[2 * i], ra[2 * i + 1], rb[2 * i + 1], bl[i], bh[i]);
        }
        if (((j0 + j + 1) & 15) == 0) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) { acc[mt][e] += __float2int_rn(accf[mt][e]); accf[mt][e] = 0.f; }
        }
      }
    }
    if (j0 + kStepsInFlight < nsteps) {
#pragma unroll
      for (int j = 0; j < kStepsInFlight; ++j)
        breg[j] = (j0 + kStepsInFlight + j < nsteps && col_ok)
                      ? ldg128_stream(brow + 64 * (j0 + kStepsInFlight + j))
                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mt][e] += __float2int_rn(accf[mt][e]);
  // Warp w's 8 columns belong to CTA w of the cluster: store the exact
  // partials into that CTA's slot for this CTA, and this slice's row sums into
  // every CTA.  Each slot is written once, so no atomics are needed.
  {
    const uint32_t owner = (uint32_t)warp;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const uint32_t a0 = mapa_shared(smem_u32(xfer + ((rank * MT + mt) * 16 + g) * 8 + 2 * t), owner);
      st_dsmem_v2(a0, (uint32_t)acc[mt][0], (uint32_t)acc[mt][1]);
      st_dsmem_v2(a0 + 8u * 8u * 4u, (uint32_t)acc[mt][2], (uint32_t)acc[mt][3]);   // row g + 8
    }
  }
  if (p.need_rowsum) {
    __syncthreads();   // this slice's row sums are complete
    for (int o = threadIdx.x; o < p.M * kCluster; o += kWarps * 32) {
      const int m = o / kCluster, q = o - m * kCluster;
      st_dsmem(mapa_shared(smem_u32(rs_x + rank * MT * 16 + m), (uint32_t)q), (uint32_t)rsum[m]);
    }
  }
  cluster_sync();   // all partials landed; nothing touches another CTA's memory after this

  // columns 8 rank .. 8 rank + 7 of the block: the sum of the 8 partials, then
  // zero-point correction, bias and output conversion
  for (int o = threadIdx.x; o < p.M * 8; o += kWarps * 32) {
    const int m = o >> 3, c = o & 7;
    const int n = n0 + 8 * rank + c;
    uint32_t S = 0u, rs = 0u;
#pragma unroll
    for (int q = 0; q < kCluster; ++q) {
      S += (uint32_t)xfer[((q * MT) * 16 + m) * 8 + c];
      rs += (uint32_t)rs_x[q * MT * 16 + m];
    }
    if (n < p.N) int8_store(p.epi, m, n, zp_correct((int32_t)S, p.epi.col_sum[n], (int32_t)rs, p.epi));
  }
}

size_t small_smem(int MT, int64_t Kp) {
  const int S64 = (int)(Kp / 64);
  const int klen = (S64 + kCluster - 1) / kCluster * 64;
  return kParamSlot + (size_t)MT * 16 * (klen + 8) * 2 + (size_t)MT * 16 * (8 * kCluster + kCluster + 1) * 4;
}

SmallParams small_params(const Int8GemmArgs& a) {
  SmallParams p{};
  p.A = a.A;
  p.lda = a.lda;
  p.M = a.M;
  p.K = a.K;
  p.N = a.N;
  p.a_xor = a.a_u8 ? 0x80808080u : 0u;
  p.B = a.B;
  p.Kp = a.Kp;
  p.need_rowsum = a.need_rowsum ? 1 : 0;
  p.epi = a.epi;
  return p;
}

template <int MT>
cudaError_t launch_mt(const SmallGroup& gp, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(int8_small_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)gp.cluster_begin[gp.nprob] * kCluster;
  return launch_pdl(int8_small_kernel<MT>, dim3(grid), dim3(kWarps * 32), smem, stream, gp);
}

}  // namespace

bool int8_small_eligible(int64_t M, int64_t K, int64_t N) {
  return M >= 1 && M <= 64 && N >= 1 && (N + kCols - 1) / kCols * kCluster <= INT32_MAX &&
         small_smem((int)(M + 15) / 16, padded_k(K)) <= kSmemBudget;
}

namespace {

// The cluster form on up to kMaxGroup problems in one launch.
cudaError_t launch_cluster_batch(const std::vector<Int8GemmArgs>& probs, cudaStream_t stream) {
  const int cnt = (int)probs.size();
  static SmallGroup gp;   // host staging copy; the launch copies it into the parameter space
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  gp = SmallGroup{};
  int MT = 1;
  int64_t clusters = 0, kp_max = 0;
  for (int i = 0; i < cnt; ++i) {
    const Int8GemmArgs& a = probs[i];
    gp.prob[i] = small_params(a);
    gp.cluster_begin[i] = (int32_t)clusters;
    clusters += (a.N + kCols - 1) / kCols;
    MT = MT > (a.M + 15) / 16 ? MT : (a.M + 15) / 16;
    kp_max = kp_max > a.Kp ? kp_max : a.Kp;
  }
  gp.cluster_begin[cnt] = (int32_t)clusters;
  gp.nprob = cnt;
  if (clusters * kCluster > INT32_MAX) return cudaErrorInvalidConfiguration;
  const size_t smem = small_smem(MT, kp_max);
  if (smem > kSmemBudget) return cudaErrorInvalidConfiguration;
  if (MT == 1) return launch_mt<1>(gp, smem, stream);
  if (MT == 2) return launch_mt<2>(gp, smem, stream);
  if (MT == 3) return launch_mt<3>(gp, smem, stream);
  return launch_mt<4>(gp, smem, stream);
}

}  // namespace

cudaError_t launch_int8_small_group(const Int8GemmArgs* probs, int n, int32_t* dev_status, cudaStream_t stream) {
  // Problems whose rows fit the streaming form's shared memory are gathered
  // into batches that fit together; a batch with at least one item (16
  // columns) per SM streams, a smaller one (too few items to fill the GPU
  // without splitting K) joins the rest in the cluster form, up to kMaxGroup
  // problems per launch.  The problems are independent, so launch order is free.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  std::vector<Int8GemmArgs> st, cl;
  cudaError_t e = cudaSuccess;
  auto to_cluster = [&](const Int8GemmArgs& a) {
    cl.push_back(a);
    if ((int)cl.size() == kMaxGroup) {
      if (e == cudaSuccess) e = launch_cluster_batch(cl, stream);
      cl.clear();
    }
  };
  auto flush_stream = [&]() {
    if (st.empty()) return;
    if (int8_stream_items(st.data(), (int)st.size()) >= sms) {
      if (e == cudaSuccess) e = launch_int8_stream_group(st.data(), (int)st.size(), dev_status, stream);
    } else {
      for (const Int8GemmArgs& a : st) to_cluster(a);
    }
    st.clear();
  };
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    if (!int8_stream_fits(&probs[i], 1)) {
      to_cluster(probs[i]);
      continue;
    }
    st.push_back(probs[i]);
    if (!int8_stream_fits(st.data(), (int)st.size())) {
      st.pop_back();
      flush_stream();
      st.push_back(probs[i]);
    }
  }
  flush_stream();
  if (e == cudaSuccess && !cl.empty()) e = launch_cluster_batch(cl, stream);
  return e;
}

cudaError_t launch_int8_small(const Int8GemmArgs& a, int32_t* dev_status, cudaStream_t stream) {
  return launch_int8_small_group(&a, 1, dev_status, stream);
}

}  // namespace qmm
