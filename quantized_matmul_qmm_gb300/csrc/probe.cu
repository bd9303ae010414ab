// Load-only HBM probe: the read bandwidth a kernel that does nothing but
// stream a buffer can reach on this GPU.  It is the roofline the decode GEMVs
// are measured against besides the copy bandwidth ("Zaya 8B Q4NX on the AMD
// NPU", round 25q: a load-only kernel over a rotating ring of buffers set the
// ceiling that the decode GEMV was then compared with).
//
// Two ways of reading, the two the GEMVs use:
//   mode 0  per-thread 16-byte loads, eight in flight per thread, a grid of
//           several blocks per SM;
//   mode 1  bulk copies (cp.async.bulk) of 32 KB chunks into a six-slot
//           shared-memory ring, one block per SM, one issuing thread.
// The loaded data is folded into one word so the loads cannot be dropped; it
// is written out only if it equals a value the caller cannot produce by
// chance, which keeps the probe free of stores.
#include <algorithm>

#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr int kLdThreads = 512;
constexpr int kLdUnroll = 8;
constexpr uint32_t kChunk = 32768;
constexpr int kSlots = 6;
constexpr uint32_t kMagic = 0x9E3779B9u;

__global__ void __launch_bounds__(kLdThreads) probe_ld_kernel(const uint4* __restrict__ buf, int64_t n16,
                                                              uint32_t* sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * kLdThreads * kLdUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kLdThreads * kLdUnroll + threadIdx.x; base < n16; base += stride) {
    uint4 v[kLdUnroll];
#pragma unroll
    for (int u = 0; u < kLdUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kLdThreads;
      v[u] = i < n16 ? ldg128_stream(buf + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLdUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  if (acc == kMagic) sink[0] = acc;
}

__global__ void __launch_bounds__(32, 1) probe_bulk_kernel(const uint8_t* __restrict__ buf, int64_t nchunks,
                                                           uint32_t* sink, int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kSlots];
  __shared__ volatile int abort_flag;
  uint8_t* ring = smem_align(smem_raw, 128);
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kSlots; ++s) mbar_init(&full[s], 1);
  abort_flag = 0;
  fence_mbar_init();
  int64_t issued = 0;
  uint32_t acc = 0;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++issued) {
    const int s = (int)(issued % kSlots);
    if (issued >= kSlots) {
      // the copy that used this slot before has landed
      if (!mbar_wait(&full[s], (uint32_t)(((issued / kSlots) - 1) & 1), &abort_flag, dev_status)) return;
      acc ^= reinterpret_cast<const uint32_t*>(ring + (size_t)s * kChunk)[0];
    }
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&full[s], kChunk);
    bulk_g2s(smem_u32(ring + (size_t)s * kChunk), buf + c * (int64_t)kChunk, kChunk, &full[s]);
  }
  // drain: every copy in flight lands before the block exits
  for (int64_t i = std::max<int64_t>(0, issued - kSlots); i < issued; ++i) {
    const int s = (int)(i % kSlots);
    if (!mbar_wait(&full[s], (uint32_t)((i / kSlots) & 1), &abort_flag, dev_status)) return;
    acc ^= reinterpret_cast<const uint32_t*>(ring + (size_t)s * kChunk)[0];
  }
  if (acc == kMagic) sink[0] = acc;
}

}  // namespace

cudaError_t launch_probe_hbm_read(const void* buf, size_t bytes, int mode, uint32_t* sink, int32_t* dev_status,
                                  cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (mode == 0) {
    const int64_t n16 = (int64_t)(bytes / 16);
    probe_ld_kernel<<<4 * sms, kLdThreads, 0, stream>>>(static_cast<const uint4*>(buf), n16, sink);
    return cudaGetLastError();
  }
  const size_t smem = 128 + (size_t)kSlots * kChunk;
  cudaError_t err = cudaFuncSetAttribute(probe_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  probe_bulk_kernel<<<sms, 32, smem, stream>>>(static_cast<const uint8_t*>(buf), (int64_t)(bytes / kChunk), sink,
                                               dev_status);
  return cudaGetLastError();
}

}  // namespace qmm
