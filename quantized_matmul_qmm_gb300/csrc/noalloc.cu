// MUL_MAT_ID without a caller-provided workspace.
//
// Some callers cannot allocate device memory.  One example is a plugin whose
// host framework owns every device buffer and hands it only inputs and
// outputs.  Another is a latency-critical path that cannot afford a
// cudaMalloc, which may synchronise the device.  For those callers,
// qmm_q4_gemm_id_noalloc keeps the routing tables of the expert grouping
// (per-expert offsets, the grouped (token, slot) list and the activation-row
// scales) in a fixed array in the library's own device memory.  Every GPU
// that loads the library holds that array until the process exits.  The rest
// of the call is qmm_q4_gemm_id, unchanged: when the packed activation rows
// also fit in the array (small calls), it packs them there; otherwise the
// grouped kernel gathers the rows itself.
#include <mutex>

#include "qmm_internal.h"

using namespace qmm;

namespace {

constexpr int64_t kNoAllocMaxExperts = 1024;
constexpr int64_t kNoAllocMaxPairs = 65536;   // T * n_used
constexpr size_t kOffsetsBytes = ((kNoAllocMaxExperts + 1) * 4 + 255) / 256 * 256;
// offsets, pair ids, row scales: 528,640 bytes
constexpr size_t kScratchBytes = kOffsetsBytes + 2 * (size_t)kNoAllocMaxPairs * 4;
static_assert(kScratchBytes % 256 == 0, "pair table padding");

// The routing scratch.  Host code must not pass this symbol to a kernel: on
// the host it names a stand-in, not device memory.  The device address comes
// from cudaGetSymbolAddress, fetched once per device below.
static __device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_moe_scratch on the current device.  It is looked up on
// the first call per device and cached.
qmm_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess || p == nullptr) return QMM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QMM_OK;
}

}  // namespace

extern "C" qmm_status qmm_q4_gemm_id_noalloc(const void* tiles, int64_t n_expert, int64_t N,
                                             int64_t K, const void* X, int64_t ldx_token,
                                             int64_t ldx_slot, const int32_t* ids, int64_t ld_ids,
                                             int64_t n_used, int64_t T, float* Y,
                                             int64_t ldy_token, int64_t ldy_slot,
                                             int32_t* dev_status, cudaStream_t stream) {
  if (n_expert < 1 || n_used < 1 || T < 1) return QMM_ERR_INVALID_ARG;
  if (n_expert > kNoAllocMaxExperts || T * n_used > kNoAllocMaxPairs) return QMM_ERR_WORKSPACE;
  void* scratch = nullptr;
  const qmm_status st = scratch_address(&scratch);
  if (st != QMM_OK) return st;
  // The router and the packing grid rewrite every offset, grouped pair, row
  // scale and packed row that later grids read, so nothing in the scratch has
  // to start at zero.
  return qmm_q4_gemm_id(tiles, n_expert, N, K, X, ldx_token, ldx_slot, ids, ld_ids, n_used, T, Y,
                        ldy_token, ldy_slot, scratch, kScratchBytes, dev_status, stream);
}
