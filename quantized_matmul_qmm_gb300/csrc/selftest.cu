// Self-test of the device error path shared by the pipelined kernels.
//
// Every pipeline wait in the library is an mbarrier wait bounded in time
// (umma::mbar_wait).  When one gives up it raises its CTA's abort flag and
// writes QMM_ERR_TIMEOUT to the caller's status word; every other wait of the
// CTA then returns false, the roles leave their loops, and the kernel frees
// its tensor memory and exits.  A healthy run never takes that path, so this
// kernel takes it on purpose: one warp waits, with a short limit, on a barrier
// that nothing arrives on, while another waits (with the library's normal
// limit) on a second barrier that nothing arrives on either and must leave as
// soon as the abort flag is up.  A third warp holds a tensor-memory
// allocation across the abort and frees it, as the kernels do.
#include "qmm_internal.h"
#include "umma.cuh"

namespace qmm {
namespace {

using namespace umma;

constexpr uint64_t kSelftestMaxLimitNs = 100000000ull;   // 100 ms

// out[0]: 1 if the short wait completed (it must not), out[1]: 1 if the
// long wait completed (it must not), out[2]: ns the short wait took,
// out[3]: ns from the abort to the long wait's return.
__global__ void __launch_bounds__(96, 1) wait_timeout_selftest_kernel(uint64_t limit_ns, int32_t* dev_status,
                                                                     int64_t* out) {
  __shared__ uint64_t never[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ unsigned long long t_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&never[0], 1);
    mbar_init(&never[1], 1);
    abort_flag = 0;
    t_abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0 && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool done = mbar_wait(&never[0], 0, &abort_flag, dev_status, limit_ns);
    const uint64_t t1 = globaltimer_ns();
    t_abort = t1;
    out[0] = done ? 1 : 0;
    out[2] = (int64_t)(t1 - t0);
  } else if (warp == 1 && lane == 0) {
    const bool done = mbar_wait(&never[1], 0, &abort_flag, dev_status);
    const uint64_t t1 = globaltimer_ns();
    out[1] = done ? 1 : 0;
    out[3] = (int64_t)t1;   // t_abort is read after the barrier below
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 32) out[3] -= (int64_t)t_abort;
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, 32);
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* dev_status, int64_t* out,
                                         cudaStream_t stream) {
  if (limit_ns > kSelftestMaxLimitNs) return cudaErrorInvalidValue;
  wait_timeout_selftest_kernel<<<1, 96, 0, stream>>>(limit_ns, dev_status, out);
  return cudaGetLastError();
}

}  // namespace qmm
