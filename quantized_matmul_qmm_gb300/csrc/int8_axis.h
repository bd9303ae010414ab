// Host-side declarations of the per-axis zero-point variant of the int8 GEMM
// (int8_axis.cu): the row sums of A' and one elementwise pass over the exact
// product S' that the per-tensor GEMM wrote.
#pragma once

#include "qmm_internal.h"

namespace qmm {

struct Int8AxisArgs {
  const uint8_t* A;
  int64_t lda;
  bool a_u8, b_u8;
  int M, K, N;
  const int32_t* zA;     // [M] in A's domain, or null (all 0)
  const int32_t* zB;     // [N] in B's domain, or null (all 0)
  const int32_t* S;      // S' (int32 [M][N], row stride N) from the per-tensor GEMM
  int32_t* row_sum;      // [M] workspace
  Int8Epi epi;           // bias, scales, output; col_sum
  int32_t* dev_status;
};

cudaError_t launch_int8_axis_zp(const Int8AxisArgs& a, cudaStream_t stream);

}  // namespace qmm
