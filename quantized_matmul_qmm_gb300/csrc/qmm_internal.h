// Host-side declarations shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "qmm.h"
#include "qmm_device.cuh"

namespace qmm {

constexpr int64_t kTileRows = 32;
constexpr int64_t kTileCols = 256;
constexpr int64_t kTileBytes = 5120;

inline int64_t padded_k(int64_t K) { return (K + 63) / 64 * 64; }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch with programmatic stream serialization: the grid may start while the
// previous grid in the stream finishes.  The kernel must execute
// griddepcontrol.wait before touching anything that grid could have written,
// and it releases its own dependents with griddepcontrol.launch_dependents.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- TMA descriptors (tmap.cu): 2-byte elements, 128-byte swizzle, box
// box_inner x box_rows (box_inner * 2 == 128 bytes) ----
bool make_tmap_2d(CUtensorMap* map, bool is_bf16_or_f16, void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);

// q4 tiles as a 4-D byte tensor {128 bytes, 40 rows, tile_cols, tile_rows},
// 128-byte swizzle, box {128, box_rows, 1, 4}: rows 0..31 of a tile are its
// codes, rows 32..39 its (scale, min) pairs; one box covers 4 tile rows.
bool make_tmap_q4_tiles(CUtensorMap* map, const void* tiles, uint64_t tile_cols, uint64_t tile_rows,
                        uint32_t box_rows);

// A row-major byte matrix [rows][row_stride] as {64 bytes, rows, k-blocks}
// (k-block stride 64 bytes), no swizzle, box {64, box_rows, box_kblocks}: a
// box lands as [k-block][row][64 bytes]; rows and k-blocks past the extents
// read as zero.
bool make_tmap_kblocks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_stride, uint64_t kblocks,
                       uint32_t box_rows, uint32_t box_kblocks);
// The same with 128-byte k-blocks and the 128-byte swizzle (row_stride a
// multiple of 128, so no k-block reaches past its row).
bool make_tmap_kblocks128_sw(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_stride,
                             uint64_t kblocks, uint32_t box_rows, uint32_t box_kblocks);

// ---- packs (pack.cu) ----
cudaError_t launch_pack_b_int8(const void* B, qmm_dtype b_type, int64_t K, int64_t N, int64_t ldb,
                               int8_t* packed, int64_t Kp, float* col_scale, int32_t* col_sum,
                               cudaStream_t stream);
cudaError_t launch_pack_q4(const float* W, int64_t N, int64_t K, int64_t ldw, uint8_t* tiles,
                           cudaStream_t stream);

// ---- int8 GEMM ----
struct Int8GemmArgs {
  const int8_t* A;         // [M][lda] bytes (uint8 or int8 codes)
  bool a_u8;
  int M, K, N;
  int64_t lda;
  const int8_t* B;         // packed [N][Kp]
  int64_t Kp;
  bool need_rowsum;        // zB' != 0
  Int8Epi epi;
};
// legacy integer MMA route (int8_mma.cu)
cudaError_t launch_int8_gemm_mma(const Int8GemmArgs& a, cudaStream_t stream);
// small-M route (int8_small.cu): clusters of 8 CTAs, f16 MMA on exact integer codes
bool int8_small_eligible(int64_t M, int64_t K, int64_t N);
cudaError_t launch_int8_small(const Int8GemmArgs& a, int32_t* dev_status, cudaStream_t stream);
// several small-M problems, one launch per 16 (each must be int8_small_eligible)
cudaError_t launch_int8_small_group(const Int8GemmArgs* probs, int n, int32_t* dev_status, cudaStream_t stream);
// the streaming form (int8_stream.cu): one CTA per SM, no clusters; for up to
// 16 problems whose rows fit its shared memory together
bool int8_stream_fits(const Int8GemmArgs* probs, int n);
int64_t int8_stream_items(const Int8GemmArgs* probs, int n);   // 16-column items
cudaError_t launch_int8_stream_group(const Int8GemmArgs* probs, int n, int32_t* dev_status, cudaStream_t stream);
// tcgen05 route (int8_umma.cu)
bool int8_umma_eligible(int64_t M, int64_t K, int64_t N);
size_t int8_umma_workspace_bytes(int64_t M, int64_t K, int64_t N, bool b16_given = false);
// b16: the weights as f16 [N][Kp] from launch_widen_b_int8, or null (widened on every call)
cudaError_t launch_int8_gemm_umma(const Int8GemmArgs& a, void* workspace, int32_t* dev_status,
                                  cudaStream_t stream, const __half* b16 = nullptr);
// packed B' [N][Kp] widened once to f16 [N][Kp] (exact)
cudaError_t launch_widen_b_int8(const int8_t* packed, int K, int N, __half* b16, int32_t* dev_status,
                                cudaStream_t stream);
// activation quantisation (quant_act.cu); the per-tensor path uses 4 bytes of workspace
cudaError_t launch_quantize_act(const void* X, bool x_bf16, int M, int K, int64_t ldx, bool per_row, int8_t* A,
                                int64_t lda, float* s_x, void* workspace, cudaStream_t stream);

// ---- W8A16 (w8.cu, and the pair kernel in int8_umma.cu for M > kW8GemvMaxM) ----
constexpr int64_t kW8MaxK = 65536;
constexpr int64_t kW8GemvMaxM = 16;
int64_t w8_padded_k(int64_t K);   // codes per row: K rounded up to 64
int64_t w8_blocks(int64_t K);     // scales per row: ceil(K / 1024)
cudaError_t launch_pack_w8(const float* W, int N, int K, int64_t ldw, int8_t* codes, float* scales,
                           cudaStream_t stream);
cudaError_t launch_w8_gemv(const int8_t* codes, const float* scales, int N, int K, const __nv_bfloat16* X,
                           int64_t ldx, int M, float* Y, int64_t ldy, int32_t* dev_status, cudaStream_t stream);
size_t w8_umma_workspace_bytes(int64_t K, int64_t N);
cudaError_t launch_w8_gemm_umma(const int8_t* codes, const float* scales, int N, int K,
                                const __nv_bfloat16* X, int64_t ldx, int M, float* Y, int64_t ldy,
                                void* workspace, int32_t* dev_status, cudaStream_t stream);
// The pair GEMM alone, on 16-bit weights W16 [N][padded_k(K)] that an earlier
// launch in the stream wrote; scales [N][nb] multiply each kPairChunkK-column
// chunk of the accumulator.  bf16 weights take bf16 activations X; f16
// weights take f16 activation rows X (act16.cu) whose inverse scales x_up
// multiply each output row.
constexpr int kPairChunkK = 1024;
cudaError_t launch_w16_gemm_umma(const void* W16, bool f16, const float* scales, int nb, int N, int K,
                                 const void* X, int64_t ldx, const float* x_up, int M, float* Y, int64_t ldy,
                                 int32_t* dev_status, cudaStream_t stream);

// ---- more weight formats (formats.cu): Q4_K -> q4_1 repack, Q8 tiles ----
constexpr int kQ8TileBytes = 8704;   // 8192 code bytes + 256 bf16 scales
constexpr int kQ8CodeBytes = 8192;
constexpr int64_t kQ8GemvMaxM = 16;
constexpr int64_t kQ8MaxK = 65536;
cudaError_t launch_repack_q4k(const uint8_t* src, int64_t row_bytes, int N, int K, uint8_t* tiles,
                              cudaStream_t stream);
cudaError_t launch_pack_q8(const float* W, int64_t ldw, int N, int K, int layout, uint8_t* tiles,
                           cudaStream_t stream);
size_t q8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);   // the M > kQ8GemvMaxM route
cudaError_t launch_q8_gemm(const uint8_t* tiles, int layout, int N, int K, const __nv_bfloat16* X, int64_t ldx,
                           int M, float* Y, int64_t ldy, void* workspace, int32_t* dev_status, cudaStream_t stream);

// ---- f16 activation operands (act16.cu) ----
// Each bf16 row scaled by a power of two into [2^14, 2^15) and rounded to f16
// (exact), with the inverse factor kept per row: f16 [rows][K], then fp32
// [rows], each padded to 256 bytes.
size_t act_f16_bytes(int64_t rows, int64_t K);
inline size_t act_f16_scale_offset(int64_t rows, int64_t K) { return ((size_t)rows * K * 2 + 255) / 256 * 256; }
cudaError_t launch_act_to_f16(const __nv_bfloat16* X, int64_t ldx, int rows, int K, void* out, cudaStream_t stream);

// ---- q4 kernels (q4_mma.cu, q4_umma.cu) ----
struct Q4DenseArgs {
  const uint8_t* tiles;
  int N, K, M;
  const __nv_bfloat16* X;
  int64_t ldx;
  float* Y;
  int64_t ldy;
  void* act16;   // tensor-core route: act_f16_bytes(M, K) of workspace
};
cudaError_t launch_q4_gemv(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_q4_gemv1(const Q4DenseArgs& a, int sms, int32_t* dev_status, cudaStream_t stream);
// grouped M = 1 GEMV (q4_gemv.cu)
struct GemvGroupProblem {
  const uint8_t* tiles;
  const __nv_bfloat16* X;
  float* Y;
  int N, K;
};
constexpr int kMaxGroupProblems = 32;   // problems per grouped launch
constexpr int kMaxGroupRows = 6144;     // tile rows per grouped launch
constexpr int kMaxGroupK = 16384;       // larger K runs the single-problem kernel
cudaError_t launch_q4_gemv_group(const GemvGroupProblem* probs, int n, int sms, int32_t* dev_status,
                                 cudaStream_t stream);
bool q4_umma_eligible(int64_t M, int64_t N, int64_t K);
cudaError_t launch_q4_gemm_umma(const Q4DenseArgs& a, int32_t* dev_status, cudaStream_t stream);

struct Q4MoEArgs {
  const uint8_t* tiles;
  const uint8_t* tiles2;   // the gate/up pair: a second weight set read with the same routing, or null
  float* Y2;               // its output
  int n_expert, N, K;
  const __nv_bfloat16* X;
  int64_t ldx_token, ldx_slot;
  const int32_t* ids;
  int64_t ld_ids;
  int n_used, T;
  float* Y;
  int64_t ldy_token, ldy_slot;
  int32_t* offsets;   // workspace: [n_expert + 1]
  int32_t* pairs;     // workspace: [T * n_used]
  float* xup;         // workspace: [T * n_used] inverse activation-row scales, by grouped rank
  __half* xperm;      // workspace: [T * n_used][K] packed f16 activations, or null (gather mode)
  int32_t* dev_status;
};
constexpr int64_t kMaxExperts = 4096;
// routing tables and row scales only (enough for the gather path)
size_t q4_moe_table_bytes(int64_t n_expert, int64_t n_used, int64_t T);
// tables + packed activations (the full workspace)
size_t q4_moe_workspace_bytes(int64_t n_expert, int64_t n_used, int64_t T, int64_t K);
cudaError_t launch_q4_moe(const Q4MoEArgs& a, cudaStream_t stream);

// ---- load-only HBM probe (probe.cu): mode 0 per-thread loads, 1 bulk copies ----
cudaError_t launch_probe_hbm_read(const void* buf, size_t bytes, int mode, uint32_t* sink, int32_t* dev_status,
                                  cudaStream_t stream);

// ---- self-test of the bounded-wait error path (selftest.cu) ----
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* dev_status, int64_t* out,
                                         cudaStream_t stream);

}  // namespace qmm
