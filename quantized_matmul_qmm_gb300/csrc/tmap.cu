// TMA descriptor construction on the host.  The driver's cuTensorMapEncodeTiled
// is reached through the runtime's entry-point query (cached once per process),
// so the library does not link libcuda and loads on machines without a driver.
#include <cuda.h>
#include <mutex>

#include "qmm_internal.h"

namespace qmm {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_once;
EncodeTiledFn g_encode = nullptr;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, bool is_bf16_or_f16, void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return false;
  (void)is_bf16_or_f16;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_q4_tiles(CUtensorMap* map, const void* tiles, uint64_t tile_cols, uint64_t tile_rows,
                        uint32_t box_rows) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return false;
  // A tile is 40 rows of 128 bytes: 32 code rows, then 8 rows of (scale, min)
  // pairs.  Tiles are [tile row][tile column]; a box spans 4 tile rows of one
  // tile column, so that one TMA fetches a 128-row unit's stage.
  const cuuint64_t dims[4] = {128, 40, tile_cols, tile_rows};
  const cuuint64_t strides[3] = {128, (cuuint64_t)kTileBytes, (cuuint64_t)kTileBytes * tile_cols};
  const cuuint32_t box[4] = {128, box_rows, 1, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(tiles), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_kblocks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_stride, uint64_t kblocks,
                       uint32_t box_rows, uint32_t box_kblocks) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return false;
  // Bytes of a row-major [rows][row_stride] matrix seen as {64 bytes, rows,
  // k-blocks}: the k-block dimension (stride 64) is outermost, so a box lands
  // in shared memory as [k-block][row][64 bytes].
  const cuuint64_t dims[3] = {64, rows, kblocks};
  const cuuint64_t strides[2] = {row_stride, 64};
  const cuuint32_t box[3] = {64, box_rows, box_kblocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_kblocks128_sw(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_stride,
                             uint64_t kblocks, uint32_t box_rows, uint32_t box_kblocks) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return false;
  // Bytes of a row-major [rows][row_stride] matrix seen as {128 bytes, rows,
  // k-blocks} (k-block stride 128 outermost): a box lands as [k-block][row]
  // [128 bytes] with the 128-byte swizzle (16-byte unit u of line l at
  // u ^ (l & 7)).
  const cuuint64_t dims[3] = {128, rows, kblocks};
  const cuuint64_t strides[2] = {row_stride, 128};
  const cuuint32_t box[3] = {128, box_rows, box_kblocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace qmm
