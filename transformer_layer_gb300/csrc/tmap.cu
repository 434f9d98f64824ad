// Host-side TMA tensor maps of the weight matrices (created with the layer).
// A map lets one cp.async.bulk.tensor instruction fetch a whole GEMV chunk
// (16 weight rows x up to 2 KB), swizzled for conflict-free fragment loads,
// where row-by-row bulk copies would need 16 instructions: on GB300 the
// per-instruction cost of small bulk copies, not HBM, otherwise caps a CTA's
// weight stream near 4 TB/s.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ring_layout.h"

namespace ds {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

bool encode_weight_map(void* map128, const void* base, int rows, size_t row_bytes, int chunk_row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr || row_bytes % kSwizzleBytes != 0 || chunk_row_bytes % kSwizzleBytes != 0 ||
      chunk_row_bytes / kSwizzleBytes > 256)
    return false;
  // The matrix as 16-bit elements (fp16 / bf16 weights, or int8 codes in
  // pairs), indexed (element within a 128-byte segment, row, segment): the
  // box's traversal order then lays a chunk out as [segment][row][128 bytes].
  const cuuint64_t dims[3] = {(cuuint64_t)(kSwizzleBytes / 2), (cuuint64_t)rows,
                              (cuuint64_t)(row_bytes / kSwizzleBytes)};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)kSwizzleBytes};
  const cuuint32_t box[3] = {(cuuint32_t)(kSwizzleBytes / 2), 16u, (cuuint32_t)(chunk_row_bytes / kSwizzleBytes)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(static_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_scale_map(void* map128, const void* base, int rows, int groups, int box_groups, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr || (groups * 2) % 16 != 0 || (box_groups * 2) % 16 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)groups, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)groups * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_groups, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(static_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tile_map(void* map128, const void* base, int rows, int cols, int box_rows, int kc) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr || rows < 1 || cols % 64 != 0 || kc % 64 != 0 || box_rows < 8 || box_rows > 256 ||
      (reinterpret_cast<uintptr_t>(base) & 15u) != 0)
    return false;
  // [rows][cols] 16-bit elements as (element within a 128-byte atom, row,
  // atom): a box of (64, box_rows, kc / 64) lands as [atom][row][128 bytes],
  // 128-byte swizzled -- the K-major operand layout of tcgen05.mma.  Rows past
  // the end read as zero.
  const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)(kc / 64)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(static_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ds
