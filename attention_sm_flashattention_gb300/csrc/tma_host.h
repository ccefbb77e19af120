// Host-side TMA tensor-map encoding (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// `mats` row-major matrices [rows x cols] of `elem_bytes`-byte elements,
// stored back to back (contiguous [mats, rows, cols]), tiled in boxes of
// box_cols x box_rows x 1.  A box that runs past `rows` is zero-filled on
// load and clipped on store inside its own matrix.
inline bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                         uint64_t mats, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                         bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, mats};
  cuuint64_t strides[2] = {cols * static_cast<uint64_t>(elem_bytes), rows * cols * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Paged cache [pages, page_rows, heads, cols] of `elem_bytes`-byte elements,
// as a 4-D tensor (cols, heads, page_rows, pages); boxes of box_cols x 1
// head x page_rows rows x 1 page, so one box is one head's rows of one page
// and lands in shared memory as a [page_rows x box_cols] tile.
inline bool make_tmap_paged(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                            uint64_t pages, uint64_t page_rows, uint64_t heads, uint64_t cols, uint32_t box_cols,
                            bool swizzle128) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const uint64_t eb = static_cast<uint64_t>(elem_bytes);
  cuuint64_t dims[4] = {cols, heads, page_rows, pages};
  cuuint64_t strides[3] = {cols * eb, heads * cols * eb, page_rows * heads * cols * eb};
  cuuint32_t box[4] = {box_cols, 1, static_cast<cuuint32_t>(page_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
