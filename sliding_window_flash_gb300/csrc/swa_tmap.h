// swa_tmap.h — host-side construction of TMA tensor maps for [BH, N, D] bf16 tensors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

namespace swa {

// cuTensorMapEncodeTiled, resolved once through the runtime so the library needs no -lcuda.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

// Tensor map over a contiguous bf16 (or, with f16, fp16) tensor viewed as [bh][rows][cols] (cols
// innermost), loaded in boxes of `box_rows` x 64 columns (128 bytes) with 128-byte swizzle.  Rows
// beyond `rows` and columns beyond `cols` read as zero, so a tile never reads into the next head.
// Returns false if the driver rejects the map.
inline bool make_tmap_3d(CUtensorMap* map, const void* base, uint64_t bh, uint64_t rows,
                         uint64_t cols, uint32_t box_rows, bool f16) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, bh};
  cuuint64_t strides[2] = {cols * 2ull, rows * cols * 2ull};  // bytes, dims 1 and 2
  cuuint32_t box[3] = {64u, box_rows, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUtensorMapDataType type =
      f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, type, 3, const_cast<void*>(base), dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace swa
