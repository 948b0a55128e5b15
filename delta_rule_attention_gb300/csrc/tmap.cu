// Host-side tensor-map encoding (see tmap.cuh).
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tmap.cuh"

namespace falcon {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_resolve_once;

void resolve_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult status;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &status) == cudaSuccess &&
      status == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

bool encode_rows_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint64_t mats, uint32_t box_cols, uint32_t box_rows) {
  std::call_once(g_resolve_once, resolve_encoder);
  if (g_encode == nullptr || rows == 0 || mats == 0) return false;
  const cuuint64_t dims[3] = {cols, rows, mats};
  const cuuint64_t strides[2] = {cols * 2, cols * 2 * rows};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace falcon
