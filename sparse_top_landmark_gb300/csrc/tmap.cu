// Host helper: TMA tensor maps for [batch, rows, 64] bf16 arrays (one 128-byte
// row per token), loaded as boxes of `box_rows` rows with 128-byte swizzle.
// The driver's encoder is looked up through the runtime, so the library does
// not link libcuda directly.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace mita {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
}  // namespace

namespace {
void init_encoder() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
}
}  // namespace

bool make_tmap_rows64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t batches,
                      uint32_t box_rows, bool fp16) {
  std::call_once(g_once, init_encoder);
  if (!g_encode || box_rows < 1 || box_rows > 256) return false;
  cuuint64_t dims[3] = {64, rows, batches};
  cuuint64_t strides[2] = {128, 128 * rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, 64] bf16 rows fetched four at a time with tile::gather4 (box one row high).
bool make_tmap_gather64(CUtensorMap* map, const void* base, uint64_t rows) {
  std::call_once(g_once, init_encoder);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mita
