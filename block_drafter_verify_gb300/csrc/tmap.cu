// Host-side TMA descriptors (CUtensorMap) for row-major bf16 and 8-bit
// matrices.
// cuTensorMapEncodeTiled is reached through the runtime's driver entry
// point, so the library needs no link against libcuda.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace dflash {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
}  // namespace

namespace {
bool make_tmap_2d(CUtensorMapDataType type, uint32_t elem_bytes,
                  CUtensorMap* map, const void* base, uint64_t inner,
                  uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  std::call_once(g_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!g_encode || rows == 0 || inner == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * elem_bytes};  // bytes between rows
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return g_encode(map, type, 2,
                  const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner,
                       uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  return make_tmap_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, map, base, inner,
                      rows, box_inner, box_rows);
}

bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner,
                     uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  return make_tmap_2d(CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, map, base, inner,
                      rows, box_inner, box_rows);
}

}  // namespace dflash
