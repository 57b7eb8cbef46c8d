// Host-side TMA descriptors (CUtensorMap) for the attention kernels.  The
// driver's encoder is reached through the runtime's entry-point query, so the
// library links only against the CUDA runtime.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool tma_available() { return encode_fn() != nullptr; }

bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int64_t row_stride,
                   int box_heads, int box_rows) {
  if (!encode_fn()) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadSize, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadSize * 2, (cuuint64_t)row_stride * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv) {
  if (!encode_fn()) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadSize, (cuuint64_t)hkv, (cuuint64_t)kBlockSize,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadSize * 2, (cuuint64_t)hkv * kHeadSize * 2,
                           (cuuint64_t)hkv * kHeadSize * 2 * kBlockSize};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kBlockSize, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_cache_map_i8(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv) {
  if (!encode_fn()) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadSize, (cuuint64_t)hkv, (cuuint64_t)kBlockSize,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadSize, (cuuint64_t)hkv * kHeadSize,
                           (cuuint64_t)hkv * kHeadSize * kBlockSize};
  cuuint32_t box[4] = {(cuuint32_t)kHeadSize, 1, (cuuint32_t)kBlockSize, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv
