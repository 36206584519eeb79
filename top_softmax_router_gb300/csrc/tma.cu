// TMA tensor-map construction (host side).  The driver entry point is looked
// up through the runtime, so the library loads on machines without a driver.
#include <cudaTypedefs.h>
#include <mutex>

#include "kernels.h"

// L2 promotion of TMA requests (the 256-byte default fetches the neighbouring 128-byte line too).
#ifndef MOE_TMA_L2_PROMOTION
#define MOE_TMA_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

namespace moe {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 128-byte swizzle, out-of-bounds elements read as zero (and are not written by stores).
static bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, MOE_TMA_L2_PROMOTION,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  return encode(m, base, 2, dims, strides, box);
}

bool make_map_2d_strided(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                         uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  return encode(m, base, 2, dims, strides, box);
}

bool make_map_gather(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, 1};
  return encode(m, base, 2, dims, strides, box);
}

bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                 uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[3] = {inner, rows, depth};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  return encode(m, base, 3, dims, strides, box);
}

bool make_map_3d_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                     uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[3] = {inner, rows, depth};
  const cuuint64_t strides[2] = {inner * 4, inner * rows * 4};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  return encode(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

}  // namespace moe
