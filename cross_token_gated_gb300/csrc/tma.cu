// TMA tensor-map creation.
#include <mutex>

#include "tg_tma.h"

namespace tg {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encoder() {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

CUtensorMapSwizzle swizzle_for(uint32_t inner_bytes) {
  if (inner_bytes == 128) return CU_TENSOR_MAP_SWIZZLE_128B;
  if (inner_bytes == 64) return CU_TENSOR_MAP_SWIZZLE_64B;
  if (inner_bytes == 32) return CU_TENSOR_MAP_SWIZZLE_32B;
  return CU_TENSOR_MAP_SWIZZLE_NONE;
}

cudaError_t encode(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box[0] * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch_elems,
                         uint32_t box_rows, uint32_t box_cols) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  return encode(map, base, 2, dims, strides, box);
}

cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, uint64_t batch, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols) {
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  return encode(map, base, 3, dims, strides, box);
}

cudaError_t make_tmap_4d_heads(CUtensorMap* map, const void* base, uint64_t batch, uint64_t rows, uint64_t heads,
                               uint64_t head_cols, uint64_t head_pitch, uint32_t box_rows, uint32_t box_cols) {
  cuuint64_t dims[4] = {head_cols, heads, rows, batch};
  cuuint64_t strides[3] = {head_pitch * 2, heads * head_pitch * 2, rows * heads * head_pitch * 2};
  cuuint32_t box[4] = {box_cols, 1, box_rows, 1};
  return encode(map, base, 4, dims, strides, box);
}

}  // namespace tg
