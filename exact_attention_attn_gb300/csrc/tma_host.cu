// Host-side TMA tensor-map encoding shared by the tensor-core kernels.
#include <cuda.h>

#include "attn_internal.h"

namespace attn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// does not link libcuda directly.
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    cudaDriverEntryPointQueryResult q;
    void *ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

}  // namespace

bool make_tile_map(CUtensorMap *m, const void *base, int cols, int rows, int planes) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * rows * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_block_map(CUtensorMap *m, const void *base, int cols, int rows, int planes, int box_rows) {
  return make_chunk_map(m, base, cols, rows, planes, box_rows, cols / 64);
}

bool make_chunk_map(CUtensorMap *m, const void *base, int cols, int rows, int planes, int box_rows, int box_chunks) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || cols % 64 != 0 || box_rows < 1 || box_rows > 256) return false;
  const int nchunks = cols / 64;
  if (nchunks > 256 || box_chunks < 1 || box_chunks > 256) return false;
  // dims: 64 elements of a chunk, rows, chunks, planes; the chunk stride (128
  // bytes) is smaller than the row stride, which the tensor map allows
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)nchunks, (cuuint64_t)planes};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 2, 128, (cuuint64_t)cols * rows * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_u8_map(CUtensorMap *m, const void *base, int inner, int rows, int planes) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || inner < 128 || inner % 16 != 0 || rows < 1 || planes < 1) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * rows};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn
