// tmap.h -- host-side construction of TMA tensor maps for BHSD tensors.
//
// A [BH, S, 128] tensor of 16-bit elements is described as a 3-D tensor map
// (innermost = head dim) with 128-byte swizzle and a box of 64 x rows x 1, so
// one box fills exactly one 128B-swizzled tile of `rows` rows.  Rows past S
// read as zero on loads, per head.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mab {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Returns nullptr when the driver entry point cannot be found.
inline EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// rows_box in [1, 256]; base must be 16-byte aligned.
inline bool make_bhsd_map(CUtensorMap* m, const void* base, bool bf16, int64_t BH, int64_t S,
                          uint32_t rows_box) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)S * 128 * 2};
  cuuint32_t box[3] = {64, rows_box, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Token-major [T, H, 128] tensor (the packed variable-length layout) as a
// 3-D tensor map (head dim, head, token) with a box of 64 x 1 x rows: one box
// is `rows` consecutive tokens of one head, laid out in shared memory exactly
// like a box of the BHSD map.  Tokens past T read as zero.
inline bool make_thd_map(CUtensorMap* m, const void* base, bool bf16, int64_t T, int64_t H,
                         uint32_t rows_box) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  cuuint32_t box[3] = {64, 1, rows_box};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mab
