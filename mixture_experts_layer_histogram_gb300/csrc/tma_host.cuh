// Host-side TMA tensor-map helpers (cuTensorMapEncodeTiled through the runtime's driver entry
// point, so libmoe links against the runtime only). Shared by the GEMM and router kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {
namespace tc {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D bf16 row-major [rows, cols] with box = box_cols x box_rows and the given swizzle. Elements of a
// box outside the tensor read as zero; stores drop them.
inline bool encode_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                       uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// operand loads: 64 columns (128 B, the swizzle span) x box_rows rows, 128-byte swizzle
inline bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return encode_map(m, base, rows, cols, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}
// epilogue stores: 32 x 32 blocks, 64-byte swizzle (matches the epilogue's shared-memory layout)
inline bool make_store_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  return encode_map(m, base, rows, cols, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// epilogue stores of 16-column blocks: 16 x 32 boxes (32-byte rows), 32-byte swizzle
inline bool make_store_map16(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  return encode_map(m, base, rows, cols, 16, 32, CU_TENSOR_MAP_SWIZZLE_32B);
}
// The gate/up weights Wgu [E, 2f, d] as a 5D view (k, row r, gate/up u, group g, expert e) ->
// Wgu[e][u f + 8 g + r][k]. One box (64 k x 8 rows x 2 x 8 groups) lands in shared memory as 128
// rows in which each group's 8 gate rows are followed by the same group's 8 up rows.
inline bool make_gateup_map(CUtensorMap *m, const void *wgu, uint64_t E, uint64_t f, uint64_t d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[5] = {d, 8, 2, f / 8, E};
  cuuint64_t strides[4] = {d * 2, f * d * 2, 8 * d * 2, 2 * f * d * 2};
  cuuint32_t box[5] = {64, 8, 2, 8, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(wgu), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace moe
