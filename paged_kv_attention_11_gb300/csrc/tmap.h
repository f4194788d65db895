// Host-side TMA descriptor (CUtensorMap) encoding, shared by the launchers.
// cuTensorMapEncodeTiled is fetched through the runtime's driver entry-point
// query, so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

namespace pkv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// K or V pool for the varlen and decode kernels, viewed as {64 columns, 8 rows, D/64
// column chunks, P/8 row groups, num_pages*H_kv}: one box {64, 8, D/64,
// rows/8, 1} is `rows` keys of one page and head, and lands in shared memory
// as [row group][column chunk][8 rows][128 bytes], 128-byte swizzled: every
// 8-row block of a chunk is one swizzle atom, atoms of one chunk sit
// (D/64)*1024 bytes apart and chunks 1024 bytes apart, uniformly across the
// boxes of a tile.
// box_cols: the columns one box covers (a multiple of 64, default all D):
// a box then lands as [row group][box_cols/64 chunks][8 rows][128 bytes].
// heads: consecutive kv heads of the page in one box (the outermost box
// dimension): the box lands as [head][row group][chunk][8 rows][128 bytes].
inline bool encode_pool_map_groups(CUtensorMap* m, const void* base, int D, int P,
                                   int64_t num_pages, int H_kv, int rows, int box_cols = 0,
                                   int heads = 1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (box_cols <= 0) box_cols = D;
  cuuint64_t dims[5] = {64, 8, (cuuint64_t)(D / 64), (cuuint64_t)(P / 8),
                        (cuuint64_t)(num_pages * H_kv)};
  cuuint64_t strides[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)8 * D * 2, (cuuint64_t)P * D * 2};
  cuuint32_t box[5] = {64, 8, (cuuint32_t)(box_cols / 64), (cuuint32_t)(rows / 8),
                       (cuuint32_t)heads};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [total_q, H_q, D] viewed as {D, G, H_kv, total_q}; box = 64 x G x 1 x (128/G)
// so one box holds 128 (position, head) rows of one kv group.
inline bool encode_q_map(CUtensorMap* m, const void* base, int D, int G, int H_kv, int total_q) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)H_kv, (cuuint64_t)total_q};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                           (cuuint64_t)H_kv * G * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv
