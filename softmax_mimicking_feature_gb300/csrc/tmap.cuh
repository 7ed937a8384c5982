// Host-side tensor maps: the q, k, v tensors handed to the library (two
// layouts) and the library's own [planes][rows][cols] buffers.
//
// The library takes two layouts of a [B] x [H] x [n] x [cols] tensor
// (cols contiguous):
//   HH_LAYOUT_BHND  [B][H][n][cols]   (heads outermost after the batch)
//   HH_LAYOUT_BNHD  [B][n][H][cols]   (what a fused QKV projection produces)
// Both are 4-D tiled maps with strides increasing outwards: dims
// (cols, n, H, B) for the first and (cols, H, n, B) for the second, boxes of
// box_rows rows of one head, so a loaded tile has the same shared-memory
// layout either way (tma_load_rows in tc_ptx.cuh picks the coordinate order).

#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hh {

typedef CUresult (*TmapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline TmapEncodeFn tmap_encode_fn() {
  static TmapEncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmapEncodeFn>(p);
  }
  return fn;
}

// bf16 map over [planes][rows][cols] (library-owned buffers: weights,
// features, states) with {box_cols, box_rows, 1} boxes.
inline bool make_plane_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                           uint64_t planes, uint32_t box_cols, uint32_t box_rows,
                           CUtensorMapSwizzle swz) {
  TmapEncodeFn enc = tmap_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 map over heads x rows of a [B][H][n][cols] or [B][n][H][cols] tensor;
// boxes of box_cols x box_rows of one head.
inline bool make_rows_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t n, uint64_t H,
                          uint64_t B, uint32_t box_cols, uint32_t box_rows,
                          CUtensorMapSwizzle swz, int seq_major) {
  TmapEncodeFn enc = tmap_encode_fn();
  if (!enc) return false;
  const uint64_t esz = 2;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  dims[0] = cols;
  box[0] = box_cols;
  if (seq_major) {
    dims[1] = H;
    dims[2] = n;
    strides[0] = cols * esz;
    strides[1] = H * cols * esz;
    box[1] = 1;
    box[2] = box_rows;
  } else {
    dims[1] = n;
    dims[2] = H;
    strides[0] = cols * esz;
    strides[1] = n * cols * esz;
    box[1] = box_rows;
    box[2] = 1;
  }
  dims[3] = B;
  strides[2] = n * H * cols * esz;
  box[3] = 1;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace hh
