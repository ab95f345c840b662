// tma_host.cuh -- host helpers shared by the tensor-core kernels: tensor-map
// encoding through the driver entry point (no link against libcuda) and the
// once-per-device shared-memory attribute.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

namespace moe {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Every map moves 16-bit units: bf16 values, or pairs of fp8 bytes (a map
// of `elem` = 1 covers cols / 2 units per row; cols must be even).  The box
// is 64 units = 128 bytes of a row wide; x coordinates count 16-bit units.
inline CUtensorMapDataType map_type(int elem) {
  return elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// 2-D map over a row-major [rows][cols] matrix of `elem`-byte elements, box
// 128 bytes of columns x box_rows, 128-byte swizzle.
inline bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, int elem = 2) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols * (uint64_t)elem / 2, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)elem};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, map_type(elem), 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over [n_mat][rows][cols], box 128 bytes of columns x box_rows x 1.
inline bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t n_mat, uint64_t rows,
                      uint64_t cols, uint32_t box_rows, int elem = 2) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols * (uint64_t)elem / 2, rows, n_mat};
  cuuint64_t strides[2] = {cols * (uint64_t)elem, rows * cols * (uint64_t)elem};
  cuuint32_t box[3] = {64u, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, map_type(elem), 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over [n_mat][rows][cols] bytes (e4m3 codes) for tiles of box_bytes
// (64 or 128) of a row x box_rows x 1, not swizzled (the tile is expanded on
// chip); the bytes move as 16-bit units.
inline bool encode_3d_codes(CUtensorMap* m, const void* ptr, uint64_t n_mat, uint64_t rows,
                            uint64_t cols, uint32_t box_rows, uint32_t box_bytes = 64) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols / 2, rows, n_mat};
  cuuint64_t strides[2] = {cols, rows * cols};
  cuuint32_t box[3] = {box_bytes / 2, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise the dynamic shared-memory limit of a kernel once per device.
template <typename K>
inline cudaError_t smem_attr_once(K kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

}  // namespace moe
