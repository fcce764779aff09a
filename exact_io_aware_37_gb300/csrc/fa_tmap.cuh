// Host helpers for the tensor-core kernels: TMA tensor maps over the
// attention tensors, obtained through the runtime's driver entry point (no
// link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fa_internal.cuh"

namespace fa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A 16-bit (bf16 or fp16, from p.f16) attention tensor viewed as a 3-D array (D, rows, slabs):
//   dense  [B, H, N, D]: rows = N, slabs = B * H;
//   packed [H, T, D]   : rows = T, slabs = H.
// Boxes are 64 columns (128 bytes, one 128-byte swizzle row) x box_rows rows
// of one slab; rows past the slab's end read as zero.
inline bool make_map16(CUtensorMap* map, const void* base, const Problem& p, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const uint64_t rows = p.cu ? (uint64_t)p.T : (uint64_t)p.N;
  const uint64_t slabs = p.cu ? (uint64_t)p.H : (uint64_t)p.B * p.H;
  cuuint64_t dims[3] = {(cuuint64_t)p.D, rows, slabs};
  cuuint64_t strides[2] = {(cuuint64_t)p.D * 2, (cuuint64_t)p.D * 2 * rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, p.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The float32 dQ accumulator [rows, D] as a 2-D array (D, rows) for tensor
// reduce-adds of boxes of 32 columns (128 bytes, one 128-byte swizzle row) x
// 128 rows, read from shared memory in the 128-byte swizzled layout.
inline bool make_map_acc32(CUtensorMap* map, float* base, uint64_t rows, int D) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa
