// Host-side helpers shared by the CUDA entry points: error conversion, argument checks and
// encoding of TMA tensor maps through the driver entry point (no link-time libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <string>

#include "fcp_internal.h"

namespace fcp {

inline fcp_status cuda_fail(cudaError_t e, const char* where) {
  set_last_error(std::string(where) + ": " + cudaGetErrorString(e));
  return FCP_ERR_CUDA;
}

#define FCP_CUDA_TRY(expr, where)              \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map over a contiguous bf16 tensor [heads, T, D], box {64, rows, 1} with 128-byte
// swizzle: one box is `rows` tokens x 64 channels (128 bytes per row). Out-of-range rows
// read as zero.
inline fcp_status make_bf16_map(CUtensorMap* map, const void* base, int heads, int64_t T, int D, int rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return FCP_ERR_CUDA;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r)));
    return FCP_ERR_CUDA;
  }
  return FCP_OK;
}

// Tensor map over a contiguous float32 tensor [heads, T, D] (D innermost) with box
// {D, rows, 1}, no swizzle: one box is `rows` tokens x D channels (the dQ accumulator that
// the backward's reduce-adds target).
inline fcp_status make_f32_map(CUtensorMap* map, const void* base, int heads, int64_t T, int D, int rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) {
    set_last_error("cuTensorMapEncodeTiled unavailable from the driver");
    return FCP_ERR_CUDA;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(T) * D * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled (float32) failed with CUresult " + std::to_string(static_cast<int>(r)));
    return FCP_ERR_CUDA;
  }
  return FCP_OK;
}

template <class T>
inline const T* dev_array(const void* d_plan, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const uint8_t*>(d_plan) + off);
}

inline int* dev_error_word(const void* d_plan) {
  return reinterpret_cast<int*>(const_cast<void*>(d_plan));
}

}  // namespace fcp
