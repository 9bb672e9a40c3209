// tmap.cuh -- host-side encoding of TMA tensor maps for bf16 row tensors.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace gqa {

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// dependency on the driver library).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [heads][row_pitch rows][cols] bf16 viewed as a 3-D tensor of which only the
// first `rows` rows of each head exist; boxes of box_rows x box_cols (box_cols
// * 2 = 128 bytes), 128-byte swizzle.  Rows past `rows` are never read: the
// copy fills them with zeros.
inline bool encode_bf16_rows(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_pitch,
                             uint64_t heads, uint32_t box_cols, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, heads};
  cuuint64_t strides[2] = {cols * 2, row_pitch * cols * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  auto encode = [&] {
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = encode();
  if (r == CUDA_ERROR_INVALID_CONTEXT) {
    // The driver call needs a current context, and the runtime makes the
    // device's primary context current only on its first call that needs
    // one, which a thread whose first CUDA work is this call has not made
    // yet: make it now, then encode again.
    if (cudaFree(nullptr) != cudaSuccess) return false;
    r = encode();
  }
  return r == CUDA_SUCCESS;
}

}  // namespace gqa
