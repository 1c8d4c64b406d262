// Host helper: encode TMA tensor maps for [rows, heads, head_dim] bf16
// activations (tokens x heads x d, head_dim contiguous) through the driver
// entry point obtained from the runtime, so the library needs no -lcuda.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cstdint>

namespace cpattn {

inline PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor of `rows` tokens, `heads` heads and `d` features (bf16, d
// contiguous, rows strided by heads*d). The box is 64 features x 1 head x
// `box_rows` tokens with 128-byte swizzle, i.e. one 128-byte swizzle atom
// column of a tile; a d=128 tile takes two boxes (x = 0 and x = 64).
// `rows` may exceed 2^31 only in principle; callers keep it below.
inline bool encode_bf16_rows_heads_d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t heads,
                                     uint64_t d, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d, heads, rows};
  cuuint64_t strides[2] = {d * 2, heads * d * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace cpattn
