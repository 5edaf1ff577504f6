// tmap.cuh -- host helpers: the driver's tensor-map encoder (looked up through
// the runtime, so the library does not link libcuda) and the tensor map used
// for every [B, S, H, d] operand.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

namespace attnb3 {

inline PFN_cuTensorMapEncodeTiled_v12000& encoder_slot() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  return fn;
}

// Returns true once the encoder entry point is available.
inline bool get_encoder() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encoder_slot() = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encoder_slot() != nullptr;
}

// Tensor map over a dense [B, S, H, d] tensor (bf16, fp16 or 8-bit), dimensions
// listed innermost first as (d, H, S, B) so the byte strides increase. One box
// is `box_elems` consecutive columns of one head for `box_rows` consecutive
// rows, landing in shared memory as box_rows rows of box_elems * esz bytes,
// swizzled in 16-byte units over a 128-byte (or 64-byte) span. Rows past S
// read as zero. Returns true on success.
inline bool encode_bshd(CUtensorMap* map, const void* base, bool fp8, int B, int S, int H, int d,
                        int box_elems, int box_rows, bool f16 = false) {
  const uint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(d * esz), (cuuint64_t)((uint64_t)H * d * esz),
                           (cuuint64_t)((uint64_t)S * H * d * esz)};
  cuuint32_t box[4] = {(cuuint32_t)box_elems, 1u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapSwizzle swz =
      box_elems * esz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = encoder_slot()(
      map,
      fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
          : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16),
      4,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace attnb3
