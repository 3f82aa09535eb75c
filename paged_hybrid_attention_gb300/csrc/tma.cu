// Host side of the tensor-map copies: the LOCAL pool's TMA descriptor (bf16 or e4m3).
#include <cuda.h>

#include "gw_internal.h"

namespace gw {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<EncodeFn>(fn);
}

}  // namespace

cudaError_t make_local_kv_map(const LocalArgs& a, CUtensorMap* map, int dtype, int box_rows) {
  static const EncodeFn encode = resolve_encode();  // thread-safe one-time lookup
  if (!encode) return cudaErrorNotSupported;
  // a row of 256 elements is 4 chunks of 64 bf16 or 2 chunks of 128 e4m3,
  // 128 bytes each
  const bool e4 = dtype == GW_KV_E4M3;
  const cuuint64_t dims[3] = {e4 ? 128u : 64u, e4 ? 2u : 4u,
                              static_cast<cuuint64_t>(a.num_pages) * a.kv_heads * 2 * kPageTokens};
  const cuuint64_t strides[2] = {128, e4 ? 256u : 512u};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {e4 ? 128u : 64u, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, e4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                            const_cast<uint8_t*>(a.pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gw
