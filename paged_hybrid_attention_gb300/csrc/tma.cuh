// Tensor-map (TMA) copies of LOCAL pool rows into 128-byte-swizzled shared
// memory.  The map is built on the host by make_local_kv_map (tma.cu): the
// pool viewed as rows of 256 bf16 (one token of K or of V of one KV head),
// each split into 4 chunks of 64 elements; row index = ((page * kv_heads +
// head) * 2 + {0: K, 1: V}) * 16 + token.  A box is {64 elements, 1 chunk,
// 16 rows}: the 16 tokens of one page head, one 64-dim chunk, 2 KB landing
// as 16 rows of 128 B with the 16-byte units of row r XOR-ed by r % 8.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace gw {

__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap* map, int chunk, int row, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(chunk), "r"(row), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Byte offset of 16-byte unit u of row r in a 128-byte-swizzled region.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

}  // namespace gw
