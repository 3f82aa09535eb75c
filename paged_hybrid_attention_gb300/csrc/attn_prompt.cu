// Prompt rows of a mixed step: sequences that contribute n > 1 query rows.
//
// "Gemma 4" (pegainfer model page), "Scheduling": a new prompt's rows are
// computed in the same batched step as the live streams' next token.  Row r
// of such a sequence sits at position p = L - n + r (the prompt's own K/V were
// appended first in the same step) and attends causally: keys
// [max(0, p - W + 1), p] on local layers, [0, p] on global layers.
//
// This file holds the tile plan shared by both families and the launchers;
// the kernels are on the tensor cores: attn_prompt_tc.cu (local layers) and
// attn_prompt_global_tc.cu (global layers).  Tiles of (sequence, KV head or
// output-dim half, query block) are enumerated by a one-CTA plan kernel and
// processed by persistent CTAs.
#include "common.cuh"

namespace gw {
namespace {

// One CTA: prompt_base[s] = prompt tiles of sequences before s.  A sequence
// with n > 1 rows contributes heads_factor * ceil(n / queries_per_tile).
__global__ void plan_prompt_kernel(const LocalArgs a, int heads_factor, int queries_per_tile) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int base = 0; base < a.batch; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int units = 0;
    if (s < a.batch) {
      const int n = a.cu_q_rows[s + 1] - a.cu_q_rows[s];
      const int L = a.seq_lens[s];
      if (n > 1) {
        if (L >= n && static_cast<int64_t>(L) <= static_cast<int64_t>(a.max_pages) * kPage)
          units = heads_factor * ((n + queries_per_tile - 1) / queries_per_tile);
        else
          set_status(a.status, GW_DEV_LEN_RANGE);
      }
    }
    int x = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      warp_sums[lane] = v;
    }
    __syncthreads();
    const int excl = carry + (w > 0 ? warp_sums[w - 1] : 0) + x - units;
    if (s < a.batch) a.prompt_base[s] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + units;
    __syncthreads();
  }
  if (threadIdx.x == 0) a.prompt_base[a.batch] = carry;
}

template <int G>
cudaError_t launch_local_g(int dtype, const LocalArgs& a, cudaStream_t st) {
  cudaError_t e = launch_pdl(plan_prompt_kernel, dim3(1), dim3(1024), 0, st, a, a.kv_heads, 128 / G);
  if (e != cudaSuccess) return e;
  return launch_local_prompt_tc(dtype, G, a, st);
}

template <int HQ>
cudaError_t launch_global_hq(int layout, const LocalArgs& a, cudaStream_t st) {
  cudaError_t e = launch_pdl(plan_prompt_kernel, dim3(1), dim3(1024), 0, st, a, 2, 128 / HQ);
  if (e != cudaSuccess) return e;
  return launch_global_prompt_tc(layout, a, st);
}


}  // namespace

cudaError_t launch_local_prompt(int dtype, int group, const LocalArgs& a, int /*max_q_rows*/, cudaStream_t st) {
  switch (group) {
    case 1: return launch_local_g<1>(dtype, a, st);
    case 2: return launch_local_g<2>(dtype, a, st);
    case 4: return launch_local_g<4>(dtype, a, st);
    case 8: return launch_local_g<8>(dtype, a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_global_prompt(int layout, const LocalArgs& a, int /*max_q_rows*/, cudaStream_t st) {
  switch (a.num_q_heads) {
    case 8: return launch_global_hq<8>(layout, a, st);
    case 16: return launch_global_hq<16>(layout, a, st);
    case 32: return launch_global_hq<32>(layout, a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gw
