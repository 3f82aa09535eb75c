// The log-sum-exp combine of split-KV partials, shared by the local and
// global decode kernels (their plans are computed in-kernel, plan.cuh).
//
// A sequence's partials are merged in chunk order, so its output depends only
// on its own length and data ("Gemma 4" (pegainfer model page), "Reproducibility
// under concurrency": a row is bit-identical whatever its companions contain).
#include "common.cuh"

namespace gw {
namespace {

// One warp per (sequence, q head, 128-dim slice); lane l owns 4 dims of the
// slice.  The sequence's units of this head's group are consecutive (unit_base
// holds the plan the decode kernel used).  The (m, l) of chunks lane,
// lane + 32, ... give the warp maximum M while the first batch of kB chunks'
// partials is already being fetched; then every lane sums w_c * o_c over its
// dims in chunk order, kB chunks' loads in flight at a time.  The result is
// written as bf16.
template <int D>
__global__ void combine_kernel(const LocalArgs a, int G) {
  constexpr int kSlices = D / 128;
  constexpr int kB = 16;  // chunks per batch
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= static_cast<int64_t>(a.batch) * a.num_q_heads * kSlices) return;
  const int slice = static_cast<int>(wid % kSlices);
  const int64_t sh = wid / kSlices;
  const int s = static_cast<int>(sh / a.num_q_heads), h = static_cast<int>(sh % a.num_q_heads);
  // independent loads, issued together (one round trip before the partials)
  const int row0 = a.cu_q_rows[s], row1 = a.cu_q_rows[s + 1];
  const int ub_s = a.unit_base[s], ub_s1 = a.unit_base[s + 1], ub_total = a.unit_base[a.batch];
  if (row1 - row0 != 1) return;
  const int groups = a.num_q_heads / G;  // units of a sequence = groups x chunks
  const int nc = ub_total <= a.max_units ? (ub_s1 - ub_s) / groups : 0;
  const int g = h / G, hh = h % G;
  const int64_t ub = ub_s + static_cast<int64_t>(g) * nc;
  const int dim0 = slice * 128 + lane * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  float4 u[kB];
  float2 ml[kB];
  auto fetch = [&](int c0) {
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      if (c0 + b < nc) {
        const int64_t row = (ub + c0 + b) * G + hh;
        ml[b] = a.part_ml[row];
        u[b] = *reinterpret_cast<const float4*>(a.part_o + row * D + dim0);
      }
    }
  };
  fetch(0);
  float M = -INFINITY;
  for (int c = lane; c < nc; c += 32) M = fmaxf(M, a.part_ml[(ub + c) * G + hh].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M != -INFINITY) {
    for (int c0 = 0; c0 < nc; c0 += kB) {
      if (c0 > 0) fetch(c0);
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        if (c0 + b < nc) {
          const float wgt = ex2(ml[b].x - M);
          den += wgt * ml[b].y;
          acc.x += wgt * u[b].x;
          acc.y += wgt * u[b].y;
          acc.z += wgt * u[b].z;
          acc.w += wgt * u[b].w;
        }
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&lo);
  w.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (static_cast<int64_t>(row0) * a.num_q_heads + h) * D + dim0) = w;
}

}  // namespace

cudaError_t launch_combine(const LocalArgs& a, int heads_per_unit, int head_dim, cudaStream_t st) {
  const int64_t warps = static_cast<int64_t>(a.batch) * a.num_q_heads * (head_dim / 128);
  const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
  if (head_dim == 256) return launch_pdl(combine_kernel<256>, grid, dim3(256), 0, st, a, heads_per_unit);
  return launch_pdl(combine_kernel<512>, grid, dim3(256), 0, st, a, heads_per_unit);
}

}  // namespace gw
