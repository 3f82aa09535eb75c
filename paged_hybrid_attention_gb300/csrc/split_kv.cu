// Split-KV bookkeeping shared by the local and global decode kernels: the
// plan (unit offsets from sequence lengths) and the log-sum-exp combine.
//
// A sequence's partials are merged in chunk order, so its output depends only
// on its own length and data ("Gemma 4" (pegainfer model page), "Reproducibility
// under concurrency": a row is bit-identical whatever its companions contain).
#include "common.cuh"

namespace gw {
namespace {

__device__ __forceinline__ bool len_ok(const LocalArgs& a, int L, int n) {
  return L >= 1 && L >= n && static_cast<int64_t>(L) <= static_cast<int64_t>(a.max_pages) * kPage;
}

__device__ __forceinline__ int seq_units(const LocalArgs& a, int mode, int chunk, int L) {
  return mode == kSplitLocal ? a.kv_heads * local_chunks(L, a.window, chunk) : global_chunks(L);
}

// One CTA: unit_base[s] = units of decode-row sequences before s; counter = 0.
__global__ void plan_kernel(const LocalArgs a, int mode, int chunk) {
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
      if (n == 1) {
        if (len_ok(a, L, n))
          units = seq_units(a, mode, chunk, L);
        else
          set_status(a.status, GW_DEV_LEN_RANGE);
      }
    }
    int x = units;  // inclusive warp scan
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
    if (s < a.batch) a.unit_base[s] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + units;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.unit_base[a.batch] = carry;
    *a.counter = 0;
    if (carry > a.max_units) set_status(a.status, GW_DEV_WORKSPACE);
  }
}

// One thread per (sequence, q head, 4 dims): merges that head's partials of
// the sequence in chunk order (log-sum-exp, base 2) and writes bf16.
template <int D>
__global__ void combine_kernel(const LocalArgs a, int mode, int G, int chunk) {
  pdl_wait();
  pdl_trigger();
  constexpr int kQ = D / 4;
  const int s = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.num_q_heads * kQ) return;
  const int h = idx / kQ, d4 = idx % kQ;
  const int n = a.cu_q_rows[s + 1] - a.cu_q_rows[s];
  if (n != 1) return;
  const int L = a.seq_lens[s];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (len_ok(a, L, 1) && a.unit_base[a.batch] <= a.max_units) {
    const int nc = mode == kSplitLocal ? local_chunks(L, a.window, chunk) : global_chunks(L);
    const int g = h / G, hh = h % G;
    const int64_t ub = a.unit_base[s] + static_cast<int64_t>(g) * nc;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, a.part_ml[(ub + c) * G + hh].x);
    if (M != -INFINITY) {
#pragma unroll 4
      for (int c = 0; c < nc; ++c) {
        const float2 ml = a.part_ml[(ub + c) * G + hh];
        const float wgt = ex2(ml.x - M);
        den += wgt * ml.y;
        const float4 u = *reinterpret_cast<const float4*>(a.part_o + ((ub + c) * G + hh) * D + d4 * 4);
        acc.x += wgt * u.x;
        acc.y += wgt * u.y;
        acc.z += wgt * u.z;
        acc.w += wgt * u.w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&lo);
  w.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (static_cast<int64_t>(a.cu_q_rows[s]) * a.num_q_heads + h) * D + d4 * 4) = w;
}

}  // namespace

cudaError_t launch_plan(const LocalArgs& a, int mode, int chunk, cudaStream_t st) {
  return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, st, a, mode, chunk);
}

cudaError_t launch_combine(const LocalArgs& a, int mode, int heads_per_unit, int head_dim, int chunk,
                           cudaStream_t st) {
  const int threads = a.num_q_heads * head_dim / 4;
  const dim3 grid((threads + 255) / 256, a.batch);
  if (head_dim == 256) return launch_pdl(combine_kernel<256>, grid, dim3(256), 0, st, a, mode, heads_per_unit, chunk);
  return launch_pdl(combine_kernel<512>, grid, dim3(256), 0, st, a, mode, heads_per_unit, chunk);
}

}  // namespace gw
