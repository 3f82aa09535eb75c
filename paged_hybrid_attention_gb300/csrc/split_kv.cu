// The log-sum-exp combine of split-KV partials, shared by the local and
// global decode kernels (their plans are computed in-kernel, plan.cuh).
//
// A sequence's partials are merged in chunk order, so its output depends only
// on its own length and data ("Gemma 4" (pegainfer model page), "Reproducibility
// under concurrency": a row is bit-identical whatever its companions contain).
#include "common.cuh"

namespace gw {
namespace {

// A task is (sequence, q head, 128-dim slice); lane l owns 4 dims of the
// slice.  The sequence's units of this head's group are consecutive
// (unit_base holds the plan the decode kernel used), and its nc chunks are
// merged in groups of kB: with M the maximum of the chunks' m and
// w_c = 2^(m_c - M),
//   S_g = sum over the group's chunks, in chunk order, of w_c * o_c
//   D_g = sum over the group's chunks, in chunk order, of w_c * l_c
//   o   = (S_0 + S_1 + ...) / (D_0 + D_1 + ...), groups added in order.
// That arithmetic depends only on nc, so a row's bits never depend on how
// the tasks are mapped to warps.  A task gets W warps (1, 4 or 8, chosen
// from the call's bound on chunks per sequence): warp j of the task merges
// groups j, j + W, ... (R rounds), the task's maximum and group sums meeting
// in shared memory, so a long sequence's partials are fetched by W warps at
// once.  Lane b < kB fetches (m, l) of the group's chunk b, every lane its
// dims of all kB chunks.  The result is written as bf16.  With `discard`,
// each merged chunk slice is then dropped from L2 unwritten (nothing reads
// it again before the next decode call rewrites it).
template <int D>
__global__ void __launch_bounds__(256, 2) combine_kernel(const LocalArgs a, int G, int W, int R, bool discard) {
  constexpr int kSlices = D / 128;
  constexpr int kB = 16;  // chunks per group
  __shared__ float4 s_sum[8][32];
  __shared__ float s_den[8], s_max[8];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j = warp % W, tw = warp - j;  // warp within the task, the task's first warp
  const int64_t task = (static_cast<int64_t>(blockIdx.x) * 8 + warp) / W;
  const bool in_grid = task < static_cast<int64_t>(a.batch) * a.num_q_heads * kSlices;
  const int slice = static_cast<int>(task % kSlices);
  const int64_t sh = task / kSlices;
  const int s = in_grid ? static_cast<int>(sh / a.num_q_heads) : 0;
  const int h = static_cast<int>(sh % a.num_q_heads);
  // independent loads, issued together (one round trip before the partials)
  const int row0 = a.cu_q_rows[s], row1 = a.cu_q_rows[s + 1];
  const int ub_s = a.unit_base[s], ub_s1 = a.unit_base[s + 1], ub_total = a.unit_base[a.batch];
  const bool live = in_grid && row1 - row0 == 1;
  const int groups = a.num_q_heads / G;  // units of a sequence = groups x chunks
  const int nc = live && ub_total <= a.max_units ? (ub_s1 - ub_s) / groups : 0;
  const int64_t ub = ub_s + static_cast<int64_t>(h / G) * nc;
  const int hh = h % G;
  const int dim0 = slice * 128 + lane * 4;
  float4 u[kB];
  float2 ml = make_float2(-INFINITY, 0.f);
  const float2* ml_base = a.part_ml + ub * G + hh;  // chunk c at ml_base[c * G]
  const float* o_base = a.part_o + (ub * G + hh) * D + dim0;  // chunk c at o_base + c * G * D
  const int o_stride = G * D;
  const float* line_base = o_base - lane * 4;  // the slice's first 128-byte line, chunk 0
  auto fetch = [&](int g) {
    const int c0 = g * kB;
    if (lane < kB && c0 + lane < nc) ml = ml_base[(c0 + lane) * G];
    const float* po = o_base + static_cast<int64_t>(c0) * o_stride;
#pragma unroll
    for (int b = 0; b < kB; ++b)
      if (c0 + b < nc) u[b] = *reinterpret_cast<const float4*>(po + b * o_stride);
  };
  fetch(j);
  // the maximum over this warp's groups, then over the task's warps
  float mx = ml.x;
  for (int r = 1; r < R; ++r) {
    const int c = (r * W + j) * kB + lane;
    if (lane < kB && c < nc) mx = fmaxf(mx, ml_base[c * G].x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float M = mx;
  if (W > 1) {
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    for (int k = 0; k < W; ++k) M = fmaxf(M, s_max[tw + k]);
  }
  float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  auto add = [&](int g, const float4& sg, float dg) {  // groups in order
    if (g == 0) {
      tot = sg;
      den = dg;
    } else {
      tot.x += sg.x;
      tot.y += sg.y;
      tot.z += sg.z;
      tot.w += sg.w;
      den += dg;
    }
  };
  for (int r = 0; r < R; ++r) {
    const int g = r * W + j;
    if (r > 0) fetch(g);
    float4 sg = make_float4(0.f, 0.f, 0.f, 0.f);
    float dg = 0.f;
    if (M != -INFINITY) {
      const float wl = lane < kB && g * kB + lane < nc ? ex2(ml.x - M) : 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        if (g * kB + b < nc) {
          const float wb = __shfl_sync(0xffffffffu, wl, b);
          const float lb = __shfl_sync(0xffffffffu, ml.y, b);
          dg = fmaf(wb, lb, dg);
          sg.x = fmaf(wb, u[b].x, sg.x);
          sg.y = fmaf(wb, u[b].y, sg.y);
          sg.z = fmaf(wb, u[b].z, sg.z);
          sg.w = fmaf(wb, u[b].w, sg.w);
        }
      }
      if (discard) {
        // every lane has consumed its loads of the group's slices: drop
        // their four 128-byte lines per chunk
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int idx = lane + 32 * k, b = idx >> 2;
          if (g * kB + b < nc)
            discard_l2(line_base + static_cast<int64_t>(g * kB + b) * o_stride + (idx & 3) * 32);
        }
      }
    }
    if (W == 1) {
      if (g * kB < nc) add(g, sg, dg);
    } else {
      s_sum[warp][lane] = sg;
      if (lane == 0) s_den[warp] = dg;
      __syncthreads();
      if (j == 0)
        for (int k = 0; k < W; ++k)
          if ((r * W + k) * kB < nc) add(r * W + k, s_sum[tw + k][lane], s_den[tw + k]);
      __syncthreads();
    }
  }
  if (j != 0 || !live) return;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(tot.x * inv, tot.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(tot.z * inv, tot.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&lo);
  w.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (static_cast<int64_t>(row0) * a.num_q_heads + h) * D + dim0) = w;
  // log-sum-exp of the row's logits, natural log (the partials are in base-2
  // units of the scaled logits): ln(sum_j e^{scale q.k_j}) = ln2 (M + log2 den)
  if (a.lse && slice == 0 && lane == 0)
    a.lse[static_cast<int64_t>(row0) * a.num_q_heads + h] = den > 0.f ? 0.6931471805599453f * (M + log2f(den)) : -INFINITY;
}

// gw_merge_lse: one warp per (row, head); lane l owns dims [8 l', ...) in
// 16-byte chunks.  Parts are added in part order.
__global__ void __launch_bounds__(256) merge_lse_kernel(const MergeArgs m) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t task = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (task >= static_cast<int64_t>(m.rows) * m.heads) return;
  float M = -INFINITY;
  for (int r = 0; r < m.n_parts; ++r) M = fmaxf(M, m.lse[r][task]);
  float w[kMaxMergeParts];
  float den = 0.f;
  for (int r = 0; r < m.n_parts; ++r) {
    w[r] = M == -INFINITY ? 0.f : __expf(m.lse[r][task] - M);
    den += w[r];
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int c = lane; c < m.head_dim / 8; c += 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < m.n_parts; ++r) {
      if (w[r] == 0.f) continue;  // a part without keys: its bytes may be anything
      float x[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(m.o[r] + task * m.head_dim + 8 * c), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[r], x[i], acc[i]);
    }
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      pk[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(m.out + task * m.head_dim + 8 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (m.lse_out && lane == 0) m.lse_out[task] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge_lse(const MergeArgs& m, cudaStream_t st) {
  const int64_t tasks = static_cast<int64_t>(m.rows) * m.heads;
  return launch_pdl(merge_lse_kernel, dim3(static_cast<unsigned>((tasks + 7) / 8)), dim3(256), 0, st, m);
}

cudaError_t launch_combine(const LocalArgs& a, int heads_per_unit, int head_dim, int max_chunks, bool discard,
                           cudaStream_t st) {
  constexpr int kB = 16;
  const int ngroups = (max_chunks + kB - 1) / kB;
  // One warp walks up to two groups itself (a serving layer's block table
  // bounds a sequence at 15 global or 9 local chunks); longer sequences
  // spread their groups over 4 or 8 warps of one CTA.
  const int W = ngroups <= 2 ? 1 : ngroups <= 4 ? 4 : 8;
  const int R = (ngroups + W - 1) / W > 0 ? (ngroups + W - 1) / W : 1;
  const int64_t warps = static_cast<int64_t>(a.batch) * a.num_q_heads * (head_dim / 128) * W;
  const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
  if (head_dim == 256) return launch_pdl(combine_kernel<256>, grid, dim3(256), 0, st, a, heads_per_unit, W, R, discard);
  return launch_pdl(combine_kernel<512>, grid, dim3(256), 0, st, a, heads_per_unit, W, R, discard);
}

}  // namespace gw
