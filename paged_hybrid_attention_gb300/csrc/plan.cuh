// The split-KV plan of a decode call, computed inside the decode kernels.
//
// Every CTA scans the batch's lengths into its own shared memory (a few
// hundred nanoseconds for serving batches), so no plan kernel and no work
// counter sit in front of the decode.  Units are dealt round-robin over the
// CTAs (or warps), so the plan is all a CTA needs to find its own work.
#pragma once

#include "common.cuh"

namespace gw {

__device__ __forceinline__ bool plan_len_ok(const LocalArgs& a, int L) {
  return L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(a.max_pages) * kPage;
}

// ub[s] = units of the decode-row sequences before s (ub[batch] = total),
// with units_of(L) the units of one decode row of length L.  Rows of invalid
// length (L < 1 or beyond the block table) get no units.  Must be called by
// every thread of the block; scratch holds 32 ints.  With `publish`, CTA 0
// also stores the plan to the workspace for the combine kernel and raises
// GW_DEV_LEN_RANGE for invalid rows; without it (a plan made before the wait
// on the previous kernel) nothing is written to global memory, and
// publish_plan does both once the wait is over.
template <class UnitsOf>
__device__ void plan_in_smem(const LocalArgs& a, int32_t* ub, int32_t* scratch, UnitsOf units_of,
                             bool publish = true) {
  const int nt = blockDim.x, t = threadIdx.x;
  const int per = (a.batch + nt - 1) / nt;
  const int s0 = min(a.batch, t * per), s1 = min(a.batch, s0 + per);
  int mine = 0;
  for (int s = s0; s < s1; ++s) {
    const int n = a.cu_q_rows[s + 1] - a.cu_q_rows[s];
    const int L = a.seq_lens[s];
    int units = 0;
    if (n == 1) {
      if (plan_len_ok(a, L))
        units = units_of(L);
      else if (blockIdx.x == 0 && publish)
        set_status(a.status, GW_DEV_LEN_RANGE);
    }
    ub[s] = units;  // per-sequence count for now
    mine += units;
  }
  // exclusive scan of the per-thread sums
  const int lane = t & 31, w = t >> 5;
  int x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[w] = x;
  __syncthreads();
  if (w == 0) {
    int v = lane < (nt >> 5) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane < (nt >> 5)) scratch[lane] = v;
  }
  __syncthreads();
  int run = (w > 0 ? scratch[w - 1] : 0) + x - mine;
  for (int s = s0; s < s1; ++s) {
    const int c = ub[s];
    ub[s] = run;
    run += c;
  }
  if (t == nt - 1) ub[a.batch] = run;
  __syncthreads();
  if (blockIdx.x == 0 && publish)
    for (int s = t; s <= a.batch; s += nt) a.unit_base[s] = ub[s];
}

// The global half of a plan made with publish = false, once the previous
// kernel has finished: CTA 0's threads t of nt store the plan and raise
// GW_DEV_LEN_RANGE for invalid decode rows.
__device__ __forceinline__ void publish_plan(const LocalArgs& a, const int32_t* ub, int t, int nt) {
  if (blockIdx.x != 0) return;
  for (int s = t; s <= a.batch; s += nt) {
    a.unit_base[s] = ub[s];
    if (s < a.batch && a.cu_q_rows[s + 1] - a.cu_q_rows[s] == 1 && !plan_len_ok(a, a.seq_lens[s]))
      set_status(a.status, GW_DEV_LEN_RANGE);
  }
}

// The sequence that owns unit u (0 <= u < ub[batch]): the largest s with
// ub[s] <= u, which skips sequences without units.
__device__ __forceinline__ int plan_seq(const int32_t* ub, int batch, int u) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ub[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace gw
