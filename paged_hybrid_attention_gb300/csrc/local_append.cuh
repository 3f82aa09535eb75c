// The append warp of the local decode kernels' fused-append variants
// (gw_append_decode_attn_local), shared by the bf16 and e4m3 kernels.
//
// "Gemma 4" (pegainfer model page), "Scheduling": every active request
// advances one token per batched step.  The warp walks its CTA's units in
// order and, for each unit that is the last chunk of its (sequence, KV head),
// writes that head's K/V row of the step at position L - 1 with
// gw_kv_append's arithmetic (append_row.cuh), executes
// fence.proxy.async.global (the tensor-map copies read through the
// asynchronous proxy) and raises the CTA's count of processed units with a
// release store; the warp that copies the unit's last page acquires it first.
//
// A row's index reads (its length, its page, its RoPE table entries) are
// issued one row ahead, the first one before the wait on the previous kernel
// when early inputs allow it (they are index inputs); only the K/V loads of
// a row follow the wait.
#pragma once

#include "append_row.cuh"
#include "plan.cuh"

namespace gw {

template <int DT>
__device__ __forceinline__ void local_append_warp(const LocalArgs& a, const int32_t* ub, int total_units,
                                                  int32_t* app_done, bool early) {
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x), stride = static_cast<int>(gridDim.x);
  // the CTA's next unit index >= j that is a last chunk, or -1
  auto next_last = [&](int j) {
    for (;; ++j) {
      const int u = cta + j * stride;
      if (u >= total_units) return -1;
      const int s = plan_seq(ub, a.batch, u);
      const int nc = (ub[s + 1] - ub[s]) / a.kv_heads;
      if ((u - ub[s]) % nc == nc - 1) return j;
    }
  };
  struct Row {
    int j, s, g, pos;
    int32_t page;
    int64_t row;  // the row's index in k_new / v_new
    CosSin8 cs;
  };
  auto fetch = [&](int j) {  // index reads of the row of unit j (j >= 0)
    Row r{};
    r.j = j;
    if (j < 0) return r;
    const int u = cta + j * stride;
    r.s = plan_seq(ub, a.batch, u);
    const int nc = (ub[r.s + 1] - ub[r.s]) / a.kv_heads;
    r.g = (u - ub[r.s]) / nc;
    r.pos = a.seq_lens[r.s] - 1;
    r.page = a.block_table[static_cast<int64_t>(r.s) * a.max_pages + r.pos / kPage];
    r.row = static_cast<int64_t>(a.cu_q_rows[r.s]) * a.kv_heads + r.g;
    if (lane < 16 && r.pos < a.max_pos) r.cs = load_cs8(a.rope_cs + (static_cast<int64_t>(r.pos) * 128 + 8 * lane) * 2);
    return r;
  };
  Row cur = fetch(early ? next_last(0) : -1);
  if (early) {
    pdl_wait();
    pdl_trigger();
  } else {
    cur = fetch(next_last(0));
  }
  for (int j = 0;; ++j) {
    if (cta + j * stride >= total_units) break;
    if (j == cur.j) {
      if (cur.pos >= a.max_pos) {
        if (lane == 0) set_status(a.status, GW_DEV_POS_RANGE);
      } else if (cur.page >= 0 && cur.page < a.num_pages) {  // else the decode side reports the page
        if (lane < 16)
          append_local_item<DT>(const_cast<uint8_t*>(a.pool), a.kv_heads, cur.page, cur.pos % kPage, cur.g,
                                a.k_new + cur.row * 256, a.v_new + cur.row * 256, cur.cs, lane);
        fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) st_release_shared(app_done, j + 1);
      cur = fetch(next_last(j + 1));
    } else {
      __syncwarp();
      if (lane == 0) st_release_shared(app_done, j + 1);
    }
  }
}

}  // namespace gw
