// gw_kv_append kernels: RoPE on the rotated slice of K, then page write.
//
// "Gemma 4" (pegainfer model page), "Architecture notes": local K rotates all
// 256 dims (theta 10k); global K rotates 128 of 512 dims with the full head
// dim as frequency denominator (theta 1M); global V is K's projection without
// RoPE.  "Gewell - Gemma4 inference engine", "the Why": a global token is
// cached as V plus the rotated K slice.  "feat(gemma4): the sliding family
// serves an opt in fp8 KV pool", "Description": local K/V may be stored e4m3
// at scale 1.0.
//
// Every thread handles 8 rotation pairs (or 8 copied elements): one 16-byte
// load per operand and one 16-byte (bf16) or 8-byte (e4m3) store per output
// chunk.  The rotation is evaluated with explicitly rounded binary32 multiply
// and add (__fmul_rn / __fsub_rn / __fadd_rn), so no multiply-add is fused
// and the stored bits are exactly those of the stated operation order.
#include "append_row.cuh"

namespace gw {
namespace {

// 0 if the row's slot and pos are in range, else the GW_DEV_* bit to report.
__device__ __forceinline__ int32_t row_check(const AppendArgs& a, int64_t row, int32_t& slot, int32_t& pos) {
  slot = a.slot[row];
  pos = a.pos[row];
  if (slot < 0 || static_cast<int64_t>(slot) >= a.num_pages * kPage) return GW_DEV_SLOT_RANGE;
  if (pos < 0 || pos >= a.max_pos) return GW_DEV_POS_RANGE;
  return 0;
}

// Programmatic dependent launch: slot, pos and the RoPE table are index
// inputs, read before the wait on the previous kernel when the caller allows
// it (gw_set_early_inputs); k, v, the pool and the status word only after.
struct PdlGate {
  bool waited;
  __device__ explicit PdlGate(const AppendArgs& a) : waited(a.early_inputs == 0) {
    if (waited) {
      pdl_wait();
      pdl_trigger();
    }
  }
  __device__ void pass() {
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
  }
};

// LOCAL: one work item = (row, kv head, j in [0,16)): pairs (8j+i, 128+8j+i)
// of K, and V chunks 8j and 128+8j.
template <int DT>
__global__ void append_local_kernel(const AppendArgs a) {
  PdlGate gate(a);
  const int64_t total = static_cast<int64_t>(a.num_rows) * a.kv_heads * 16;
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(w % 16);
    const int64_t rh = w / 16;
    const int g = static_cast<int>(rh % a.kv_heads);
    const int64_t row = rh / a.kv_heads;
    int32_t slot, pos;
    const int32_t bad = row_check(a, row, slot, pos);
    const CosSin8 cs = load_cs8(a.rope_cs + (static_cast<int64_t>(bad ? 0 : pos) * 128 + 8 * j) * 2);
    gate.pass();
    if (bad) {
      if (j == 0 && g == 0) set_status(a.status, bad);
      continue;
    }
    const int64_t page = slot / kPage, off = slot % kPage;
    append_local_item<DT>(a.pool, a.kv_heads, page, static_cast<int>(off), g, a.k + (row * a.kv_heads + g) * 256,
                          a.v + (row * a.kv_heads + g) * 256, cs, j);
  }
}

// GLOBAL FOLDED: row = V[0:512] || k_rot[0:128]; items per row: 64 V chunks
// + 8 rotation items (pairs 8t..8t+7 and 64+8t..).  The e4m3 folded pool has
// the same items, each rounding its 8 elements once to e4m3 (8-byte stores).
// GLOBAL FULL:   row = K[0:512] || V[0:512]; items per row: 8 rotation items,
// 48 copies of k[128:512], 64 V chunks.
template <int LAYOUT>
__global__ void append_global_kernel(const AppendArgs a) {
  using R = GlobalRow<LAYOUT>;
  PdlGate gate(a);
  const int64_t total = static_cast<int64_t>(a.num_rows) * R::kItems;
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int it = static_cast<int>(w % R::kItems);
    const int64_t row = w / R::kItems;
    int32_t slot, pos;
    const int32_t bad = row_check(a, row, slot, pos);
    const int t = R::rot_item(it);
    CosSin8 cs{};
    if (t >= 0) cs = load_cs8(a.rope_cs + (static_cast<int64_t>(bad ? 0 : pos) * 64 + 8 * t) * 2);
    gate.pass();
    if (bad) {
      if (it == 0) set_status(a.status, bad);
      continue;
    }
    append_global_item<LAYOUT>(a.pool, slot / kPage, slot % kPage, a.k + row * 512, a.v + row * 512, cs, it);
  }
}

// One (cos, sin) entry per item: item w = pos * half + i.  The frequency,
// the angle and both trigonometric values are float64; each value is rounded
// once to float32.
__global__ void rope_cs_kernel(float2* out, double theta, int half, int head_dim, int64_t total) {
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(w % half);
    const int64_t p = w / half;
    const double inv_f = pow(theta, (-2.0 * static_cast<double>(i)) / static_cast<double>(head_dim));
    const double ang = static_cast<double>(p) * inv_f;
    double s, c;
    sincos(ang, &s, &c);
    out[w] = make_float2(__double2float_rn(c), __double2float_rn(s));
  }
}

int grid_for(int64_t items, int block) {
  int64_t blocks = (items + block - 1) / block;
  const int64_t cap = static_cast<int64_t>(grid_ctas()) * 16;
  return static_cast<int>(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace

cudaError_t launch_rope_cs(float* out, double theta, int rot_dim, int head_dim, int max_pos, cudaStream_t st) {
  constexpr int kBlock = 256;
  const int64_t total = static_cast<int64_t>(max_pos) * (rot_dim / 2);
  return launch_pdl(rope_cs_kernel, dim3(grid_for(total, kBlock)), dim3(kBlock), 0, st, reinterpret_cast<float2*>(out),
                    theta, rot_dim / 2, head_dim, total);
}

cudaError_t launch_append(int layout, int dtype, const AppendArgs& a, cudaStream_t st) {
  constexpr int kBlock = 256;
  if (layout == GW_LAYOUT_LOCAL) {
    const int grid = grid_for(static_cast<int64_t>(a.num_rows) * a.kv_heads * 16, kBlock);
    if (dtype == GW_KV_BF16) return launch_pdl(append_local_kernel<GW_KV_BF16>, dim3(grid), dim3(kBlock), 0, st, a);
    return launch_pdl(append_local_kernel<GW_KV_E4M3>, dim3(grid), dim3(kBlock), 0, st, a);
  }
  if (layout == GW_LAYOUT_GLOBAL_FOLDED_E4M3)
    return launch_pdl(append_global_kernel<GW_LAYOUT_GLOBAL_FOLDED_E4M3>,
                      dim3(grid_for(static_cast<int64_t>(a.num_rows) * 72, kBlock)), dim3(kBlock), 0, st, a);
  if (layout == GW_LAYOUT_GLOBAL_FOLDED)
    return launch_pdl(append_global_kernel<GW_LAYOUT_GLOBAL_FOLDED>,
                      dim3(grid_for(static_cast<int64_t>(a.num_rows) * 72, kBlock)), dim3(kBlock), 0, st, a);
  return launch_pdl(append_global_kernel<GW_LAYOUT_GLOBAL_FULL>,
                    dim3(grid_for(static_cast<int64_t>(a.num_rows) * 120, kBlock)), dim3(kBlock), 0, st, a);
}

}  // namespace gw
