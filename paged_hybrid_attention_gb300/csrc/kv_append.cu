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
#include "common.cuh"

namespace gw {
namespace {

__device__ __forceinline__ void load_bf16x8(const uint16_t* p, float (&f)[8]) {
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(p), f);
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // .x = low half
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint2 f32x8_to_e4m3(const float (&f)[8]) {
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i], f[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
    uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i + 2], f[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
    w[i] = (lo & 0xFFFFu) | (hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

// The (cos, sin) table entries of 8 rotation pairs: cs[2i], cs[2i+1].
struct CosSin8 {
  float c[8], s[8];
};

__device__ __forceinline__ CosSin8 load_cs8(const float* cs) {
  CosSin8 r;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    float4 t = *reinterpret_cast<const float4*>(cs + 2 * i);
    r.c[i] = t.x;
    r.s[i] = t.y;
    r.c[i + 1] = t.z;
    r.s[i + 1] = t.w;
  }
  return r;
}

// Rotate 8 pairs (x0[i], x1[i]) by the angles of cs.
__device__ __forceinline__ void rotate8(float (&x0)[8], float (&x1)[8], const CosSin8& cs) {
  const float (&c)[8] = cs.c;
  const float (&s)[8] = cs.s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float r0 = __fsub_rn(__fmul_rn(x0[i], c[i]), __fmul_rn(x1[i], s[i]));
    const float r1 = __fadd_rn(__fmul_rn(x1[i], c[i]), __fmul_rn(x0[i], s[i]));
    x0[i] = r0;
    x1[i] = r1;
  }
}

template <int DT>
__device__ __forceinline__ void store8(uint8_t* base, int64_t elem, const float (&f)[8]) {
  if constexpr (DT == GW_KV_BF16) {
    *reinterpret_cast<uint4*>(base + elem * 2) = f32x8_to_bf16(f);
  } else {
    *reinterpret_cast<uint2*>(base + elem) = f32x8_to_e4m3(f);
  }
}

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
    const uint16_t* krow = a.k + (row * a.kv_heads + g) * 256;
    const uint16_t* vrow = a.v + (row * a.kv_heads + g) * 256;
    float x0[8], x1[8];
    load_bf16x8(krow + 8 * j, x0);
    load_bf16x8(krow + 128 + 8 * j, x1);
    rotate8(x0, x1, cs);
    const int64_t kbase = (((page * a.kv_heads + g) * 2 + 0) * kPage + off) * 256;
    const int64_t vbase = (((page * a.kv_heads + g) * 2 + 1) * kPage + off) * 256;
    store8<DT>(a.pool, kbase + 8 * j, x0);
    store8<DT>(a.pool, kbase + 128 + 8 * j, x1);
    if constexpr (DT == GW_KV_BF16) {
      uint16_t* p = reinterpret_cast<uint16_t*>(a.pool);
      *reinterpret_cast<uint4*>(p + vbase + 8 * j) = *reinterpret_cast<const uint4*>(vrow + 8 * j);
      *reinterpret_cast<uint4*>(p + vbase + 128 + 8 * j) = *reinterpret_cast<const uint4*>(vrow + 128 + 8 * j);
    } else {
      float v0[8], v1[8];
      load_bf16x8(vrow + 8 * j, v0);
      load_bf16x8(vrow + 128 + 8 * j, v1);
      store8<DT>(a.pool, vbase + 8 * j, v0);
      store8<DT>(a.pool, vbase + 128 + 8 * j, v1);
    }
  }
}

// Element index of (page, token o, row element e) in a GLOBAL page whose
// rows have kRow elements, blocked 8 tokens x 8 elements.
template <int kRow>
__device__ __forceinline__ int64_t tiled(int64_t page, int o, int e) {
  constexpr int kBlk = kRow / 8;
  return page * (kPage * kRow) + ((static_cast<int64_t>(o / 8) * kBlk + e / 8) * 8 + (o % 8)) * 8 + (e % 8);
}

// Byte offset of (page, token o, row element e) in a GLOBAL_FOLDED_E4M3 page:
// rows of 640 one-byte elements, blocked 8 tokens x 16 elements.
__device__ __forceinline__ int64_t tiled_e4m3(int64_t page, int o, int e) {
  return page * (kPage * 640) + ((static_cast<int64_t>(o / 8) * 40 + e / 16) * 8 + (o % 8)) * 16 + (e % 16);
}

// GLOBAL FOLDED: row = V[0:512] || k_rot[0:128]; items per row: 64 V chunks
// + 8 rotation items (pairs 8t..8t+7 and 64+8t..).  The e4m3 folded pool has
// the same items, each rounding its 8 elements once to e4m3 (8-byte stores).
// GLOBAL FULL:   row = K[0:512] || V[0:512]; items per row: 8 rotation items,
// 48 copies of k[128:512], 64 V chunks.
template <int LAYOUT>
__global__ void append_global_kernel(const AppendArgs a) {
  constexpr bool kE4 = LAYOUT == GW_LAYOUT_GLOBAL_FOLDED_E4M3;
  constexpr bool kFolded = LAYOUT == GW_LAYOUT_GLOBAL_FOLDED || kE4;
  constexpr int kRow = kFolded ? 640 : 1024;
  constexpr int kItems = kFolded ? 72 : 120;
  PdlGate gate(a);
  const int64_t total = static_cast<int64_t>(a.num_rows) * kItems;
  uint16_t* pool = reinterpret_cast<uint16_t*>(a.pool);
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int it = static_cast<int>(w % kItems);
    const int64_t row = w / kItems;
    int32_t slot, pos;
    const int32_t bad = row_check(a, row, slot, pos);
    const int rot_item = kFolded ? it - 64 : it;  // rotation items
    const bool rot = rot_item >= 0 && rot_item < 8;
    CosSin8 cs{};
    if (rot) cs = load_cs8(a.rope_cs + (static_cast<int64_t>(bad ? 0 : pos) * 64 + 8 * rot_item) * 2);
    gate.pass();
    if (bad) {
      if (it == 0) set_status(a.status, bad);
      continue;
    }
    const int64_t page = slot / kPage;
    const int off = slot % kPage;
    const uint16_t* krow = a.k + row * 512;
    const uint16_t* vrow = a.v + row * 512;
    if (rot) {
      const int t = rot_item;
      float x0[8], x1[8];
      load_bf16x8(krow + 8 * t, x0);
      load_bf16x8(krow + 64 + 8 * t, x1);
      rotate8(x0, x1, cs);
      const int e0 = kFolded ? 512 + 8 * t : 8 * t;
      if constexpr (kE4) {
        *reinterpret_cast<uint2*>(a.pool + tiled_e4m3(page, off, e0)) = f32x8_to_e4m3(x0);
        *reinterpret_cast<uint2*>(a.pool + tiled_e4m3(page, off, e0 + 64)) = f32x8_to_e4m3(x1);
      } else {
        *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e0)) = f32x8_to_bf16(x0);
        *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e0 + 64)) = f32x8_to_bf16(x1);
      }
    } else if (kE4) {  // V chunk it in [0, 64), rounded to e4m3
      float x[8];
      load_bf16x8(vrow + 8 * it, x);
      *reinterpret_cast<uint2*>(a.pool + tiled_e4m3(page, off, 8 * it)) = f32x8_to_e4m3(x);
    } else if (kFolded) {  // V chunk it in [0, 64)
      *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, 8 * it)) =
          *reinterpret_cast<const uint4*>(vrow + 8 * it);
    } else if (it < 56) {  // K[128:512] chunk
      const int e = 128 + 8 * (it - 8);
      *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e)) = *reinterpret_cast<const uint4*>(krow + e);
    } else {  // V chunk
      const int e = 8 * (it - 56);
      *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, 512 + e)) =
          *reinterpret_cast<const uint4*>(vrow + e);
    }
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
