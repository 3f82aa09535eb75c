// The row arithmetic of gw_kv_append, shared by the append kernels and the
// decode kernels that append their step's rows themselves, so that both
// write the same pool bytes.
//
// A local row (one KV head) is 16 work items: item j rotates the K pairs
// (8j + i, 128 + 8j + i), i < 8, and writes V chunks 8j and 128 + 8j.  A
// global folded row is 72 items (64 V chunks, then 8 rotation items of pairs
// 8t..8t+7 and 64+8t..), a full row 120 (8 rotation items, 48 copies of
// k[128:512], 64 V chunks).  The rotation uses explicitly rounded binary32
// multiply and add (__fmul_rn / __fsub_rn / __fadd_rn): no multiply-add is
// fused, so the stored bits are those of the stated operation order.
#pragma once

#include "common.cuh"

namespace gw {

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

// Local item j of the row of KV head g at (page, off): krow, vrow are the
// head's 256 K and V values, cs the (cos, sin) entries of pairs 8j..8j+7.
template <int DT>
__device__ __forceinline__ void append_local_item(uint8_t* pool, int kv_heads, int64_t page, int off, int g,
                                                  const uint16_t* krow, const uint16_t* vrow, const CosSin8& cs,
                                                  int j) {
  float x0[8], x1[8];
  load_bf16x8(krow + 8 * j, x0);
  load_bf16x8(krow + 128 + 8 * j, x1);
  rotate8(x0, x1, cs);
  const int64_t kbase = (((page * kv_heads + g) * 2 + 0) * kPage + off) * 256;
  const int64_t vbase = (((page * kv_heads + g) * 2 + 1) * kPage + off) * 256;
  store8<DT>(pool, kbase + 8 * j, x0);
  store8<DT>(pool, kbase + 128 + 8 * j, x1);
  if constexpr (DT == GW_KV_BF16) {
    uint16_t* p = reinterpret_cast<uint16_t*>(pool);
    *reinterpret_cast<uint4*>(p + vbase + 8 * j) = *reinterpret_cast<const uint4*>(vrow + 8 * j);
    *reinterpret_cast<uint4*>(p + vbase + 128 + 8 * j) = *reinterpret_cast<const uint4*>(vrow + 128 + 8 * j);
  } else {
    float v0[8], v1[8];
    load_bf16x8(vrow + 8 * j, v0);
    load_bf16x8(vrow + 128 + 8 * j, v1);
    store8<DT>(pool, vbase + 8 * j, v0);
    store8<DT>(pool, vbase + 128 + 8 * j, v1);
  }
}

// Items of a global row.
template <int LAYOUT>
struct GlobalRow {
  static constexpr bool kE4 = LAYOUT == GW_LAYOUT_GLOBAL_FOLDED_E4M3;
  static constexpr bool kFolded = LAYOUT == GW_LAYOUT_GLOBAL_FOLDED || kE4;
  static constexpr int kRow = kFolded ? 640 : 1024;
  static constexpr int kItems = kFolded ? 72 : 120;
  // rotation item of work item `it`, or -1
  __device__ static int rot_item(int it) {
    const int r = kFolded ? it - 64 : it;
    return r >= 0 && r < 8 ? r : -1;
  }
};

// Global item `it` of the row at (page, off): krow, vrow its 512 K and V
// values, cs the (cos, sin) entries of the item's pairs (rotation items only).
template <int LAYOUT>
__device__ __forceinline__ void append_global_item(uint8_t* pool8, int64_t page, int off, const uint16_t* krow,
                                                   const uint16_t* vrow, const CosSin8& cs, int it) {
  using R = GlobalRow<LAYOUT>;
  constexpr int kRow = R::kRow;
  uint16_t* pool = reinterpret_cast<uint16_t*>(pool8);
  const int t = R::rot_item(it);
  if (t >= 0) {
    float x0[8], x1[8];
    load_bf16x8(krow + 8 * t, x0);
    load_bf16x8(krow + 64 + 8 * t, x1);
    rotate8(x0, x1, cs);
    const int e0 = R::kFolded ? 512 + 8 * t : 8 * t;
    if constexpr (R::kE4) {
      *reinterpret_cast<uint2*>(pool8 + tiled_e4m3(page, off, e0)) = f32x8_to_e4m3(x0);
      *reinterpret_cast<uint2*>(pool8 + tiled_e4m3(page, off, e0 + 64)) = f32x8_to_e4m3(x1);
    } else {
      *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e0)) = f32x8_to_bf16(x0);
      *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e0 + 64)) = f32x8_to_bf16(x1);
    }
  } else if (R::kE4) {  // V chunk it in [0, 64), rounded to e4m3
    float x[8];
    load_bf16x8(vrow + 8 * it, x);
    *reinterpret_cast<uint2*>(pool8 + tiled_e4m3(page, off, 8 * it)) = f32x8_to_e4m3(x);
  } else if (R::kFolded) {  // V chunk it in [0, 64)
    *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, 8 * it)) = *reinterpret_cast<const uint4*>(vrow + 8 * it);
  } else if (it < 56) {  // K[128:512] chunk
    const int e = 128 + 8 * (it - 8);
    *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, e)) = *reinterpret_cast<const uint4*>(krow + e);
  } else {  // V chunk
    const int e = 8 * (it - 56);
    *reinterpret_cast<uint4*>(pool + tiled<kRow>(page, off, 512 + e)) = *reinterpret_cast<const uint4*>(vrow + e);
  }
}

}  // namespace gw
