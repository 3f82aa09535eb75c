// Prompt rows of a mixed step on LOCAL layers, on the tensor cores (tcgen05).
//
// "Gemma 4" (pegainfer model page), "Scheduling": a new prompt's rows are
// computed in the same batched step as the live streams' next token;
// "Chunked walk": a prompt may continue over pages cached earlier.  Row r of
// a sequence with n > 1 query rows sits at position p = L - n + r and attends
// causally within the window: keys [max(0, p - W + 1), p].
//
// These rows are a dense contraction, so they run on UMMA with fp32
// accumulators in tensor memory:
//   * a work tile is (sequence, KV head, block of 128/G queries); its 128
//     rows are (G heads x 128/G queries), so every K/V tile feeds the whole
//     GQA group;
//   * per 64-key tile:  S[128 x 64]  = Q[128 x 256] . K^T      (M=128, N=64)
//                       O[128 x 256] += P[128 x 64] . V         (M=128, N=256)
//     S (two buffers) and O live in TMEM; TMEM lane i is row i, so each
//     softmax thread owns one row and needs no cross-thread reduction;
//   * softmax is base 2 with a lazily raised reference max per row (O is
//     rescaled only when a logit exceeds it by more than 8); P is rounded to
//     bf16 and l sums the rounded weights;
//   * K and V tiles arrive by TMA (cp.async.bulk.tensor): one 2 KB copy per
//     (page, 64-dim chunk) lands 16 key rows x 128 B in the 128-byte-swizzled
//     UMMA layout, so a 64-key tile is 16 copies for K and 16 for V, issued
//     together by 16 lanes of a producer warp.  K feeds Q.K^T as a K-major
//     operand, V feeds P.V as an MN-major operand, three stages each.
//   * Q and P never touch shared memory: the softmax threads write their Q
//     rows (once per work tile) and their bf16 P rows (over the S columns
//     just read) into tensor memory, and both contractions take A from there.
//     TMEM: S at columns 0 and 64 (P over their first 32), Q at 128..255,
//     O at 256..511.
//     V rows of keys outside the tile's range are cleared before P.V (0 *
//     anything must stay 0), K rows of pages not loaded before Q.K^T.
// Warp roles (256 threads, persistent CTAs):
//   warps 0-3  load Q rows, softmax, epilogue (warp w owns TMEM lanes 32w..)
//   warps 4, 6 TMA producers of K and of V tiles (16 lanes issue a tile's copies)
//   warp 5     Q.K^T issue (elect.sync) and TMEM owner
//   warp 7     P.V issue, so that neither contraction's issue waits on the other
// Every wait is bounded; a timeout raises GW_DEV_TIMEOUT and the CTA stops.
#include "tcgen05.cuh"
#include "tma.cuh"
namespace gw {
namespace {

constexpr int kTM = 128;              // rows per work tile (UMMA M)
constexpr int kTN = 64;               // keys per key tile (UMMA N of S)
constexpr int kTcThreads = 256;
constexpr float kTcLazy = 8.f;
// TMEM columns: S buffers at 0 and 64, Q at 128..255, O at 256..511
constexpr uint32_t kColS = 0, kColQ = 128, kColO = 256;
constexpr uint32_t kPlane = kTN * 128;  // one 128-byte chunk column of a K/V tile: 64 rows x 128 B
constexpr int kKS = 3, kVS = 3;         // K and V stages

// 128-byte chunks per 256-element row: 4 of 64 bf16, 2 of 128 e4m3
template <int DT>
constexpr int chunks_of() { return DT == GW_KV_BF16 ? 4 : 2; }

template <int DT>
struct TcSmem {
  static constexpr int kC = chunks_of<DT>();
  uint8_t k[kKS][kC * kPlane];    // [chunk][64 keys][128 B], 128-byte swizzled
  uint8_t v[kVS][kC * kPlane];    // same layout
  uint64_t kfull[kKS], kempty[kKS], vfull[kVS], vempty[kVS];
  uint64_t s_ready[2], p_ready[2], pfree[2];
  uint64_t q_full, q_free, o_done, o_free;
  int32_t kmask[kKS], vmask[kVS];  // pages of the K / V tile that were loaded (bits 0-3)
  uint32_t tmem_base;
};

__device__ __forceinline__ void zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0) : "memory");
}

// Zero key rows of a K/V stage (every 16-byte unit of the row's chunks);
// `want(r)` selects rows r in [0, 64).  The warp's lanes share the units.
template <int DT, class Want>
__device__ __forceinline__ void zero_rows(uint32_t base, int lane, Want want) {
  constexpr int kU = chunks_of<DT>() * 8;  // 16-byte units per row
  for (int idx = lane; idx < kTN * kU; idx += 32) {
    const int r = idx / kU, u = idx % kU;
    if (want(r)) zero16(base + (u >> 3) * kPlane + r * 128 + (u & 7) * 16);
  }
}

// q (or a weight) x as two e4m3 terms: hi = e4m3(x), lo = e4m3(x - hi); the
// pair (x0, x1) gives one 16-bit word of each (x0 in the low byte).  With
// `sum`, the value hi + lo the contraction will use.
__device__ __forceinline__ void split_e4m3(float x0, float x1, uint32_t& hi, uint32_t& lo, float2* sum = nullptr) {
  const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
  const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
  const __nv_fp8x2_storage_t l2 =
      __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
  hi = h2;
  lo = l2;
  if (sum) {
    const float2 lf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(l2, __NV_E4M3)));
    *sum = make_float2(hf.x + lf.x, hf.y + lf.y);
  }
}


__device__ __forceinline__ int prompt_seq(const int32_t* base, int batch, int t) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct WorkTile {
  int s, g, q0, nq, P0, lo, hi, t_lo, t_hi, row0;
};

template <int G>
__device__ __forceinline__ WorkTile work_tile(const LocalArgs& a, int tile) {
  constexpr int BQ = kTM / G;
  WorkTile w;
  w.s = prompt_seq(a.prompt_base, a.batch, tile);
  const int n = a.cu_q_rows[w.s + 1] - a.cu_q_rows[w.s];
  const int nqb = (n + BQ - 1) / BQ;
  const int r0 = tile - a.prompt_base[w.s];
  w.g = r0 / nqb;
  const int qb = r0 % nqb;
  const int L = a.seq_lens[w.s];
  w.P0 = L - n;
  w.q0 = qb * BQ;
  w.nq = min(BQ, n - w.q0);
  w.lo = max(0, w.P0 + w.q0 - a.window + 1);
  w.hi = w.P0 + w.q0 + w.nq - 1;
  w.t_lo = w.lo / kTN;
  w.t_hi = w.hi / kTN;
  w.row0 = a.cu_q_rows[w.s];
  return w;
}

template <int DT, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    local_prompt_tc_kernel(const LocalArgs a, const __grid_constant__ CUtensorMap kv_map) {
  constexpr int BQ = kTM / G;
  constexpr bool kE4 = DT == GW_KV_E4M3;
  constexpr int kC = chunks_of<DT>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  TcSmem<DT>& sm = *reinterpret_cast<TcSmem<DT>*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  int32_t* st = a.status;

  if (tid == 0) {
    for (int b = 0; b < kKS; ++b) {
      mbar_init(&sm.kfull[b], 1);
      mbar_init(&sm.kempty[b], 1);
    }
    for (int b = 0; b < kVS; ++b) {
      mbar_init(&sm.vfull[b], 1);
      mbar_init(&sm.vempty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], kTM);
      mbar_init(&sm.pfree[b], 1);
    }
    mbar_init(&sm.q_full, kTM);
    mbar_init(&sm.q_free, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, kTM);
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  const int total = a.prompt_base[a.batch];
  if (warp == 5) {
    tc::alloc(&sm.tmem_base, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4 || warp == 6) {
    // ------------------------------------------------------ TMA producers
    // warp 4 loads K tiles, warp 6 V tiles; lane l < 4 kC issues the copy of
    // page l / kC, 128-byte chunk l % kC (a tile's copies go out together)
    const bool is_v = warp == 6;
    // every K/V tile is read again by the neighbouring query blocks (a window
    // of W keys is shared by W / 64 of them): keep it in L2 (evict last)
    const uint64_t pol = policy_evict_last();
    const int j = lane / kC, c = lane % kC;
    uint32_t gi = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const WorkTile w = work_tile<G>(a, tile);
      const int32_t* bt = a.block_table + static_cast<int64_t>(w.s) * a.max_pages;
      for (int t = w.t_lo; t <= w.t_hi; ++t, ++gi) {
        const int ns = is_v ? kVS : kKS;
        const int b = static_cast<int>(gi % ns);
        const uint32_t ph = gi / ns;  // use of this stage
        // page j of the tile: loaded if it overlaps [lo, hi] and is valid
        int32_t row = -1;
        if (lane < 4 * kC) {
          const int k0 = t * kTN + j * kPage;
          if (k0 + kPage - 1 >= w.lo && k0 <= w.hi) {
            const int32_t pg = bt[k0 / kPage];
            if (pg >= 0 && pg < a.num_pages) {
              row = (pg * a.kv_heads + w.g) * 2 * kPage + (is_v ? kPage : 0);
            } else if (c == 0) {
              set_status(st, GW_DEV_PAGE_RANGE);
            }
          }
        }
        const uint32_t loaded = __ballot_sync(0xffffffffu, row >= 0 && c == 0);  // bit kC j: page j
        int mask = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) mask |= ((loaded >> (kC * q)) & 1) << q;
        uint64_t* full = is_v ? &sm.vfull[b] : &sm.kfull[b];
        uint64_t* empty = is_v ? &sm.vempty[b] : &sm.kempty[b];
        if (ph >= 1 && !__all_sync(0xffffffffu, mbar_wait(empty, (ph - 1) & 1, st))) { ok = false; break; }
        if (lane == 0) {
          if (is_v) sm.vmask[b] = mask; else sm.kmask[b] = mask;
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(mask)) * kC * 2048);
        }
        __syncwarp();
        if (row >= 0)
          tma_rows(smem_u32(is_v ? sm.v[b] : sm.k[b]) + c * kPlane + j * 2048, &kv_map, c, row, full, pol);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------- Q.K^T issue
    const uint32_t id_s = kE4 ? tc::idesc_e4m3(kTM, kTN, false, false) : tc::idesc_bf16(kTM, kTN, false, false);
    uint32_t gi = 0;
    int wt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++wt) {
      const WorkTile w = work_tile<G>(a, tile);
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_full, wt & 1, st))) break;
      const int nt = w.t_hi - w.t_lo + 1;
      for (int j = 0; j < nt; ++j, ++gi) {
        const int b = static_cast<int>(gi % kKS), sb = gi & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.kfull[b], (gi / kKS) & 1, st))) { ok = false; break; }
        // this S buffer holds P of tile gi - 2 until its P.V is done
        if (gi >= 2 && !__all_sync(0xffffffffu, mbar_wait(&sm.pfree[sb], ((gi >> 1) - 1) & 1, st))) {
          ok = false;
          break;
        }
        const uint32_t ka = smem_u32(sm.k[b]);
        const int kmask = sm.kmask[b];
        if (kmask != 0xF) {
          // pages not loaded (outside the range or invalid): finite zeros, so no
          // stale bytes can turn into NaN logits
          zero_rows<DT>(ka, lane, [&](int r) { return ((kmask >> (r / kPage)) & 1) == 0; });
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc::fence_after();
        // a K-step is 32 bytes of each key row: 16 bf16 or 32 e4m3 dims
#pragma unroll
        for (int ks = 0; ks < 16 / (kE4 ? 2 : 1); ++ks) {
          const uint64_t bd = tc::smem_desc_sw128(ka + (ks >> 2) * kPlane + (ks & 3) * 32, 16);
          if constexpr (kE4) {
            // S = (q_hi + q_lo) . K^T: q_hi at Q columns 0..63, q_lo at 64..127
            tc::mma_e4m3_ts_warp(tmem + kColS + 64 * sb, tmem + kColQ + 8 * ks, bd, id_s, ks > 0);
            tc::mma_e4m3_ts_warp(tmem + kColS + 64 * sb, tmem + kColQ + 64 + 8 * ks, bd, id_s, true);
          } else {
            tc::mma_bf16_ts_warp(tmem + kColS + 64 * sb, tmem + kColQ + 8 * ks, bd, id_s, ks > 0);
          }
        }
        tc::commit_warp(&sm.kempty[b]);
        tc::commit_warp(&sm.s_ready[sb]);
        if (j == nt - 1) tc::commit_warp(&sm.q_free);
      }
    }
  } else if (warp == 7) {
    // ------------------------------------------------------- P.V issue
    const uint32_t id_o = kE4 ? tc::idesc_e4m3(kTM, 256, false, true) : tc::idesc_bf16(kTM, 256, false, true);
    uint32_t gi = 0;
    int wt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++wt) {
      const WorkTile w = work_tile<G>(a, tile);
      const int nt = w.t_hi - w.t_lo + 1;
      for (int j = 0; j < nt; ++j, ++gi) {
        const int b = static_cast<int>(gi % kVS), sb = gi & 1;
        if (j == 0 && wt >= 1 && !__all_sync(0xffffffffu, mbar_wait(&sm.o_free, (wt - 1) & 1, st))) {
          ok = false;
          break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.vfull[b], (gi / kVS) & 1, st))) { ok = false; break; }
        // V rows of keys outside [lo, hi] or of pages not loaded: clear them
        const int key0 = (w.t_lo + j) * kTN;
        const int mask = sm.vmask[b];
        if (mask != 0xF || key0 < w.lo || key0 + kTN - 1 > w.hi) {
          zero_rows<DT>(smem_u32(sm.v[b]), lane, [&](int kr) {
            const int key = key0 + kr;
            return !(((mask >> (kr >> 4)) & 1) && key >= w.lo && key <= w.hi);
          });
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_ready[sb], (gi >> 1) & 1, st))) { ok = false; break; }
        tc::fence_after();
        const uint32_t va = smem_u32(sm.v[b]);
        if constexpr (kE4) {
          // K-steps of 32 keys (4 swizzle atoms of 8 rows); O += (P_hi + P_lo) . V,
          // P_hi at S columns 0..15, P_lo at 16..31
#pragma unroll
          for (int kk = 0; kk < kTN / 32; ++kk) {
            const uint64_t bd = tc::smem_desc_sw128(va + kk * 4096, kPlane);
            tc::mma_e4m3_ts_warp(tmem + kColO, tmem + kColS + 64 * sb + 8 * kk, bd, id_o, !(j == 0 && kk == 0));
            tc::mma_e4m3_ts_warp(tmem + kColO, tmem + kColS + 64 * sb + 16 + 8 * kk, bd, id_o, true);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kTN / 16; ++kk)
            tc::mma_bf16_ts_warp(tmem + kColO, tmem + kColS + 64 * sb + 8 * kk, tc::smem_desc_sw128(va + kk * 2048, kPlane),
                                 id_o, !(j == 0 && kk == 0));
        }
        tc::commit_warp(&sm.vempty[b]);
        tc::commit_warp(&sm.pfree[sb]);
        if (j == nt - 1) tc::commit_warp(&sm.o_done);
      }
    }
  } else {
    // ---------------------------------------- Q rows, softmax, epilogue
    const int r = tid;  // row of the work tile = TMEM lane
    const int hh = r / BQ, qi = r % BQ;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    // Q row of a work tile -> tensor memory (128 columns of bf16 pairs), then
    // signal the MMA warp; rows past the prompt are zeros
    // e4m3 pools: the row is scaled by an exact power of two 2^e that puts its
    // largest |q| in [128, 256) and split into two e4m3 terms; sc_q = 2^-e
    // scales the logits back (1 for bf16 pools)
    float sc_q = 1.f;
    auto load_q = [&](const WorkTile& w) {
      const bool ok_row = qi < w.nq;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + (static_cast<int64_t>(w.row0 + w.q0 + (ok_row ? qi : 0)) * a.num_q_heads + w.g * G + hh) * 256);
      if constexpr (kE4) {
        // pass 1: the row's largest |q|; pass 2 reads the row again (from L1)
        // a quarter at a time
        float mq = 0.f;
#pragma unroll 8
        for (int c = 0; c < 32; ++c) {
          const uint4 x = ok_row ? src[c] : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t u4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            mq = fmaxf(mq, fmaxf(fabsf(__uint_as_float(u4[i] << 16)), fabsf(__uint_as_float(u4[i] & 0xFFFF0000u))));
        }
        const int ex = mq > 0.f ? static_cast<int>((__float_as_uint(mq) >> 23) & 0xFF) - 127 : 7;
        const int e = min(125, max(-125, 7 - ex));
        const float up = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        sc_q = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        // 4 dims per 32-bit column: q_hi at columns 0..63, q_lo at 64..127,
        // a quarter (64 dims: 16 columns of each) at a time
#pragma unroll 1
        for (int qtr = 0; qtr < 4; ++qtr) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 x = ok_row ? src[8 * qtr + c8] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t u4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
              const uint32_t w0 = u4[2 * hv], w1 = u4[2 * hv + 1];
              uint32_t h0, l0, h1, l1;
              split_e4m3(__uint_as_float(w0 << 16) * up, __uint_as_float(w0 & 0xFFFF0000u) * up, h0, l0);
              split_e4m3(__uint_as_float(w1 << 16) * up, __uint_as_float(w1 & 0xFFFF0000u) * up, h1, l1);
              hi[2 * c8 + hv] = h0 | (h1 << 16);
              lo[2 * c8 + hv] = l0 | (l1 << 16);
            }
          }
          tc::st16(tmem + lane_base + kColQ + 16 * qtr, hi);
          tc::st16(tmem + lane_base + kColQ + 64 + 16 * qtr, lo);
        }
      } else {
        uint32_t qv[128];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint4 x = ok_row ? src[c] : make_uint4(0u, 0u, 0u, 0u);
          qv[4 * c] = x.x;
          qv[4 * c + 1] = x.y;
          qv[4 * c + 2] = x.z;
          qv[4 * c + 3] = x.w;
        }
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
          tc::st32(tmem + lane_base + kColQ + 32 * blk, *reinterpret_cast<uint32_t(*)[32]>(&qv[32 * blk]));
      }
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(&sm.q_full);
    };
    uint32_t gi = 0;
    int wt = 0;
    if (static_cast<int>(blockIdx.x) < total) load_q(work_tile<G>(a, blockIdx.x));
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++wt) {
      const WorkTile w = work_tile<G>(a, tile);
      const bool row_ok = qi < w.nq;
      const int pos = w.P0 + w.q0 + qi;
      // this row's keys: [kmin, kmax] (empty for rows past the prompt)
      const int kmin = max(w.lo, pos - a.window + 1), kmax = row_ok ? pos : -1;
      float m_ref = -INFINITY;            // reference max, scaled log2 units
      float lp[4] = {0.f, 0.f, 0.f, 0.f};  // partial sums of the rounded weights
      const int nt = w.t_hi - w.t_lo + 1;
      bool ok = true;
      for (int j = 0; j < nt; ++j, ++gi) {
        const int b = gi & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_ready[b], (gi >> 1) & 1, st))) { ok = false; break; }
        tc::fence_after();
        uint32_t sv[64];
        tc::ld32(tmem + lane_base + kColS + 64 * b, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tc::ld32(tmem + lane_base + kColS + 64 * b + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tc::wait_ld();
        const int key0 = (w.t_lo + j) * kTN;
        if (!(key0 >= kmin && key0 + kTN - 1 <= kmax)) {
          // edge tile for this row: keys outside [kmin, kmax] get -inf
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (key0 + c < kmin || key0 + c > kmax) sv[c] = __float_as_uint(-INFINITY);
        }
        float mg[8];
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const float* x = reinterpret_cast<const float*>(&sv[g8 * 8]);
          mg[g8] = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
        }
        const float mraw = fmaxf(fmaxf(fmaxf(mg[0], mg[1]), fmaxf(mg[2], mg[3])), fmaxf(fmaxf(mg[4], mg[5]), fmaxf(mg[6], mg[7])));
        const float sc = a.scale_log2 * sc_q;  // sc_q: the row's q descale (e4m3 pools)
        const float mx = mraw * sc;            // -inf stays -inf (scale > 0)
        const bool raise = mx > m_ref + kTcLazy;  // false while the row has no key
        if (__any_sync(0xffffffffu, raise)) {
          const float m_new = raise ? mx : m_ref;
          const float alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new);
          if (__any_sync(0xffffffffu, raise && m_ref != -INFINITY)) {
            // O *= alpha for this warp's rows once P.V of the previous tile is done
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.pfree[(gi - 1) & 1], ((gi - 1) >> 1) & 1, st))) {
              ok = false;
              break;
            }
            tc::fence_after();
#pragma unroll 1
            for (int blk = 0; blk < 8; ++blk) {
              uint32_t o[32];
              const uint32_t ad = tmem + lane_base + kColO + 32 * blk;
              tc::ld32(ad, o);
              tc::wait_ld();
              if (raise && m_ref != -INFINITY) {
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              }
              tc::st32(ad, o);
            }
            tc::wait_st();
          }
          if (raise) {
#pragma unroll
            for (int i = 0; i < 4; ++i) lp[i] *= alpha;
            m_ref = m_new;
          }
        }
        // ---- P row (bf16 pairs) over the S columns just read: s_ready of this
        // tile means every earlier MMA, P.V two tiles back included, is done.
        // p = 2^(s * scale - m): masked keys (s = -inf) give 0; a row with no
        // key yet uses m = 0 so that no inf - inf arises
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        uint32_t pw[32];
        if constexpr (kE4) {
          // P = P_hi + P_lo, two e4m3 terms (p <= 2^8 under the lazy max), 4
          // keys per column: P_hi at columns 0..15, P_lo at 16..31
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            uint32_t h[2], l[2];
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
              const float p0 = ex2(fmaf(__uint_as_float(sv[4 * u + 2 * hv]), sc, neg_m));
              const float p1 = ex2(fmaf(__uint_as_float(sv[4 * u + 2 * hv + 1]), sc, neg_m));
              float2 used;
              split_e4m3(p0, p1, h[hv], l[hv], &used);
              lp[u & 3] += used.x + used.y;
            }
            pw[u] = h[0] | (h[1] << 16);
            pw[16 + u] = l[0] | (l[1] << 16);
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float p0 = ex2(fmaf(__uint_as_float(sv[2 * u]), sc, neg_m));
            const float p1 = ex2(fmaf(__uint_as_float(sv[2 * u + 1]), sc, neg_m));
            __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            lp[u & 3] += __low2float(pb) + __high2float(pb);
            pw[u] = *reinterpret_cast<uint32_t*>(&pb);
          }
        }
        tc::st32(tmem + lane_base + kColS + 64 * b, pw);
        tc::wait_st();
        tc::fence_before();
        mbar_arrive(&sm.p_ready[b]);
      }
      if (!ok) break;
      // ---- next work tile's Q: the last QK^T of this one is done (its S was
      // read above); the next work tile's first QK^T then overlaps this epilogue
      const int next = tile + gridDim.x;
      if (next < total) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_free, wt & 1, st))) break;
        tc::fence_after();
        load_q(work_tile<G>(a, next));
      }
      // ---- epilogue: O / l -> bf16
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_done, wt & 1, st))) break;
      tc::fence_after();
      const float l = (lp[0] + lp[1]) + (lp[2] + lp[3]);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* dst = a.out + (static_cast<int64_t>(w.row0 + w.q0 + qi) * a.num_q_heads + w.g * G + hh) * 256;
#pragma unroll 1
      for (int blk = 0; blk < 8; blk += 2) {
        uint32_t o[64];
        tc::ld32(tmem + lane_base + kColO + 32 * blk, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tc::ld32(tmem + lane_base + kColO + 32 * blk + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tc::wait_ld();
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[c + 2 * e]) * inv,
                                                        __uint_as_float(o[c + 2 * e + 1]) * inv);
              pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(dst + blk * 32 + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      tc::fence_before();
      mbar_arrive(&sm.o_free);
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
}

template <int DT, int G>
cudaError_t launch_g(const LocalArgs& a, cudaStream_t st) {
  CUtensorMap map;
  cudaError_t e = make_local_kv_map(a, &map, DT);
  if (e != cudaSuccess) return e;
  auto kern = local_prompt_tc_kernel<DT, G>;
  const size_t smem = sizeof(TcSmem<DT>);
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid_ctas()), dim3(kTcThreads), smem, st, a, map);
}


template <int DT>
cudaError_t launch_dt(int group, const LocalArgs& a, cudaStream_t st) {
  switch (group) {
    case 1: return launch_g<DT, 1>(a, st);
    case 2: return launch_g<DT, 2>(a, st);
    case 4: return launch_g<DT, 4>(a, st);
    case 8: return launch_g<DT, 8>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_local_prompt_tc(int dtype, int group, const LocalArgs& a, cudaStream_t st) {
  return dtype == GW_KV_E4M3 ? launch_dt<GW_KV_E4M3>(group, a, st) : launch_dt<GW_KV_BF16>(group, a, st);
}

}  // namespace gw
