// Prompt rows of a mixed step on GLOBAL layers, on the tensor cores (tcgen05).
//
// "Gemma 4" (pegainfer model page), "Scheduling" and "Chunked walk": a
// prompt's rows run in the same step as the live streams; row r of a
// sequence with n > 1 rows sits at position p = L - n + r and attends to
// keys [0, p] of the single KV head (head dim 512).  "Gewell - Gemma4
// inference engine", "the Why": on a FOLDED pool K = k_rot || V[128:512] is
// read from the same page tile as V.
//
// All q heads share the KV head, so a work tile's 128 rows are (128/HQ
// queries) x (HQ heads).  O[128 x 512] in fp32 would fill all 512 TMEM
// columns by itself, so a work tile is split in two by output dims: the two
// halves run as separate work tiles, each computing the full
//   S[128 x N]    = Q[128 x 512] . K^T       (UMMA M=128, N = keys per tile)
// and its half of
//   O[128 x 256] += P[128 x N] . V[:, half]  (UMMA M=128, N=256, A = P in TMEM)
// (the logits are computed twice; the alternative, one CTA per block with
// all of O, does not fit).  TMEM: S at columns 0 and N (P over their first
// N/2), Q dims [0, 256) at 128..255, the O half at 256..511; Q dims
// [256, 512) sit in shared memory, so the K-steps of Q.K^T take A from TMEM
// for the first 16 and from shared memory for the other 16.
//
// Key tiles are whole pages (4 folded pages = 64 keys, or 2 full pages = 32
// keys) brought by cp.async.bulk into a 2-stage ring.  A page is already laid
// out as 8 x 8 UMMA core matrices: it is the K-major B operand of Q.K^T (K
// dims from the k_rot and V column blocks) and the MN-major B operand of P.V
// (this half's V column blocks).  Rows are owned by softmax threads (TMEM
// lane = row): causal mask, lazily raised reference max (rescale of O only
// when a logit exceeds it by more than 8), P rounded to bf16 and written over
// the S columns just read; l sums the rounded weights.  V rows of tokens past
// the last query position (and whole pages that were not loaded) are cleared
// before P.V.
// Warp roles (224 threads): warps 0-3 Q rows / softmax / epilogue, warp 4
// page producer (one thread), warp 5 issues Q.K^T (and owns TMEM), warp 6
// issues P.V, so neither contraction's issue time holds up the other (32
// Q.K^T MMAs per tile take longer to issue than the softmax takes).  Every
// wait is bounded; a timeout raises GW_DEV_TIMEOUT.
#include "tcgen05.cuh"

namespace gw {
namespace {

constexpr int kGM = 128;
constexpr int kGThreads = 224;
constexpr float kGLazy = 8.f;
constexpr uint32_t kGColS = 0, kGColQ = 128, kGColO = 256;

template <int LAYOUT>
struct GPL;
template <>
struct GPL<GW_LAYOUT_GLOBAL_FOLDED> {
  static constexpr int kPageBytes = 20480;
  static constexpr int kBlk = 80;   // 8-column blocks per 8-token block
  static constexpr int kVcb = 0;    // column block of V dim 0
  static constexpr int kPages = 4;  // pages per key tile
  __device__ static int k_cb(int ks) { return ks < 8 ? 64 + 2 * ks : 2 * ks; }
};
template <>
struct GPL<GW_LAYOUT_GLOBAL_FULL> {
  static constexpr int kPageBytes = 32768;
  static constexpr int kBlk = 128;
  static constexpr int kVcb = 64;
  static constexpr int kPages = 2;
  __device__ static int k_cb(int ks) { return 2 * ks; }
};

template <int LAYOUT>
struct GPSmem {
  using T = GPL<LAYOUT>;
  uint8_t tiles[2][T::kPages * T::kPageBytes];
  uint8_t q[kGM * 512];  // Q dims [256, 512): [row block 16][dim block 32][8][16 B]
  uint64_t full[2], empty[2], s_ready[2], p_ready[2], pfree[2];
  uint64_t q_full, q_free, o_done, o_free;
  int32_t mask[2];  // pages of the tile that were loaded
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t cm_off(int r, int c, int chunks) {
  return static_cast<uint32_t>(((r >> 3) * chunks + c) * 128 + (r & 7) * 16);
}
__device__ __forceinline__ void zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0) : "memory");
}

__device__ __forceinline__ int gp_seq(const int32_t* base, int batch, int t) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct GWork {
  int s, half, q0, nq, P0, pmax, nt, row0;
};

template <int HQ, int KN>
__device__ __forceinline__ GWork g_work(const LocalArgs& a, int tile) {
  constexpr int QB = kGM / HQ;  // queries per work tile
  GWork w;
  w.s = gp_seq(a.prompt_base, a.batch, tile);
  const int n = a.cu_q_rows[w.s + 1] - a.cu_q_rows[w.s];
  const int nqb = (n + QB - 1) / QB;
  const int r0 = tile - a.prompt_base[w.s];
  w.half = r0 / nqb;
  const int qb = r0 % nqb;
  const int L = a.seq_lens[w.s];
  w.P0 = L - n;
  w.q0 = qb * QB;
  w.nq = min(QB, n - w.q0);
  w.pmax = w.P0 + w.q0 + w.nq - 1;
  w.nt = w.pmax / KN + 1;
  w.row0 = a.cu_q_rows[w.s];
  return w;
}

template <int LAYOUT, int HQ>
__global__ void __launch_bounds__(kGThreads, 1) global_prompt_tc_kernel(const LocalArgs a) {
  using T = GPL<LAYOUT>;
  using SM = GPSmem<LAYOUT>;
  constexpr int KN = T::kPages * kPage;  // keys per tile (UMMA N of S)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  int32_t* st = a.status;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], 1);
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], kGM);
      mbar_init(&sm.pfree[b], 1);
    }
    mbar_init(&sm.q_full, kGM);
    mbar_init(&sm.q_free, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, kGM);
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

  if (warp == 4) {
    // ------------------------------------------------------ page producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // every later query block re-reads these pages
      uint32_t gi = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const GWork w = g_work<HQ, KN>(a, tile);
        const int32_t* bt = a.block_table + static_cast<int64_t>(w.s) * a.max_pages;
        for (int t = 0; t < w.nt; ++t, ++gi) {
          const int b = gi & 1;
          int32_t pg[T::kPages];
          int mask = 0;
#pragma unroll
          for (int j = 0; j < T::kPages; ++j) {
            const int k0 = (t * T::kPages + j) * kPage;
            pg[j] = -1;
            if (k0 <= w.pmax) {
              const int32_t p = bt[k0 / kPage];
              if (p >= 0 && p < a.num_pages) {
                pg[j] = p;
                mask |= 1 << j;
              } else {
                set_status(st, GW_DEV_PAGE_RANGE);
              }
            }
          }
          if (gi >= 2 && !mbar_wait(&sm.empty[b], ((gi >> 1) - 1) & 1, st)) { ok = false; break; }
          sm.mask[b] = mask;
          mbar_arrive_expect_tx(&sm.full[b], static_cast<uint32_t>(__popc(mask)) * T::kPageBytes);
#pragma unroll
          for (int j = 0; j < T::kPages; ++j)
            if (pg[j] >= 0)
              bulk_g2s(sm.tiles[b] + j * T::kPageBytes, a.pool + static_cast<int64_t>(pg[j]) * T::kPageBytes,
                       T::kPageBytes, &sm.full[b], pol);
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------- Q.K^T issue
    const uint32_t id_s = tc::idesc_bf16(kGM, KN, false, false);
    // Q dims [256, 512): no-swizzle K-major, LBO = 128, SBO = 4096
    const uint64_t dq = tc::smem_desc(smem_u32(sm.q), 128, 4096);
    uint32_t i = 0;
    int wt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++wt) {
      const GWork w = g_work<HQ, KN>(a, tile);
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_full, wt & 1, st))) break;
      for (int j = 0; j < w.nt; ++j, ++i) {
        const int b = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.full[b], (i >> 1) & 1, st))) { ok = false; break; }
        // this S buffer holds P of tile i - 2 until its P.V is done
        if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(&sm.pfree[b], ((i >> 1) - 1) & 1, st))) {
          ok = false;
          break;
        }
        // pages not loaded (past the last query or invalid): finite zeros
        const uint32_t ta = smem_u32(sm.tiles[b]);
        const int mask = sm.mask[b];
        if (mask != (1 << T::kPages) - 1) {
          for (int pgi = 0; pgi < T::kPages; ++pgi) {
            if ((mask >> pgi) & 1) continue;
            for (int o = lane * 16; o < T::kPageBytes; o += 32 * 16) zero16(ta + pgi * T::kPageBytes + o);
          }
        }
        // V rows of tokens past the last query position (unwritten bytes)
        const int key0 = j * KN;
        if (key0 + KN - 1 > w.pmax) {
          for (int k = max(w.pmax + 1 - key0, 0); k < KN; ++k) {
            const int tbk = k >> 3;  // token block of the tile
            for (int cb = lane; cb < 64; cb += 32) zero16(ta + (tbk * T::kBlk + T::kVcb + cb) * 128 + (k & 7) * 16);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        tc::fence_after();
        const uint64_t dk = tc::smem_desc(ta, 128, T::kBlk * 128);
#pragma unroll
        for (int ks = 0; ks < 32; ++ks) {
          const uint64_t bd = dk + ((T::k_cb(ks) * 128) >> 4);
          if (ks < 16)
            tc::mma_bf16_ts_warp(tmem + kGColS + KN * b, tmem + kGColQ + 8 * ks, bd, id_s, ks > 0);
          else
            tc::mma_bf16_warp(tmem + kGColS + KN * b, dq + (((ks - 16) * 256) >> 4), bd, id_s, true);
        }
        tc::commit_warp(&sm.s_ready[b]);
        if (j == w.nt - 1) tc::commit_warp(&sm.q_free);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------- P.V issue
    const uint32_t id_o = tc::idesc_bf16(kGM, 256, false, true);
    uint32_t i = 0;
    int wt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++wt) {
      const GWork w = g_work<HQ, KN>(a, tile);
      for (int j = 0; j < w.nt; ++j, ++i) {
        const int b = i & 1;
        if (j == 0 && wt >= 1 && !__all_sync(0xffffffffu, mbar_wait(&sm.o_free, (wt - 1) & 1, st))) {
          ok = false;
          break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_ready[b], (i >> 1) & 1, st))) { ok = false; break; }
        tc::fence_after();
        const uint32_t ta = smem_u32(sm.tiles[b]);
        const uint64_t dv = tc::smem_desc(ta + (T::kVcb + 32 * w.half) * 128, T::kBlk * 128, 128);
#pragma unroll
        for (int kk = 0; kk < KN / 16; ++kk)
          tc::mma_bf16_ts_warp(tmem + kGColO, tmem + kGColS + KN * b + 8 * kk,
                               dv + ((kk * 2 * T::kBlk * 128) >> 4), id_o, !(j == 0 && kk == 0));
        tc::commit_warp(&sm.empty[b]);
        tc::commit_warp(&sm.pfree[b]);
        if (j == w.nt - 1) tc::commit_warp(&sm.o_done);
      }
    }
  } else {
    // ---------------------------------------- Q rows, softmax, epilogue
    const int r = tid;
    const int qi = r / HQ, hd = r % HQ;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t qs = smem_u32(sm.q);
    auto load_q = [&](const GWork& w) {
      const bool ok_row = qi < w.nq;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + (static_cast<int64_t>(w.row0 + w.q0 + (ok_row ? qi : 0)) * HQ + hd) * 512);
      uint32_t qv[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {  // dims [0, 256) -> TMEM
        const uint4 x = ok_row ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        qv[4 * c] = x.x;
        qv[4 * c + 1] = x.y;
        qv[4 * c + 2] = x.z;
        qv[4 * c + 3] = x.w;
      }
#pragma unroll
      for (int blk = 0; blk < 4; ++blk)
        tc::st32(tmem + lane_base + kGColQ + 32 * blk, *reinterpret_cast<uint32_t(*)[32]>(&qv[32 * blk]));
#pragma unroll 8
      for (int c = 0; c < 32; ++c) {  // dims [256, 512) -> shared memory
        const uint4 x = ok_row ? src[32 + c] : make_uint4(0u, 0u, 0u, 0u);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qs + cm_off(r, c, 32)), "r"(x.x), "r"(x.y),
                     "r"(x.z), "r"(x.w)
                     : "memory");
      }
      tc::wait_st();
      fence_proxy_async_smem();
      tc::fence_before();
      mbar_arrive(&sm.q_full);
    };
    uint32_t gi = 0;
    int wt = 0;
    if (static_cast<int>(blockIdx.x) < total) load_q(g_work<HQ, KN>(a, blockIdx.x));
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++wt) {
      const GWork w = g_work<HQ, KN>(a, tile);
      const bool row_ok = qi < w.nq;
      const int kmax = row_ok ? w.P0 + w.q0 + qi : -1;  // this row's keys: [0, kmax]
      float m_ref = -INFINITY;
      float lp[4] = {0.f, 0.f, 0.f, 0.f};
      bool ok = true;
      for (int j = 0; j < w.nt; ++j, ++gi) {
        const int b = gi & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_ready[b], (gi >> 1) & 1, st))) { ok = false; break; }
        tc::fence_after();
        uint32_t sv[KN];
#pragma unroll
        for (int c0 = 0; c0 < KN; c0 += 32)
          tc::ld32(tmem + lane_base + kGColS + KN * b + c0, *reinterpret_cast<uint32_t(*)[32]>(&sv[c0]));
        tc::wait_ld();
        const int key0 = j * KN;
        if (key0 + KN - 1 > kmax) {
#pragma unroll
          for (int c = 0; c < KN; ++c)
            if (key0 + c > kmax) sv[c] = __float_as_uint(-INFINITY);
        }
        float mg[KN / 8];
#pragma unroll
        for (int g8 = 0; g8 < KN / 8; ++g8) {
          const float* x = reinterpret_cast<const float*>(&sv[g8 * 8]);
          mg[g8] = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
        }
        float mraw = mg[0];
#pragma unroll
        for (int g8 = 1; g8 < KN / 8; ++g8) mraw = fmaxf(mraw, mg[g8]);
        const float mx = mraw * a.scale_log2;
        const bool raise = mx > m_ref + kGLazy;
        if (__any_sync(0xffffffffu, raise)) {
          const float m_new = raise ? mx : m_ref;
          const float alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new);
          if (__any_sync(0xffffffffu, raise && m_ref != -INFINITY)) {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.pfree[(gi - 1) & 1], ((gi - 1) >> 1) & 1, st))) {
              ok = false;
              break;
            }
            tc::fence_after();
#pragma unroll 1
            for (int blk = 0; blk < 8; ++blk) {
              uint32_t o[32];
              const uint32_t ad = tmem + lane_base + kGColO + 32 * blk;
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
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        uint32_t pw[KN / 2];
#pragma unroll
        for (int u = 0; u < KN / 2; ++u) {
          const float p0 = ex2(fmaf(__uint_as_float(sv[2 * u]), a.scale_log2, neg_m));
          const float p1 = ex2(fmaf(__uint_as_float(sv[2 * u + 1]), a.scale_log2, neg_m));
          __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          lp[u & 3] += __low2float(pb) + __high2float(pb);
          pw[u] = *reinterpret_cast<uint32_t*>(&pb);
        }
        if constexpr (KN / 2 == 32) {
          tc::st32(tmem + lane_base + kGColS + KN * b, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
        } else {
          uint32_t pw32[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) pw32[u] = u < KN / 2 ? pw[u % (KN / 2)] : 0u;
          tc::st32(tmem + lane_base + kGColS + KN * b, pw32);
        }
        tc::wait_st();
        tc::fence_before();
        mbar_arrive(&sm.p_ready[b]);
      }
      if (!ok) break;
      const int next = tile + gridDim.x;
      if (next < total) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_free, wt & 1, st))) break;
        tc::fence_after();
        load_q(g_work<HQ, KN>(a, next));
      }
      // ---- epilogue: this half of O / l -> bf16
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_done, wt & 1, st))) break;
      tc::fence_after();
      const float l = (lp[0] + lp[1]) + (lp[2] + lp[3]);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* dst = a.out + (static_cast<int64_t>(w.row0 + w.q0 + qi) * HQ + hd) * 512 + 256 * w.half;
#pragma unroll 1
      for (int blk = 0; blk < 8; blk += 2) {
        uint32_t o[64];
        tc::ld32(tmem + lane_base + kGColO + 32 * blk, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tc::ld32(tmem + lane_base + kGColO + 32 * blk + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
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

template <int LAYOUT, int HQ>
cudaError_t launch_lh(const LocalArgs& a, cudaStream_t st) {
  auto kern = global_prompt_tc_kernel<LAYOUT, HQ>;
  const size_t smem = sizeof(GPSmem<LAYOUT>);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid_ctas()), dim3(kGThreads), smem, st, a);
}

template <int LAYOUT>
cudaError_t launch_l(const LocalArgs& a, cudaStream_t st) {
  switch (a.num_q_heads) {
    case 8: return launch_lh<LAYOUT, 8>(a, st);
    case 16: return launch_lh<LAYOUT, 16>(a, st);
    case 32: return launch_lh<LAYOUT, 32>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_global_prompt_tc(int layout, const LocalArgs& a, cudaStream_t st) {
  return layout == GW_LAYOUT_GLOBAL_FOLDED ? launch_l<GW_LAYOUT_GLOBAL_FOLDED>(a, st)
                                           : launch_l<GW_LAYOUT_GLOBAL_FULL>(a, st);
}

}  // namespace gw
