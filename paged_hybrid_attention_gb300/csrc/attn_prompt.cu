// Prompt rows of a mixed step: sequences that contribute n > 1 query rows.
//
// "Gemma 4" (pegainfer model page), "Scheduling": a new prompt's rows are
// computed in the same batched step as the live streams' next token.  Row r
// of such a sequence sits at position p = L - n + r (the prompt's own K/V were
// appended first in the same step) and attends causally: keys
// [max(0, p - W + 1), p] on local layers, [0, p] on global layers.
//
// This file holds the tile plan shared by both families and the global-layer
// kernel; the local-layer kernel (tcgen05, tensor memory) is in
// attn_prompt_tc.cu.  The global kernel is FlashAttention-2 style with
// warp-level mma.sync (m16n8k16, bf16 in, fp32 accumulate) and an online
// base-2 softmax: a CTA owns 64 rows = (64/HQ queries) x HQ heads; pairs of
// warps split the head dim, exchange their partial logits through shared
// memory and each accumulate half of O.  Pages are copied whole with
// cp.async.bulk; the folded page's 8x8 blocks are read directly by ldmatrix,
// K = k_rot || V[128:512] by addressing.  Tiles of (sequence, KV head, query
// block) are enumerated by a small plan kernel and processed by persistent
// CTAs.
#include "common.cuh"

namespace gw {
namespace {

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void st_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
}
__device__ __forceinline__ void pair_bar(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// Byte offset of 16-byte chunk c of row r in a row-major tile whose rows are
// kChunks chunks long, with the chunk index XOR-swizzled by r mod 8.
template <int kChunks>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r * kChunks + (c ^ (r & 7))) * 16);
}

__device__ __forceinline__ int find_seq(const int32_t* base, int batch, int t) {
  int lo = 0, hi = batch;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One CTA: prompt_base[s] = prompt tiles of sequences before s.  A sequence
// with n > 1 rows contributes heads_factor * ceil(n / queries_per_tile).
__global__ void plan_prompt_kernel(const LocalArgs a, int heads_factor, int queries_per_tile) {
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
      if (n > 1) {
        if (L >= n && static_cast<int64_t>(L) <= static_cast<int64_t>(a.max_pages) * kPage)
          units = heads_factor * ((n + queries_per_tile - 1) / queries_per_tile);
        else
          set_status(a.status, GW_DEV_LEN_RANGE);
      }
    }
    int x = units;
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
    if (s < a.batch) a.prompt_base[s] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + units;
    __syncthreads();
  }
  if (threadIdx.x == 0) a.prompt_base[a.batch] = carry;
}

// =========================================================== global (hd 512)
constexpr int kRows = 64;     // query rows x heads per CTA
constexpr int kKeys = 32;     // keys per K/V tile
constexpr int kGlobalThreads = 256;

template <int LAYOUT>
struct GPT;
template <>
struct GPT<GW_LAYOUT_GLOBAL_FOLDED> {
  static constexpr int kPageBytes = 20480, kBlk = 80, kVcb = 0;
  __device__ static int k_cb(int d8) { return d8 < 16 ? 64 + d8 : d8; }  // 8-dim block of K dims [8 d8, 8 d8 + 8)
};
template <>
struct GPT<GW_LAYOUT_GLOBAL_FULL> {
  static constexpr int kPageBytes = 32768, kBlk = 128, kVcb = 64;
  __device__ static int k_cb(int d8) { return d8; }
};

template <int LAYOUT>
struct GlobalPromptSmem {
  uint8_t q[kRows * 1024];                       // [64 rows][512] bf16, swizzled
  uint8_t kv[2][2 * GPT<LAYOUT>::kPageBytes];    // two pages = 32 keys, per buffer
  float sx[2][8][16][32];                        // partial logits exchanged by warp pairs
  uint64_t bar[2];
  int32_t page_ok[2];                            // bit j: page j of the buffer was loaded
};

template <int LAYOUT, int HQ>
__global__ void __launch_bounds__(kGlobalThreads, 1) global_prompt_kernel(const LocalArgs a) {
  using T = GPT<LAYOUT>;
  constexpr int BQ = kRows / HQ;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  GlobalPromptSmem<LAYOUT>& sm = *reinterpret_cast<GlobalPromptSmem<LAYOUT>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;
  const int rg = warp >> 1, dh = warp & 1;  // row group (16 rows) and head-dim half
  pdl_wait();
  pdl_trigger();
  const int total = a.prompt_base[a.batch];
  const uint32_t q_s = smem_u32(sm.q);
  if (tid == 0) {
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    fence_mbar_init();
  }
  // zero the page buffers once: masked keys get p = 0, and 0 * finite = 0
  for (int i = tid; i < static_cast<int>(sizeof(sm.kv) / 16); i += kGlobalThreads) st_zero16(smem_u32(sm.kv) + i * 16);
  fence_proxy_async_smem();
  __syncthreads();
  uint32_t uses[2] = {0, 0};  // completed phases per buffer
  // a key's page is read again by every later query block of the prompt:
  // keep the pages in L2 (evict last)
  const uint64_t pol = policy_evict_last();

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int s = find_seq(a.prompt_base, a.batch, tile);
    const int n = a.cu_q_rows[s + 1] - a.cu_q_rows[s];
    const int qb = tile - a.prompt_base[s];
    const int L = a.seq_lens[s];
    const int P0 = L - n;
    const int q0 = qb * BQ;
    const int nq = min(BQ, n - q0);
    const int hi = P0 + q0 + nq - 1;
    const int t_hi = hi / kKeys;
    const int32_t* bt = a.block_table + static_cast<int64_t>(s) * a.max_pages;

    __syncthreads();
    for (int i = tid; i < kRows * 64; i += kGlobalThreads) {
      const int r = i >> 6, c = i & 63;
      const int qi = r / HQ, h = r % HQ;
      const uint32_t dst = q_s + swz<64>(r, c);
      if (qi < nq)
        cp_async16(dst, a.q + (static_cast<int64_t>(a.cu_q_rows[s] + q0 + qi) * HQ + h) * 512 + c * 8);
      else
        st_zero16(dst);
    }
    cp_commit();
    // page copies of tile t into buffer b (thread 0); returns the page validity bits
    auto issue = [&](int t, int b) {
      if (tid == 0) {
        uint32_t bytes = 0;
        int32_t pg[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int lp = t * 2 + j;
          pg[j] = -1;
          if (lp * kPage <= hi) {
            const int32_t p = bt[lp];
            if (p >= 0 && p < a.num_pages) {
              pg[j] = p;
              bytes += T::kPageBytes;
            } else {
              set_status(a.status, GW_DEV_PAGE_RANGE);
            }
          }
        }
        sm.page_ok[b] = (pg[0] >= 0 ? 1 : 0) | (pg[1] >= 0 ? 2 : 0);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sm.bar[b], bytes);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (pg[j] >= 0)
            bulk_g2s(sm.kv[b] + j * T::kPageBytes, a.pool + static_cast<int64_t>(pg[j]) * T::kPageBytes,
                     T::kPageBytes, &sm.bar[b], pol);
      }
    };
    issue(0, 0);

    int pos[2];
    bool rv[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int r = rg * 16 + g8 + 8 * h2;
      rv[h2] = (r / HQ) < nq;
      pos[h2] = P0 + q0 + r / HQ;
    }
    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    cp_wait<0>();
    __syncthreads();

    for (int t = 0; t <= t_hi; ++t) {
      const int b = t & 1;
      if (t < t_hi) issue(t + 1, b ^ 1);
      mbar_wait(&sm.bar[b], uses[b] & 1, a.status);  // on timeout the status says so; keep the CTA in step
      ++uses[b];
      const int page_ok = sm.page_ok[b];
      // keys of this tile at or past L sit in a page that may hold unwritten bytes
      for (int key_j = tid >> 4; key_j < kKeys; key_j += kGlobalThreads >> 4) {
        const int key = t * kKeys + key_j;
        if (key >= L && key / kPage * kPage < L) {
          const int j = key_j >> 4, tok = key_j & 15;
          const uint32_t row = smem_u32(sm.kv[b]) + j * T::kPageBytes + (tok >> 3) * T::kBlk * 128 + (tok & 7) * 16;
          for (int cb = tid & 15; cb < T::kBlk; cb += 16) st_zero16(row + cb * 128);
        }
      }
      __syncthreads();
      const uint32_t kv = smem_u32(sm.kv[b]);
      // ---- partial S over this warp's 256 dims
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        uint32_t af[4];
        const int r = rg * 16 + (lane & 15);
        const int dchunk = dh * 32 + 2 * kk + (lane >> 4);  // 8-dim chunk of the 512
        ldsm_x4(q_s + swz<64>(r, dchunk), af);
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // page j = keys 16j..16j+15
          uint32_t bf[4];
          const int mi = lane >> 3;
          const int d8 = dh * 32 + 2 * kk + (mi & 1);
          const int tb = mi >> 1;
          ldsm_x4(kv + j * T::kPageBytes + (tb * T::kBlk + T::k_cb(d8)) * 128 + (lane & 7) * 16, bf);
          mma16816(sacc[2 * j], af, bf[0], bf[1]);
          mma16816(sacc[2 * j + 1], af, bf[2], bf[3]);
        }
      }
      // ---- exchange with the partner warp (other dim half)
      float* mine = &sm.sx[t & 1][warp][0][lane];
      const float* theirs = &sm.sx[t & 1][warp ^ 1][0][lane];
#pragma unroll
      for (int i = 0; i < 16; ++i) mine[i * 32] = sacc[i >> 2][i & 3];
      pair_bar(1 + rg);
#pragma unroll
      for (int i = 0; i < 16; ++i) sacc[i >> 2][i & 3] += theirs[i * 32];
      // ---- mask, online softmax
      float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h2 = e >> 1;
          const int key = t * kKeys + nt * 8 + 2 * c4 + (e & 1);
          const bool ok = rv[h2] && key <= pos[h2] && ((page_ok >> (nt >> 1)) & 1);
          const float sv = ok ? sacc[nt][e] * a.scale_log2 : -INFINITY;
          sacc[nt][e] = sv;
          rmax[h2] = fmaxf(rmax[h2], sv);
        }
      }
      float alpha[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        rmax[h2] = fmaxf(rmax[h2], __shfl_xor_sync(0xffffffffu, rmax[h2], 1));
        rmax[h2] = fmaxf(rmax[h2], __shfl_xor_sync(0xffffffffu, rmax[h2], 2));
        const float mn = fmaxf(m[h2], rmax[h2]);
        alpha[h2] = mn == -INFINITY ? 1.f : ex2(m[h2] - mn);
        m[h2] = mn;
      }
      uint32_t pf[2][4];
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = sacc[nt][e] == -INFINITY ? 0.f : ex2(sacc[nt][e] - m[e >> 1]);
        const uint32_t lo2 = pack_bf16(p[0], p[1]), hi2 = pack_bf16(p[2], p[3]);
        const __nv_bfloat162 bl = *reinterpret_cast<const __nv_bfloat162*>(&lo2);
        const __nv_bfloat162 bh = *reinterpret_cast<const __nv_bfloat162*>(&hi2);
        rs[0] += __low2float(bl) + __high2float(bl);
        rs[1] += __low2float(bh) + __high2float(bh);
        pf[nt >> 1][(nt & 1) * 2 + 0] = lo2;
        pf[nt >> 1][(nt & 1) * 2 + 1] = hi2;
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) l[h2] = l[h2] * alpha[h2] + rs[h2];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      // ---- O += P V over this warp's 256 dims
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t bf[4];
          const int mi = lane >> 3;
          const int tb = mi & 1;
          const int cb = T::kVcb + dh * 32 + 2 * np + (mi >> 1);
          ldsm_x4_t(kv + j * T::kPageBytes + (tb * T::kBlk + cb) * 128 + (lane & 7) * 16, bf);
          mma16816(o[2 * np], pf[j], bf[0], bf[1]);
          mma16816(o[2 * np + 1], pf[j], bf[2], bf[3]);
        }
      }
      __syncthreads();
    }
    // ---- epilogue
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
      l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
    }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      if (!rv[h2]) continue;
      const int r = rg * 16 + g8 + 8 * h2;
      const int qi = r / HQ, h = r % HQ;
      const float inv = l[h2] > 0.f ? 1.f / l[h2] : 0.f;
      uint16_t* dst = a.out + (static_cast<int64_t>(a.cu_q_rows[s] + q0 + qi) * HQ + h) * 512 + dh * 256;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        *reinterpret_cast<uint32_t*>(dst + i * 8 + 2 * c4) = pack_bf16(o[i][2 * h2] * inv, o[i][2 * h2 + 1] * inv);
    }
  }
}

template <int G>
cudaError_t launch_local_g(const LocalArgs& a, cudaStream_t st) {
  cudaError_t e = launch_pdl(plan_prompt_kernel, dim3(1), dim3(1024), 0, st, a, a.kv_heads, 128 / G);
  if (e != cudaSuccess) return e;
  return launch_local_prompt_tc(G, a, st);
}

template <int LAYOUT, int HQ>
cudaError_t launch_global_hq(const LocalArgs& a, cudaStream_t st) {
  cudaError_t e = launch_pdl(plan_prompt_kernel, dim3(1), dim3(1024), 0, st, a, 1, kRows / HQ);
  if (e != cudaSuccess) return e;
  auto kern = global_prompt_kernel<LAYOUT, HQ>;
  const size_t smem = sizeof(GlobalPromptSmem<LAYOUT>);
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms()), dim3(kGlobalThreads), smem, st, a);
}

template <int LAYOUT>
cudaError_t launch_global_layout(const LocalArgs& a, cudaStream_t st) {
  switch (a.num_q_heads) {
    case 8: return launch_global_hq<LAYOUT, 8>(a, st);
    case 16: return launch_global_hq<LAYOUT, 16>(a, st);
    case 32: return launch_global_hq<LAYOUT, 32>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_local_prompt(int dtype, int group, const LocalArgs& a, int /*max_q_rows*/, cudaStream_t st) {
  if (dtype != GW_KV_BF16) return cudaErrorNotSupported;
  switch (group) {
    case 1: return launch_local_g<1>(a, st);
    case 2: return launch_local_g<2>(a, st);
    case 4: return launch_local_g<4>(a, st);
    case 8: return launch_local_g<8>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_global_prompt(int layout, const LocalArgs& a, int /*max_q_rows*/, cudaStream_t st) {
  return layout == GW_LAYOUT_GLOBAL_FOLDED ? launch_global_layout<GW_LAYOUT_GLOBAL_FOLDED>(a, st)
                                           : launch_global_layout<GW_LAYOUT_GLOBAL_FULL>(a, st);
}

}  // namespace gw
