// Sliding-window decode attention over an e4m3 LOCAL pool on the tensor
// cores (tcgen05, kind::f8f6f4).
//
// "feat(gemma4): the sliding family serves an opt in fp8 KV pool",
// "Description": the sliding family's K/V may be stored as e4m3 at scale
// 1.0, halving the decode step's dominant KV read.  "Gemma 4" (pegainfer
// model page), "Architecture notes": a decode row of q head h attends to the
// last `window` keys of KV head h / G.
//
// The split plan is the one of the other local decode kernels: a unit is
// (sequence, KV head, chunk of 8 pages of the window), its partial (m, l, o)
// per q head goes to the workspace and the combine merges the chunks.  Here a
// unit is exactly one 128-token tile, so it needs no online rescaling:
//   S^T[128 tok x 16] = K[128 x 256] . [q_hi; q_lo; 0]^T    (UMMA M=128, N=16, K=256: 8 MMAs)
//   O^T[256 x 16]    = V^T[256 x 128] . [P_hi | P_lo | 0]    (M=128 per 128 dims, N=16, K=128: 8 MMAs)
// with fp32 accumulators in tensor memory; logit h is column h plus column
// G + h, and likewise for O.  q enters as two e4m3 terms after an exact
// power-of-two scaling per head (its largest |q| lands in [128, 256)), P as
// two e4m3 terms of the max-subtracted weights (p <= 1), and l sums exactly
// the weights the contraction uses.
//
// K and V arrive by tensor-map copies of the pool (16 token rows x 128 B per
// box, two 128-dim chunks per row, 128-byte swizzled): a unit's 8 pages are
// 32 boxes, issued by four producer warps (8 lanes each: one warp issuing
// all 32 took about 2 us per unit), into one of three 64 KB stages.  K is the
// K-major A operand of Q.K^T, V the MN-major A operand of P.V (the same
// swizzled rows).
//
// Warp roles (352 threads, one persistent CTA per SM, units dealt
// round-robin from the in-kernel plan):
//   warps 0-3  softmax (thread t owns token t of the unit, TMEM lane t) and
//              epilogue (thread t owns dims t and 128 + t of O^T)
//   warps 4-7  producers: the unit's page numbers, 8 tensor-map boxes each
//   warp 8     Q.K^T issue and TMEM owner
//   warp 9     q loader: scaling and the two-term split of the unit's G heads
//   warp 10    P.V issue
//   warp 11    (fused append only, gw_append_decode_attn_local) writes the
//              step's row of each (sequence, KV head) whose last chunk this
//              CTA decodes, in the order of the CTA's units; the producer
//              warp that copies that unit's last page waits for it.
// Every wait is bounded; a timeout raises GW_DEV_TIMEOUT and the roles stop.
#include "local_append.cuh"
#include "plan.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace gw {
namespace {

constexpr int kE8Producers = 4;                // producer warps: 8 boxes (2 pages) each
constexpr int kE8Threads = (4 + kE8Producers + 3) * 32;
constexpr int kE8WarpQK = 4 + kE8Producers, kE8WarpQL = kE8WarpQK + 1, kE8WarpPV = kE8WarpQK + 2;
constexpr int kE8Tok = 128;                    // tokens per unit (8 pages)
constexpr int kE8Chunk = kLocalChunkPagesE4m3;  // pages per unit
constexpr int kE8Stages = 3;
constexpr uint32_t kE8Plane = kE8Tok * 128;    // one 128-dim chunk of K or V: 16 KB
constexpr uint32_t kE8Stage = 4 * kE8Plane;    // K chunk 0, K chunk 1, V chunk 0, V chunk 1
constexpr int kE8N = 16;                       // UMMA N: [hi (G) | lo (G) | zeros]
// TMEM columns: S^T buffers at 0 and 16, O^T buffers at 64 and 96 (2 x 16 each)
constexpr uint32_t kE8ColS = 0, kE8ColO = 64;

struct E8Unit {
  int32_t unit, s, g, last;  // last: the sequence's last chunk
  int32_t lp0, tok_lo, tok_hi;  // first logical page; token range [tok_lo, tok_hi) in the window
  int32_t mask;                 // pages of the unit that were loaded (bit j: page lp0 + j)
};

struct __align__(1024) E8Smem {
  uint8_t stage[kE8Stages][kE8Stage];
  uint8_t q[2][kE8N * 256];  // [hi; lo; 0] K-major: [row block 2][dim block 16][8 rows][16 B]
  uint8_t p[2][kE8Tok * 16];  // P^T MN-major: [token block 16][8 tokens][16 columns]
  float qscale[4][8];         // per unit (mod 4), per head: 2^-e of q's scaling
  float red[4][2][8];         // per-warp reductions: max and sum per head
  E8Unit ring[kE8Stages];
  uint64_t full[kE8Stages], empty[kE8Stages];
  uint64_t s_ready[2], p_ready[2], pfree[2], o_done[2], o_free[2], q_ready[2], q_free[2], qs_ready[4];
  uint32_t tmem_base;
  int32_t app_done;  // fused append: units of this CTA (in order) whose rows are written
  int32_t ub[kMaxBatch + 1 + 32];  // split plan (+ scan scratch)
};
static_assert(sizeof(E8Smem) <= 232448, "shared memory of one CTA");

__device__ __forceinline__ void e8_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// x as two e4m3 terms (x0 in the low byte of each 16-bit word); `sum` gets
// hi + lo, the value the contraction uses.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo, float2& sum) {
  const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
  const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
  const __nv_fp8x2_storage_t l2 =
      __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
  const float2 lf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(l2, __NV_E4M3)));
  hi = h2;
  lo = l2;
  sum = make_float2(hf.x + lf.x, hf.y + lf.y);
}

// kApp: the fused-append variant, with warp 11.
template <int G, bool kApp>
__global__ void __launch_bounds__(kE8Threads + (kApp ? 32 : 0), 1)
    local_decode_e4m3_tc_kernel(const LocalArgs a, const __grid_constant__ CUtensorMap kv_map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  E8Smem& sm = *reinterpret_cast<E8Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  int32_t* st = a.status;

  // the q buffers' padding rows (2G..15) stay zero
  for (int i = tid; i < static_cast<int>(sizeof(sm.q) / 16); i += kE8Threads)
    if (tid < kE8Threads) reinterpret_cast<uint4*>(sm.q)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    sm.app_done = 0;
    for (int b = 0; b < kE8Stages; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], 128);
      mbar_init(&sm.pfree[b], 1);
      mbar_init(&sm.o_done[b], 1);
      mbar_init(&sm.o_free[b], 128);
      mbar_init(&sm.q_ready[b], 1);
      mbar_init(&sm.q_free[b], 1);
    }
    for (int b = 0; b < 4; ++b) mbar_init(&sm.qs_ready[b], 1);
    fence_mbar_init();
  }
  if (warp == kE8WarpQK) {
    tc::alloc(&sm.tmem_base, 128);
    tc::relinquish();
  }
  // With early inputs the plan and the producer's first page numbers are
  // read before the wait on the previous kernel (gw_set_early_inputs).
  const bool early = a.early_inputs != 0;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  plan_in_smem(a, sm.ub, sm.ub + kMaxBatch + 1,
               [&](int L) { return a.kv_heads * local_chunks(L, a.window, kE8Chunk); }, !early);
  const int total = sm.ub[a.batch];
  auto wait_prev = [&]() {
    if (early) {
      pdl_wait();
      pdl_trigger();
    }
  };
  fence_proxy_async_smem();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (total > a.max_units) {  // uniform
    wait_prev();
    if (blockIdx.x == 0 && tid == 0) set_status(st, GW_DEV_WORKSPACE);
  } else if (warp >= 4 && warp < 4 + kE8Producers) {
    // ------------------------------------------------------------ producers
    // Producer warp w issues pages 2w, 2w + 1 of each unit: lane l < 8 the
    // box of page 2w + (l >> 2), K or V ((l >> 1) & 1), chunk l & 1.  Lanes
    // 0-7 of every producer read the unit's 8 page numbers; the first
    // producer publishes the unit and the bytes to expect.  The index loads
    // run one unit ahead of the copies.
    const int pw = warp - 4;
    const uint64_t pol = policy_evict_first();
    const int j = 2 * pw + ((lane >> 2) & 1), kv = (lane >> 1) & 1, c = lane & 1;
    const int stride = static_cast<int>(gridDim.x);
    auto unit_of = [&](int uu, int L) {  // the unit's pages from its sequence length
      E8Unit d;
      d.unit = uu;
      d.s = plan_seq(sm.ub, a.batch, uu);
      const int first = L > a.window ? L - a.window : 0;
      const int p0 = first / kPage, p1 = (L - 1) / kPage;
      const int nc = (p1 - p0 + kE8Chunk) / kE8Chunk;
      const int r = uu - sm.ub[d.s];
      d.g = r / nc;
      d.lp0 = p0 + (r % nc) * kE8Chunk;
      const int lp1 = min(d.lp0 + kE8Chunk, p1 + 1);
      d.tok_lo = max(first, d.lp0 * kPage);
      d.tok_hi = min(L, lp1 * kPage);
      d.last = d.tok_hi == L;
      d.mask = 0;
      return d;
    };
    auto len_of = [&](int uu) { return uu < total ? a.seq_lens[plan_seq(sm.ub, a.batch, uu)] : 1; };
    auto pages_of = [&](const E8Unit& d, int uu) {  // lane l < 8: physical page l of the unit
      const int lp = d.lp0 + lane;
      return uu < total && lane < kE8Chunk && lp * kPage < d.tok_hi
                 ? a.block_table[static_cast<int64_t>(d.s) * a.max_pages + lp]
                 : -1;
    };
    int u = blockIdx.x;
    E8Unit d0 = unit_of(u, len_of(u));
    int32_t pg0 = pages_of(d0, u);
    int L1 = len_of(u + stride);
    wait_prev();
    for (int k = 0; u < total; u += stride, ++k) {
      const int b = k % kE8Stages;
      const E8Unit d1 = unit_of(u + stride, L1);
      const int32_t pg1 = pages_of(d1, u + stride);
      const int L2 = len_of(u + 2 * stride);
      const bool page_in = lane < kE8Chunk && (d0.lp0 + lane) * kPage < d0.tok_hi;
      const bool page_ok = page_in && pg0 >= 0 && pg0 < a.num_pages;
      if (pw == 0 && page_in && !page_ok) set_status(st, GW_DEV_PAGE_RANGE);
      const uint32_t pages = __ballot_sync(0xffffffffu, page_ok);  // bit j: page j loaded
      const int32_t mine = __shfl_sync(0xffffffffu, pg0, j);
      const bool ok = lane < 8 && ((pages >> j) & 1);
      if (k >= kE8Stages && !warp_wait(&sm.empty[b], ((k / kE8Stages) - 1) & 1, st)) break;
      if (kApp && d0.last && ((d0.tok_hi - 1) / kPage - d0.lp0) / 2 == pw) {
        // this warp copies the page holding the step's row: wait until the
        // append warp wrote it
        if (lane == 0)
          wait_counter(&sm.app_done, (u - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1, st);
        __syncwarp();
        fence_proxy_async_global();
      }
      if (pw == 0 && lane == 0) {
        E8Unit e = d0;
        e.mask = static_cast<int32_t>(pages & 0xFF);
        sm.ring[b] = e;
        mbar_arrive_expect_tx(&sm.full[b], static_cast<uint32_t>(__popc(pages & 0xFF)) * 4 * 2048);
      }
      __syncwarp();
      if (ok)
        tma_rows(smem_u32(sm.stage[b]) + (2 * kv + c) * kE8Plane + j * 2048, &kv_map, c,
                 ((mine * a.kv_heads + d0.g) * 2 + kv) * kPage, &sm.full[b], pol);
      d0 = d1;
      pg0 = pg1;
      L1 = L2;
    }
  } else if (warp == kE8WarpQK) {
    // ----------------------------------------------------------- Q.K^T issue
    wait_prev();
    const uint32_t id_s = tc::idesc_e4m3(128, kE8N, false, false);
    int k = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++k) {
      const int b = k % kE8Stages, sb = k & 1, qb = k & 1;
      if (!warp_wait(&sm.full[b], (k / kE8Stages) & 1, st)) break;
      if (!warp_wait(&sm.q_ready[qb], (k >> 1) & 1, st)) break;
      // S buffer sb is free once the softmax of unit k - 2 has read it
      if (k >= 2 && !warp_wait(&sm.p_ready[sb], ((k >> 1) - 1) & 1, st)) break;
      tc::fence_after();
      const uint32_t ka = smem_u32(sm.stage[b]);
      const uint64_t qd = tc::smem_desc(smem_u32(sm.q[qb]), 128, 16 * 128);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // 32 dims per K-step
        tc::mma_e4m3_warp(tmem + kE8ColS + 16 * sb, tc::smem_desc_sw128(ka + (ks >> 2) * kE8Plane + (ks & 3) * 32, 16),
                          qd + ((ks * 2 * 128) >> 4), id_s, ks > 0);
      tc::commit_warp(&sm.s_ready[sb]);
      tc::commit_warp(&sm.q_free[qb]);
    }
  } else if (warp == kE8WarpPV) {
    // ------------------------------------------------------------ P.V issue
    wait_prev();
    const uint32_t id_o = tc::idesc_e4m3(128, kE8N, true, true);
    int k = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++k) {
      const int b = k % kE8Stages, pb = k & 1, ob = k & 1;
      if (!warp_wait(&sm.p_ready[pb], (k >> 1) & 1, st)) break;
      if (k >= 2 && !warp_wait(&sm.o_free[ob], ((k >> 1) - 1) & 1, st)) break;
      tc::fence_after();
      const uint32_t va = smem_u32(sm.stage[b]) + 2 * kE8Plane;
      const uint64_t pd = tc::smem_desc(smem_u32(sm.p[pb]), 128, 128);
#pragma unroll
      for (int c = 0; c < 2; ++c)      // 128 dims per M block
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 tokens per K-step
          tc::mma_e4m3_warp(tmem + kE8ColO + 32 * ob + 16 * c,
                            tc::smem_desc_sw128(va + c * kE8Plane + kk * 4096, kE8Plane),
                            pd + ((kk * 4 * 128) >> 4), id_o, kk > 0);
      tc::commit_warp(&sm.empty[b]);
      tc::commit_warp(&sm.pfree[pb]);
      tc::commit_warp(&sm.o_done[ob]);
    }
  } else if (warp == kE8WarpQL) {
    // ------------------------------------------------------------- q loader
    // Unit k + 1's q rows are loaded while unit k's are converted.
    wait_prev();
    const int stride = static_cast<int>(gridDim.x);
    auto q_src = [&](int uu) {  // this lane's 8 dims of the unit's first head
      const int s = plan_seq(sm.ub, a.batch, uu);
      const int L = a.seq_lens[s];
      const int row = a.cu_q_rows[s];
      const int first = L > a.window ? L - a.window : 0;
      const int nc = ((L - 1) / kPage - first / kPage + kE8Chunk) / kE8Chunk;
      const int g = (uu - sm.ub[s]) / nc;
      return a.q + (static_cast<int64_t>(row) * a.num_q_heads + g * G) * 256 + 8 * lane;
    };
    float x[G][8];
    auto load = [&](const uint16_t* src) {
#pragma unroll
      for (int h = 0; h < G; ++h) bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + h * 256), x[h]);
    };
    if (static_cast<int>(blockIdx.x) < total) load(q_src(blockIdx.x));
    int k = 0;
    for (int u = blockIdx.x; u < total; u += stride, ++k) {
      const int qb = k & 1;
      const uint16_t* next = u + stride < total ? q_src(u + stride) : nullptr;  // index loads in flight
      if (k >= 2 && !warp_wait(&sm.q_free[qb], ((k >> 1) - 1) & 1, st)) break;
      uint8_t* qd = sm.q[qb];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[h][i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int ex = m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 : 7;
        const int e = min(125, max(-125, 7 - ex));
        const float up = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        if (lane == 0) sm.qscale[k & 3][h] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t hi, lo;
          float2 used;
          split2(x[h][2 * i] * up, x[h][2 * i + 1] * up, hi, lo, used);
          hw[i >> 1] |= hi << (16 * (i & 1));
          lw[i >> 1] |= lo << (16 * (i & 1));
        }
        // rows h (hi) and G + h (lo), dims [8 lane, 8 lane + 8)
        auto at = [&](int r) { return qd + ((r >> 3) * 16 + (lane >> 1)) * 128 + (r & 7) * 16 + (lane & 1) * 8; };
        *reinterpret_cast<uint2*>(at(h)) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(at(G + h)) = make_uint2(lw[0], lw[1]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.q_ready[qb]);
        mbar_arrive(&sm.qs_ready[k & 3]);
      }
      if (next) load(next);
    }
  } else if (kApp && warp == kE8Threads / 32) {
    // -------------------------------------------- fused append (local_append.cuh)
    local_append_warp<GW_KV_E4M3>(a, sm.ub, total, &sm.app_done, early);
  } else if (warp < 4) {
    // ------------------------------------------------ softmax + epilogue
    // The four warps meet at a named barrier twice per unit, so none may
    // leave the loop alone: after a wait gives up (warp-uniform), a warp
    // skips the rest of the work but still passes every barrier.
    wait_prev();
    if (early) publish_plan(a, sm.ub, tid, 128);
    const int t = tid;  // token of the unit = TMEM lane; dims t, 128 + t in the epilogue
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    bool bad = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (!bad && !warp_wait(bar, parity, st)) bad = true;
      return !bad;
    };
    // Iteration k computes the weights of unit k, then writes the partial of
    // unit k - 1 (whose P.V has had the softmax of unit k to complete).
    int32_t prev_unit = -1;
    float prev_m[G], prev_l[G];
    int k = 0;
    for (int u = blockIdx.x;; u += gridDim.x, ++k) {
      const bool have = u < total;
      if (!have && prev_unit < 0) break;
      if (have) {
        const int b = k % kE8Stages, sb = k & 1, pb = k & 1;
        E8Unit d{};
        if (wait(&sm.full[b], (k / kE8Stages) & 1)) d = sm.ring[b];
        wait(&sm.qs_ready[k & 3], (k >> 2) & 1);
        wait(&sm.s_ready[sb], (k >> 1) & 1);
        tc::fence_after();
        uint32_t r[16];
        tc::ld16(tmem + lane_base + kE8ColS + 16 * sb, r);
        tc::wait_ld();
        const int tabs = d.lp0 * kPage + t;
        const bool valid = !bad && tabs >= d.tok_lo && tabs < d.tok_hi && ((d.mask >> (t >> 4)) & 1);
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h)
          s[h] = valid ? (__uint_as_float(r[h]) + __uint_as_float(r[G + h])) * (sm.qscale[k & 3][h] * a.scale_log2)
                       : -INFINITY;
        // maximum per head over the unit's tokens
        float mx[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float v = s[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          mx[h] = v;
        }
        if (lane == 0)
#pragma unroll
          for (int h = 0; h < G; ++h) sm.red[warp][0][h] = mx[h];
        e8_bar();
#pragma unroll
        for (int h = 0; h < G; ++h)
          mx[h] = fmaxf(fmaxf(sm.red[0][0][h], sm.red[1][0][h]), fmaxf(sm.red[2][0][h], sm.red[3][0][h]));
        // weights as two e4m3 terms; P^T row t: columns h (hi), G + h (lo)
        if (k >= 2) wait(&sm.pfree[pb], ((k >> 1) - 1) & 1);
        uint8_t prow[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        float lw[G];
#pragma unroll
        for (int h = 0; h < G; h += 2) {
          const float p0 = valid && mx[h] != -INFINITY ? ex2(s[h] - mx[h]) : 0.f;
          const float p1 = h + 1 < G && valid && mx[h + 1] != -INFINITY ? ex2(s[h + 1] - mx[h + 1]) : 0.f;
          uint32_t hi, lo;
          float2 used;
          split2(p0, p1, hi, lo, used);
          prow[h] = hi & 0xFF;
          prow[G + h] = lo & 0xFF;
          lw[h] = used.x;
          if (h + 1 < G) {
            prow[h + 1] = (hi >> 8) & 0xFF;
            prow[G + h + 1] = (lo >> 8) & 0xFF;
            lw[h + 1] = used.y;
          }
        }
        if (!bad) {
          uint4 pv;
          pv.x = prow[0] | (prow[1] << 8) | (prow[2] << 16) | (static_cast<uint32_t>(prow[3]) << 24);
          pv.y = prow[4] | (prow[5] << 8) | (prow[6] << 16) | (static_cast<uint32_t>(prow[7]) << 24);
          pv.z = prow[8] | (prow[9] << 8) | (prow[10] << 16) | (static_cast<uint32_t>(prow[11]) << 24);
          pv.w = prow[12] | (prow[13] << 8) | (prow[14] << 16) | (static_cast<uint32_t>(prow[15]) << 24);
          *reinterpret_cast<uint4*>(sm.p[pb] + (t >> 3) * 128 + (t & 7) * 16) = pv;
          if (!valid) {
            // a key outside the unit's range (or in a page not loaded): its V
            // row may hold anything the pool did (even NaN patterns); 0 * NaN
            // would reach O, so the row is cleared
            uint8_t* vrow = sm.stage[b] + 2 * kE8Plane + t * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4*>(vrow + c * kE8Plane + q * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        // l per head: sum over tokens of the weights used (fixed order)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float v = lw[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          lw[h] = v;
        }
        if (lane == 0)
#pragma unroll
          for (int h = 0; h < G; ++h) sm.red[warp][1][h] = lw[h];
        fence_proxy_async_smem();
        tc::fence_before();
        if (!bad) mbar_arrive(&sm.p_ready[pb]);
        e8_bar();
        // what the epilogue of this unit needs, held for the next iteration
        float lsum[G];
#pragma unroll
        for (int h = 0; h < G; ++h)
          lsum[h] = ((sm.red[0][1][h] + sm.red[1][1][h]) + sm.red[2][1][h]) + sm.red[3][1][h];
        // ---- the partial of the previous unit
        if (prev_unit >= 0) {
          const int ok = (k - 1) & 1;
          wait(&sm.o_done[ok], ((k - 1) >> 1) & 1);
          tc::fence_after();
          float* po = a.part_o + static_cast<int64_t>(prev_unit) * G * 256;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[16];
            tc::ld16(tmem + lane_base + kE8ColO + 32 * ok + 16 * c, o);
            tc::wait_ld();
            if (!bad)
#pragma unroll
              for (int h = 0; h < G; ++h) po[h * 256 + 128 * c + t] = __uint_as_float(o[h]) + __uint_as_float(o[G + h]);
          }
          if (!bad)
#pragma unroll
            for (int h = 0; h < G; ++h)
              if (t == h) a.part_ml[static_cast<int64_t>(prev_unit) * G + h] = make_float2(prev_m[h], prev_l[h]);
          tc::fence_before();
          if (!bad) mbar_arrive(&sm.o_free[ok]);
        }
        prev_unit = d.unit;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          prev_m[h] = mx[h];
          prev_l[h] = lsum[h];
        }
      } else {
        // ---- no unit left: the partial of the last one
        const int ok = (k - 1) & 1;
        wait(&sm.o_done[ok], ((k - 1) >> 1) & 1);
        tc::fence_after();
        float* po = a.part_o + static_cast<int64_t>(prev_unit) * G * 256;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[16];
          tc::ld16(tmem + lane_base + kE8ColO + 32 * ok + 16 * c, o);
          tc::wait_ld();
          if (!bad)
#pragma unroll
            for (int h = 0; h < G; ++h) po[h * 256 + 128 * c + t] = __uint_as_float(o[h]) + __uint_as_float(o[G + h]);
        }
        if (!bad)
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (t == h) a.part_ml[static_cast<int64_t>(prev_unit) * G + h] = make_float2(prev_m[h], prev_l[h]);
        break;
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == kE8WarpQK) {
    tc::fence_after();
    tc::dealloc(tmem, 128);
  }
}

template <int G>
cudaError_t launch_g(const LocalArgs& a, cudaStream_t st) {
  CUtensorMap map;
  cudaError_t e = make_local_kv_map(a, &map, GW_KV_E4M3);
  if (e != cudaSuccess) return e;
  auto kern = a.k_new ? local_decode_e4m3_tc_kernel<G, true> : local_decode_e4m3_tc_kernel<G, false>;
  const size_t smem = sizeof(E8Smem);
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid_ctas()), dim3(kE8Threads + (a.k_new ? 32 : 0)), smem, st, a, map);
  if (e != cudaSuccess) return e;
  return launch_combine(a, G, 256, local_max_chunks(a.max_pages, a.window, kE8Chunk), true, st);
}

}  // namespace

cudaError_t launch_local_decode_e4m3_tc(int group, const LocalArgs& a, cudaStream_t st) {
  switch (group) {
    case 1: return launch_g<1>(a, st);
    case 2: return launch_g<2>(a, st);
    case 4: return launch_g<4>(a, st);
    case 8: return launch_g<8>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gw
