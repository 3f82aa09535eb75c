// Sliding-window (local) decode attention over the paged LOCAL pool.
//
// "Gemma 4" (pegainfer model page), "Architecture notes" and "Scheduling":
// five of six layers attend over the last 1024 tokens with head dim 256 and
// grouped KV heads, each in its own pool of 16-token pages; every active
// request advances one token per batched step.  "feat(gemma4): the sliding
// family serves an opt in fp8 KV pool", "Description": the pool may hold
// e4m3 at scale 1.0; those pools are served by the tcgen05 kernel of
// attn_local_e4m3_tc.cu, this file holds the bf16 kernel.
//
// Split-KV flash decoding (the plan, the partials and the combine are also
// the e4m3 kernel's):
//   * Work unit = (sequence, KV head, chunk of up to 8 pages of the window).
//     The split depends on the sequence's own length only.
//   * Persistent CTAs, one per SM, of independent warps.  Every CTA computes
//     the batch's split plan (unit offsets) into its own shared memory, so no
//     plan kernel and no work counter sit in front of the decode; units are
//     dealt round-robin over the warps, SM-minor, so each round spreads evenly
//     over the SMs.
//   * Each warp streams its units' pages through a private 2-stage ring,
//     prefetching across unit boundaries, and writes an unnormalised partial
//     (m, l, o) per unit; a combine kernel merges a sequence's partials in
//     chunk order (log-sum-exp) into bf16.
//   * Softmax is base 2 in fp32 against a reference max; P is rounded to the
//     multiplicand format and l sums exactly the rounded weights.
//
// bf16 pools (local_decode_tc_kernel, 6 warps): a stage is one 16-token page
// head (K and V, 16 KB) brought by 4 TMA tensor copies into 128-byte-swizzled
// shared memory; q.K^T and P.V run on warp-level tensor cores (mma.sync
// m16n8k16, the G heads of the group as rows) with P kept in registers.
#include "local_append.cuh"
#include "plan.cuh"
#include "tma.cuh"

namespace gw {
namespace {

struct Unit {
  int32_t s, g, hp_lo, n, tok_lo, tok_hi, unit, row;
  int32_t last;  // the sequence's last chunk (its range ends at the sequence's end)
};

template <class T>
__device__ __forceinline__ Unit decode_unit(const LocalArgs& a, const int32_t* ub, int u) {
  const int lo = plan_seq(ub, a.batch, u);
  Unit d;
  d.s = lo;
  const int L = a.seq_lens[lo];
  const int first = L > a.window ? L - a.window : 0;
  const int p0 = first / kPage, p1 = (L - 1) / kPage;
  const int nc = (p1 - p0 + T::kChunk) / T::kChunk;
  const int r = u - ub[lo];
  d.g = r / nc;
  const int c = r % nc;
  const int lpa = p0 + c * T::kChunk;
  const int lpb = min(lpa + T::kChunk, p1 + 1);
  d.tok_lo = max(first, lpa * kPage);
  d.tok_hi = min(L, lpb * kPage);
  d.hp_lo = d.tok_lo / T::kTok;
  d.n = (d.tok_hi - 1) / T::kTok + 1 - d.hp_lo;
  d.unit = u;
  d.row = a.cu_q_rows[lo];
  d.last = d.tok_hi == L;
  return d;
}

// Warps per CTA that take units.  Units are dealt in rounds of warps x CTAs
// and are nearly all the same size, so a call lasts as long as the warps
// that get the most rounds; a partial last round leaves the others idle.  Of
// wmax, wmax - 1 and wmax - 2 warps, take the one that wastes least of the
// final round, counting each warp given up as 3% of streaming capacity.
// Which warp runs a unit never changes its arithmetic.
__device__ __forceinline__ int active_warps(int units, int wmax) {
  int best = wmax;
  float best_score = -1.f;
  for (int w = wmax; w >= wmax - 2 && w >= 1; --w) {
    const int slots = w * static_cast<int>(gridDim.x);
    const int rounds = (units + slots - 1) / slots;
    const float eff = rounds > 0 ? static_cast<float>(units) / static_cast<float>(rounds * slots) : 1.f;
    const float score = eff * (1.f - 0.03f * static_cast<float>(wmax - w));
    if (score > best_score) {
      best_score = score;
      best = w;
    }
  }
  return best;
}

template <int kChunk>
__device__ __forceinline__ void local_plan(const LocalArgs& a, int32_t* ub, bool publish) {
  plan_in_smem(a, ub, ub + kMaxBatch + 1, [&](int L) { return a.kv_heads * local_chunks(L, a.window, kChunk); },
               publish);
}


// ---------------------------------------------------------------------------
// bf16 pages on warp-level tensor cores (mma.sync), fed by TMA.  A stage is
// one 16-token page head: K and V (4 chunks x 16 rows x 128 B each), 16 KB
// copied as 4 tensor boxes of 4 KB (a chunk's 16 K rows and 16 V rows, which
// are adjacent in the pool) issued by 4 lanes, landing 128-byte swizzled so
// that every ldmatrix below reads 8 distinct bank groups.
//   S[16 x 16]   = Q[16 x 256] . K^T      (m16n8k16 x 2 token halves; rows
//                                          = the G heads of the KV head)
//   O^T[256 x 8] += V^T[256 x 16] . P^T   (m16n8k16; columns = heads)
// The accumulator layout of S (lane: head lane/4, tokens 2(lane%4)+{0,1} of
// each half) is the B-operand layout of P^T, so the weights stay in
// registers; about 60 warp instructions per 16 tokens instead of ~700.
constexpr int kTcWarps = 6;
constexpr int kTcStages = 2;
// A stage holds, per 64-dim chunk c, the page head's 16 K rows then its 16 V
// rows (one 4 KB tensor-map box: K and V of a page head are adjacent in the
// pool), so K chunk c sits at 4096 c and V chunk c at 4096 c + 2048.
constexpr int kTcStage = 16384;

struct __align__(1024) TcWarpSmem {
  uint8_t stage[kTcStages][kTcStage];
  uint64_t bar[kTcStages];
  int32_t valid[kTcStages];
  Unit ring[kTcStages + 2];
};

struct TcTraits {
  static constexpr int kTok = 16;  // tokens per stage
  static constexpr int kChunk = kLocalChunkPagesBf16;
};

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a . b with a 16 x 16 (rows 8..15 zero: a1 = a3 = 0), b 16 x 8
__device__ __forceinline__ void hmma_q(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void hmma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int G>
__global__ void __launch_bounds__(kTcWarps * 32 + 32, 1)
    local_decode_tc_kernel(const LocalArgs a, const __grid_constant__ CUtensorMap kv_map) {
  using T = TcTraits;
  constexpr int kTok = T::kTok;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TcWarpSmem& sm = reinterpret_cast<TcWarpSmem*>(smem_raw)[warp < kTcWarps ? warp : 0];
  if (lane == 0 && warp < kTcWarps) {
#pragma unroll
    for (int i = 0; i < kTcStages; ++i) mbar_init(&sm.bar[i], 1);
    fence_mbar_init();
  }
  int32_t* ub = reinterpret_cast<int32_t*>(smem_raw + sizeof(TcWarpSmem) * kTcWarps);
  // fused append: units of this CTA (in order) whose rows are written
  int32_t* app_done = ub + kMaxBatch + 1 + 32;
  if (threadIdx.x == 0) *app_done = 0;
  // With early inputs the plan and the first units' page numbers are read
  // before the wait on the previous kernel (gw_set_early_inputs).
  const bool early = a.early_inputs != 0;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  local_plan<T::kChunk>(a, ub, !early);
  const int total_units = ub[a.batch];
  if (total_units > a.max_units) {
    if (early) pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(a.status, GW_DEV_WORKSPACE);
    return;
  }
  if (warp == kTcWarps) {
    // ---- fused append (launched only with one): the step's K/V row of each
    // (sequence, KV head) whose last chunk this CTA decodes (local_append.cuh);
    // the decode warp of such a unit waits for it before copying the unit's
    // last page.
    local_append_warp<GW_KV_BF16>(a, ub, total_units, app_done, early);
    return;
  }
  const int n_active = active_warps(total_units, kTcWarps);
  if (warp >= n_active) return;
  const uint64_t pol = policy_evict_first();
  const int n_warps = gridDim.x * n_active;
  int next_u = warp * gridDim.x + blockIdx.x;
  constexpr int kRing = kTcStages + 2;

  int f_slot = 0, f_i = 0;
  bool f_done = false, have_next = false;
  uint32_t issued = 0, consumed = 0;
  // Lane i holds the physical page of page i of the unit being issued (cur)
  // and of the unit after it (nxt).  A unit's page numbers are loaded when
  // the unit before it starts issuing, so no stage issue waits for a load.
  int32_t pg_cur = -1, pg_nxt = -1;

  auto grab = [&](int slot, int32_t& pg) -> bool {
    const int u = next_u;
    next_u += n_warps;
    if (u >= total_units) return false;
    const Unit d = decode_unit<T>(a, ub, u);
    if (lane == 0) sm.ring[slot] = d;
    pg = lane < d.n ? a.block_table[static_cast<int64_t>(d.s) * a.max_pages + d.hp_lo + lane] : -1;
    __syncwarp();
    return true;
  };

  auto issue = [&]() {
    const Unit d = sm.ring[f_slot];
    const int st = issued % kTcStages;
    const int32_t phys = __shfl_sync(0xffffffffu, pg_cur, f_i);  // one page per stage
    if (a.k_new && d.last && f_i == d.n - 1) {
      // the page holding the step's row: wait until the append warp wrote it
      if (lane == 0)
        wait_counter(app_done, (d.unit - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1, a.status);
      __syncwarp();
      fence_proxy_async_global();
    }
    if (phys < 0 || phys >= a.num_pages) {
      if (lane == 0) {
        sm.valid[st] = 0;
        set_status(a.status, GW_DEV_PAGE_RANGE);
        mbar_arrive(&sm.bar[st]);
      }
    } else {
      if (lane == 0) {
        sm.valid[st] = 1;
        mbar_arrive_expect_tx(&sm.bar[st], kTcStage);
      }
      __syncwarp();
      if (lane < 4)  // lane: 64-dim chunk; K and V rows of the page head in one box
        tma_rows(smem_u32(sm.stage[st]) + lane * 4096, &kv_map, lane, (phys * a.kv_heads + d.g) * 2 * kPage,
                 &sm.bar[st], pol);
    }
    ++issued;
    if (++f_i == d.n) {
      f_i = 0;
      f_slot = (f_slot + 1) % kRing;
      f_done = !have_next;
      if (have_next) {
        pg_cur = pg_nxt;
        have_next = grab((f_slot + 1) % kRing, pg_nxt);
      }
    }
  };

  f_done = !grab(0, pg_cur);
  if (!f_done) have_next = grab(1, pg_nxt);
  if (early) {
    // Warm L2 with the first unit's first pages (K and V of the unit's KV
    // head, 16 KB each) while the previous kernel finishes: a prefetch only
    // fills L2, which that kernel's writes (the append of the sequence's
    // last row) keep coherent; the copies to shared memory follow the wait.
    if (!f_done && lane < kTcStages && pg_cur >= 0 && pg_cur < a.num_pages)
      prefetch_l2(a.pool + ((static_cast<int64_t>(pg_cur) * a.kv_heads + sm.ring[0].g) * 2) * kPage * 512, kTcStage);
    pdl_wait();
    pdl_trigger();
    publish_plan(a, ub, threadIdx.x, n_active * 32);
  }
  while (!f_done && issued - consumed < kTcStages) issue();

  const int hq = lane >> 2;        // S row (q head of the group) this lane holds
  const int kq = (lane & 3) * 2;   // first of its two S columns in each token half
  uint32_t qa[16][2];              // A fragments of Q: dims 16s + kq + {0,1} and 16s + 8 + kq + {0,1}
  float o[16][4];                  // O^T: dims 16j + lane/4 (+8) x heads kq, kq + 1
  float m_ref = -INFINITY, lsum = 0.f;
  int c_slot = 0, c_i = 0;
  while (consumed < issued) {
    const Unit d = sm.ring[c_slot];
    if (c_i == 0) {
      if (hq < G) {
        const uint32_t* qrow =
            reinterpret_cast<const uint32_t*>(a.q + (static_cast<int64_t>(d.row) * a.num_q_heads + d.g * G + hq) * 256);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          qa[s][0] = qrow[(16 * s + kq) >> 1];
          qa[s][1] = qrow[(16 * s + 8 + kq) >> 1];
        }
      } else {
#pragma unroll
        for (int s = 0; s < 16; ++s) qa[s][0] = qa[s][1] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      m_ref = -INFINITY;
      lsum = 0.f;
    }
    const int st = consumed % kTcStages;
    if (!mbar_wait(&sm.bar[st], (consumed / kTcStages) & 1, a.status)) {
      for (uint32_t k = consumed + 1; k < issued; ++k) mbar_wait(&sm.bar[k % kTcStages], (k / kTcStages) & 1, nullptr);
      return;
    }
    const uint32_t kb = smem_u32(sm.stage[st]), vb = kb + 2048;  // chunk c: + 4096 c
    const int t0 = (d.hp_lo + c_i) * kTok;
    const bool stage_ok = sm.valid[st] != 0;

    // ---- S = Q . K^T for the two 8-token halves
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) {  // 32 dims: chunk s2 / 2, units (s2 % 2) * 4 + 0..3
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t b[4];
        const int row = h * 8 + (lane & 7);
        ldsm4(kb + (s2 >> 1) * 4096 + sw128(row, (s2 & 1) * 4 + (lane >> 3)), b);
        hmma_q(sacc[h], qa[2 * s2][0], qa[2 * s2][1], b[0], b[1]);
        hmma_q(sacc[h], qa[2 * s2 + 1][0], qa[2 * s2 + 1][1], b[2], b[3]);
      }
    }

    // ---- online softmax (base 2) against a lazily raised reference max
    float sv[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tk = t0 + h * 8 + kq + e;
        const bool ok = stage_ok && hq < G && tk >= d.tok_lo && tk < d.tok_hi;
        sv[h][e] = ok ? sacc[h][e] * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sv[h][e]);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const bool raise = mx > m_ref + 8.f;
    if (__any_sync(0xffffffffu, raise)) {
      const float m_new = raise ? mx : m_ref;
      const float alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new);
      m_ref = m_new;
      lsum *= alpha;
      const float aa = __shfl_sync(0xffffffffu, alpha, (lane & 3) * 8);
      const float ab = __shfl_sync(0xffffffffu, alpha, (lane & 3) * 8 + 4);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= aa;
        o[j][1] *= ab;
        o[j][2] *= aa;
        o[j][3] *= ab;
      }
    }
    uint32_t pb[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      pb[h] = pack2_bf16(sv[h][0] == -INFINITY ? 0.f : ex2(sv[h][0] - m_ref),
                         sv[h][1] == -INFINITY ? 0.f : ex2(sv[h][1] - m_ref));
      lsum += __uint_as_float(pb[h] << 16) + __uint_as_float(pb[h] & 0xFFFF0000u);
    }

    // ---- O^T += V^T . P^T; V rows of tokens outside the unit are cleared
    // first (their bytes may be anything, even NaN patterns)
    if (stage_ok) {
      if (t0 < d.tok_lo || t0 + kTok > d.tok_hi) {
        for (int r = 0; r < kTok; ++r) {
          if (t0 + r >= d.tok_lo && t0 + r < d.tok_hi) continue;
          *reinterpret_cast<uint4*>(sm.stage[st] + 2048 + (lane >> 3) * 4096 + r * 128 + (lane & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // ordered before the next TMA into this stage
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {  // dims 16j..16j+15: chunk j / 4, units (j % 4) * 2 + {0, 1}
        uint32_t v[4];
        const int m = lane >> 3;
        const int row = (m >> 1) * 8 + (lane & 7);
        ldsm4_t(vb + (j >> 2) * 4096 + sw128(row, (j & 3) * 2 + (m & 1)), v);
        hmma(o[j], v, pb[0], pb[1]);
      }
    }
    __syncwarp();
    ++consumed;
    if (++c_i == d.n) {
      // ---- unit done: write the unnormalised partial (m, l, o)
      float l = lsum + __shfl_xor_sync(0xffffffffu, lsum, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if ((lane & 3) == 0 && hq < G) a.part_ml[static_cast<int64_t>(d.unit) * G + hq] = make_float2(m_ref, l);
      float* po = a.part_o + static_cast<int64_t>(d.unit) * G * 256 + (lane >> 2);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (kq < G) {
          po[kq * 256 + 16 * j] = o[j][0];
          po[kq * 256 + 16 * j + 8] = o[j][2];
        }
        if (kq + 1 < G) {
          po[(kq + 1) * 256 + 16 * j] = o[j][1];
          po[(kq + 1) * 256 + 16 * j + 8] = o[j][3];
        }
      }
      c_i = 0;
      c_slot = (c_slot + 1) % kRing;
    }
    while (!f_done && issued - consumed < kTcStages) issue();
  }
}

template <int G>
cudaError_t launch_tc(const LocalArgs& a, cudaStream_t st) {
  CUtensorMap map;
  cudaError_t e = make_local_kv_map(a, &map, GW_KV_BF16, 32);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(TcWarpSmem) * kTcWarps + sizeof(int32_t) * (kMaxBatch + 1 + 32 + 4);
  auto kern = local_decode_tc_kernel<G>;
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid_ctas()), dim3(kTcWarps * 32 + (a.k_new ? 32 : 0)), smem, st, a, map);
  if (e != cudaSuccess) return e;
  // the merged partials are dropped from L2 unwritten: their write-back no
  // longer competes with the next layers' streams (serving step 0.2873 vs
  // 0.2936 ms, measured)
  return launch_combine(a, G, 256, local_max_chunks(a.max_pages, a.window, TcTraits::kChunk), true, st);
}

}  // namespace

cudaError_t launch_local_decode(int dtype, int group, const LocalArgs& a, cudaStream_t st) {
  if (dtype != GW_KV_BF16) return launch_local_decode_e4m3_tc(group, a, st);
  switch (group) {
    case 1: return launch_tc<1>(a, st);
    case 2: return launch_tc<2>(a, st);
    case 4: return launch_tc<4>(a, st);
    case 8: return launch_tc<8>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gw
