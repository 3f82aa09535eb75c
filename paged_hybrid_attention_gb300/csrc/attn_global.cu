// Global decode attention on the tensor cores (tcgen05 / TMEM), head dim 512,
// one KV head shared by all q heads.
//
// "Gemma 4" (pegainfer model page), "Architecture notes": global layers have a
// single KV head of dim 512; K and V come from one projection, K through
// k_norm and RoPE on 128 of the 512 dims.  "Gewell - Gemma4 inference
// engine", "the Why": so a token can be cached as V plus the rotated K slice
// (0.625x of K+V) and K rebuilt for the math.  Here that rebuild costs
// nothing: the folded pages in shared memory hold V[0:512] and k_rot[0:128]
// as 8x8 core matrices, and the QK^T contraction simply points its
// K-dimension descriptors at k_rot for dims [0,128) and at V for dims
// [128,512) - the same V bytes then feed P.V.
//
// All q heads share one KV head, so per 64-token tile the work is two real
// dense contractions (~51 flop per KV byte):
//   S^T[64 tok x HQ] = K_tile[64 x 512] . Q^T     (UMMA M=64, N=HQ, K=512: 32 MMAs)
//   O^T[512 x HQ]   += V_tile^T[512 x 64] . P^T   (UMMA M=128 x4 per page, K=16)
// with fp32 accumulators in tensor memory.
//
// A tile's four pages sit in page slots that are released one by one: P.V
// commits each page's MMAs to that slot's barrier and the producer refills
// the slot at once.  The folded layout double-buffers its tiles, so one tile
// streams in while the other is computed; the full K+V control layout, whose
// pages are 1.6x larger, has room for one tile only; the e4m3 folded layout,
// whose pages are half the size, keeps three tiles in flight.
//
// On the e4m3 folded pool the same contractions run as kind::f8f6f4 MMAs
// straight on the stored tiles (K = 32 per MMA): q enters as two e4m3 terms
// [q_hi; q_lo] stacked along N (one MMA of N = 2 HQ per K-step, the softmax
// adds the two logit columns), and P as two e4m3 terms accumulated into O by
// two MMAs per K-step.  (One 128-token tile of
// eight slots halves the MMAs per byte but leaves nothing streaming during
// QK^T and the softmax, and was slower.)
//
// Warp roles (256 threads, one persistent CTA per SM):
//   warps 0-3  softmax + epilogue: warp w owns TMEM lanes [32w, 32w+32), i.e.
//              tokens [16w, 16w+16) of the tile (the M=64 accumulator uses
//              lanes 0-15 of each 32-lane quadrant) and dims of O^T.
//   warp 4     producer: walks the CTA's split-KV units (sequence, chunk of
//              pages; dealt round-robin from the in-kernel plan).  Lane j owns
//              page slot j of each buffer: it fetches its page number of the
//              next tile early, waits for its slot and issues the page's bulk
//              copy.
//   warp 5     QK^T issue and TMEM owner.
//   warp 6     loads each unit's q rows into the K-major Q operand as soon as
//              the previous unit's last QK^T has completed, and prefetches
//              the next unit's rows into L2.
//   warp 7     P.V issue.
// With a fused append (gw_append_decode_attn_global) warp 6 also writes the
// step's row of each sequence whose last chunk this CTA decodes, one unit
// ahead of its q loads (the first unit's right after that unit's q); the
// producer waits for it before copying the tile that holds the sequence's
// last page.  (A ninth warp for it would cap the
// kernel at 168 registers, and the softmax's spills cost long contexts more
// than the separate append: 245 vs 238-240 us per long-context call.)
// QK^T and P.V are issued by different warps so that QK^T of the next tile
// never waits behind the softmax of the current one.
#include "append_row.cuh"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace gw {
namespace {

constexpr int kThreads = 256;
constexpr int kTilePages = 4;  // 64 tokens = UMMA M of QK^T
constexpr int kRing = 4;       // tile descriptors in flight
constexpr float kLazyThreshold = 8.f;

// Page geometry per layout.  Every layout stores 8-token x 16-byte blocks
// (8 bf16 or 16 e4m3 elements per block row); kBlk is the number of such
// column blocks per 8-token block.  A QK^T K-step covers 16 dims (bf16) or
// 32 dims (e4m3), i.e. two column blocks either way.
template <int LAYOUT>
struct GTraits;
template <>
struct GTraits<GW_LAYOUT_GLOBAL_FOLDED> {
  static constexpr bool kE4 = false;
  static constexpr int kPageBytes = 20480;
  static constexpr int kBlk = 80;   // 16-byte column blocks per 8-token block
  static constexpr int kNumBuf = 2;  // tile buffers
  static constexpr int kVcb = 0;    // column block of V dim 0
  static constexpr int kKSteps = 32;
  // column block holding K dims [16 ks, 16 ks + 16)
  __device__ static int k_cb(int ks) { return ks < 8 ? 64 + 2 * ks : 2 * ks; }
};
template <>
struct GTraits<GW_LAYOUT_GLOBAL_FULL> {
  static constexpr bool kE4 = false;
  static constexpr int kPageBytes = 32768;
  static constexpr int kBlk = 128;
  static constexpr int kNumBuf = 1;
  static constexpr int kVcb = 64;
  static constexpr int kKSteps = 32;
  __device__ static int k_cb(int ks) { return 2 * ks; }
};
template <>
struct GTraits<GW_LAYOUT_GLOBAL_FOLDED_E4M3> {
  static constexpr bool kE4 = true;
  static constexpr int kPageBytes = 10240;
  static constexpr int kBlk = 40;
  static constexpr int kNumBuf = 3;
  static constexpr int kVcb = 0;
  static constexpr int kKSteps = 16;
  // column block holding K dims [32 ks, 32 ks + 32): k_rot (elements
  // 512..639, blocks 32..39) for dims 0..127, V for dims 128..511
  __device__ static int k_cb(int ks) { return ks < 4 ? 32 + 2 * ks : 2 * ks; }
};

struct TileDesc {
  int32_t unit, s, q_row, L;
  int32_t tok0;   // absolute position of the tile's first token
  int32_t flags;  // bit0 first tile of unit, bit1 last tile, bit2 end; bits 8.. page valid
  int32_t pad[2];
};
constexpr int kFirst = 1, kLast = 2, kEnd = 4;

template <int LAYOUT, int HQ>
struct GSmem {
  using T = GTraits<LAYOUT>;
  static constexpr int kNP = HQ < 16 ? 16 : HQ;  // P.V N (M=128 needs N % 16 == 0)
  // One Q buffer, written once the previous unit's last QK^T has completed.
  // (The e4m3 pool spends the room a second buffer would take on a third
  // tile buffer: 198 vs 216 us per 8 x 131072-token call.  Its loader stages
  // and scales the next unit's q before waiting for the buffer.)
  static constexpr int kQBuf = 1;
  // bf16: K-major Q [hb][cb 64][8 heads][8 dims].  e4m3: the hi term then
  // the lo term, each K-major [hb][cb 32][8 heads][16 dims].
  static constexpr int kQBytes = HQ * 512 * 2;
  // bf16: MN-major P^T [tb 8][hb 8-head blocks][8 tokens][8 heads].  e4m3:
  // the hi term then the lo term, each [tb 8][16-head blocks][8 tokens][16 heads].
  static constexpr int kPBytes = 64 * kNP * 2;
  uint8_t tiles[T::kNumBuf][kTilePages][T::kPageBytes];
  uint8_t q[kQBuf][kQBytes];
  uint8_t p[2][kPBytes];
  float red[4][32];            // per-warp head reductions
  float mvec[32];              // reference max per head (log2 units)
  float qscale[4][32];         // e4m3: per unit (mod 4), per head: 2^-e of q's scaling
  // e4m3: the unit's bf16 q rows staged for conversion, rows padded by 16 B
  // so that the 8 heads a conversion step reads sit in different banks
  static constexpr int kStageRow = 1040;
  uint8_t qstage[T::kE4 ? HQ * kStageRow : 16];
  TileDesc ring[kRing];
  uint64_t full[T::kNumBuf], slot_empty[T::kNumBuf][kTilePages];
  uint64_t s_ready[2], p_ready[2], pfree[2], o_done[2], o_free[2], q_ready[2], q_free[2], qs_ready[4];
  uint32_t tmem_base;
  int32_t flag[2];  // per tile parity: index + 1 of the last tile that asked for a new max
  int32_t app_done;  // fused append: units of this CTA (in order) whose rows are written
  int32_t ub[kMaxBatch + 1 + 32];  // split plan (+ scan scratch)
};
static_assert(sizeof(GSmem<GW_LAYOUT_GLOBAL_FOLDED, 32>) <= 232448, "shared memory of one CTA");
static_assert(sizeof(GSmem<GW_LAYOUT_GLOBAL_FULL, 32>) <= 232448, "shared memory of one CTA");
static_assert(sizeof(GSmem<GW_LAYOUT_GLOBAL_FOLDED_E4M3, 32>) <= 232448, "shared memory of one CTA");

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded wait whose outcome is the same for every lane of the warp (the
// warp-uniform MMA issue must never diverge).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}

// Adds `bytes` to the transaction count the current phase of `bar` waits for
// (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Per-head reduction over the 32 lanes of a warp by a transposing fold: at
// each level a lane keeps half of its heads and merges the partner's copy of
// them.  Returns head (lane & (HQ-1)) reduced over all lanes; x is consumed.
template <int N, bool kMax>
__device__ __forceinline__ void head_fold(float* x, int lane) {
  if constexpr (N > 1) {
    constexpr int H = N / 2;
    const bool up = lane & H;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float send = up ? x[i] : x[i + H];
      const float keep = up ? x[i + H] : x[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, H);
      x[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
    head_fold<H, kMax>(x, lane);
  }
}
template <int HQ, bool kMax>
__device__ __forceinline__ float head_reduce(float (&x)[HQ], int lane) {
  head_fold<HQ, kMax>(x, lane);
  float v = x[0];
#pragma unroll
  for (int o = HQ; o < 32; o <<= 1) {
    const float r = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, r) : v + r;
  }
  return v;
}

// The fused append, by the q-loader warp: the row of the CTA's j-th unit if
// that unit is its sequence's last chunk, at position L - 1, with
// gw_kv_append's arithmetic; then the CTA's count of appended units becomes
// j + 1 (a release store the producer acquires).
template <int LAYOUT>
__device__ __noinline__ void append_unit_row(const LocalArgs& a, const int32_t* ub, int32_t* app_done, int j,
                                             int total_units) {
  using R = GlobalRow<LAYOUT>;
  const int lane = threadIdx.x & 31;
  const int u = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
  if (u < total_units) {
    const int s = plan_seq(ub, a.batch, u);
    if (u - ub[s] == ub[s + 1] - ub[s] - 1) {  // the sequence's last chunk
      const int pos = a.seq_lens[s] - 1;
      const int32_t page = a.block_table[static_cast<int64_t>(s) * a.max_pages + pos / kPage];
      if (pos >= a.max_pos) {
        if (lane == 0) set_status(a.status, GW_DEV_POS_RANGE);
      } else if (page >= 0 && page < a.num_pages) {  // else the producer reports the page
        const int64_t row = a.cu_q_rows[s];
        for (int it = lane; it < R::kItems; it += 32) {
          const int rt = R::rot_item(it);
          const CosSin8 cs =
              rt >= 0 ? load_cs8(a.rope_cs + (static_cast<int64_t>(pos) * 64 + 8 * rt) * 2) : CosSin8{};
          append_global_item<LAYOUT>(const_cast<uint8_t*>(a.pool), page, pos % kPage, a.k_new + row * 512,
                                     a.v_new + row * 512, cs, it);
        }
        fence_proxy_async_global();
      }
    }
  }
  __syncwarp();
  if (lane == 0) st_release_shared(app_done, j + 1);
}

// kApp: the fused-append variant (a kernel of its own, so that the plain
// call's code is unchanged).
template <int LAYOUT, int HQ, bool kApp>
__global__ void __launch_bounds__(kThreads, 1) global_decode_kernel(const LocalArgs a) {
  using T = GTraits<LAYOUT>;
  using SM = GSmem<LAYOUT, HQ>;
  constexpr int NB = T::kNumBuf;
  constexpr int NP = SM::kNP;
  constexpr bool kE4 = T::kE4;
  constexpr int QB = SM::kQBuf;
  constexpr uint32_t kTileBytes = kTilePages * T::kPageBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  int32_t* st = a.status;

  // Stale tile / P slots must hold finite values: masked tokens get p = 0 and
  // 0 * finite = 0 in the P.V contraction.
  {
    uint4* z = reinterpret_cast<uint4*>(sm.tiles);
    for (int i = tid; i < static_cast<int>(sizeof(sm.tiles) / 16); i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(sm.p);
    for (int i = tid; i < static_cast<int>(sizeof(sm.p) / 16); i += kThreads) zp[i] = make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    sm.app_done = 0;
    for (int b = 0; b < NB; ++b) {
      mbar_init(&sm.full[b], 1);
      for (int j = 0; j < kTilePages; ++j) mbar_init(&sm.slot_empty[b][j], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_ready[b], 1);
      mbar_init(&sm.p_ready[b], 128);
      mbar_init(&sm.pfree[b], 1);
      mbar_init(&sm.o_done[b], 1);
      mbar_init(&sm.o_free[b], 128);
      sm.flag[b] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_ready[b], 1);
      mbar_init(&sm.q_free[b], 1);
    }
    for (int b = 0; b < 4; ++b) mbar_init(&sm.qs_ready[b], 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::alloc(&sm.tmem_base, 512);
    tc::relinquish();
  }
  // With early inputs the plan and the producer's first page numbers are
  // read before the wait on the previous kernel (gw_set_early_inputs); every
  // role then waits before its first access to pages, q or the workspace.
  const bool early = a.early_inputs != 0;
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  plan_in_smem(a, sm.ub, sm.ub + kMaxBatch + 1, [](int L) { return global_chunks(L); }, !early);
  const int total_units = sm.ub[a.batch];
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
  // TMEM columns: S^T buffers at 0 and kSCols; O^T buffers at kOBase and
  // kOBase + 128 (4 blocks of 32).  bf16: S^T is 64 x HQ (kSCols 32).  e4m3:
  // S^T is 64 x 2HQ, the logits against q_hi then against q_lo (kSCols 64).
  constexpr uint32_t kSCols = kE4 ? 64 : 32;
  constexpr uint32_t kOBase = 2 * kSCols;
  if (total_units > a.max_units) {  // uniform
    wait_prev();
    if (blockIdx.x == 0 && tid == 0) set_status(st, GW_DEV_WORKSPACE);
  } else if (warp == 4) {
    // ------------------------------------------------------------- producer
    const uint64_t pol = policy_evict_first();
    int u = blockIdx.x;
    int s = 0, p0 = 0, p1 = 0, ntiles = 0, q_row = 0, L = 0, t = 0;
    auto unit_info = [&]() {
      s = plan_seq(sm.ub, a.batch, u);
      L = a.seq_lens[s];
      q_row = a.cu_q_rows[s];
      const int cpg = global_chunk_pages(L);
      p0 = (u - sm.ub[s]) * cpg;
      p1 = min(p0 + cpg, (L + kPage - 1) / kPage);
      ntiles = (p1 - p0 + kTilePages - 1) / kTilePages;
    };
    // lane j < 4: physical page of page j of tile t (raw; checked after the
    // slot wait so that the load's latency hides behind it)
    auto fetch_page = [&](bool& in_unit) -> int32_t {
      const int lp = p0 + t * kTilePages + lane;
      in_unit = lane < kTilePages && lp < p1;
      return in_unit ? a.block_table[static_cast<int64_t>(s) * a.max_pages + lp] : -1;
    };
    bool end = u >= total_units;
    if (!end) unit_info();
    bool in_unit = false;
    int32_t pg = end ? -1 : fetch_page(in_unit);
    if (early && !end) {
      // Warm L2 with the first two tiles' pages while the previous kernel
      // finishes.  A prefetch only fills L2, which the previous kernel's
      // writes (the append of the sequence's last row) keep coherent, so it
      // may run before the wait; the copies to shared memory come after it.
      const int lp = p0 + lane;
      if (lane < 2 * kTilePages && lp < p1) {
        const int32_t pp = a.block_table[static_cast<int64_t>(s) * a.max_pages + lp];
        if (pp >= 0 && pp < a.num_pages) prefetch_l2(a.pool + static_cast<int64_t>(pp) * T::kPageBytes, T::kPageBytes);
      }
    }
    wait_prev();
    for (uint32_t n = 0;; ++n) {
      const int b = n % NB;
      const uint32_t k = n / NB;  // use of buffer b
      bool waited = true, ok = false;
      if (kApp && !end && t == ntiles - 1 && p1 * kPage >= L) {
        // the tile holds the step's row, which the append warp writes
        if (lane == 0)
          wait_counter(&sm.app_done, (u - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1, st);
        __syncwarp();
        fence_proxy_async_global();
      }
      if (lane < kTilePages) {
        // This lane's slot is free once P.V of the buffer's previous tile has
        // read it.  That P.V followed the softmax of that tile, so the
        // previous phase of full[b] is complete before this tile adds to it
        // (the end marker waits too, so its arrival never lands on an open
        // phase).
        if (k > 0) waited = mbar_wait(&sm.slot_empty[b][lane], (k - 1) & 1, st);
        ok = !end && waited && in_unit && pg >= 0 && pg < a.num_pages;
        if (!end && waited && in_unit && !ok) set_status(st, GW_DEV_PAGE_RANGE);
        if (ok) {
          mbar_expect_tx(&sm.full[b], T::kPageBytes);
          bulk_g2s(sm.tiles[b][lane], a.pool + static_cast<int64_t>(pg) * T::kPageBytes, T::kPageBytes,
                   &sm.full[b], pol);
        }
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, ok);
      if (__any_sync(0xffffffffu, !waited)) break;
      if (lane == 0) {
        TileDesc d{};
        if (end) {
          d.flags = kEnd;
        } else {
          d.unit = u;
          d.s = s;
          d.q_row = q_row;
          d.L = L;
          d.tok0 = (p0 + t * kTilePages) * kPage;
          d.flags = (t == 0 ? kFirst : 0) | (t == ntiles - 1 ? kLast : 0) | static_cast<int>(mask << 8);
        }
        sm.ring[n % kRing] = d;
        mbar_arrive(&sm.full[b]);  // after every expect_tx of this tile (ordered by the votes above)
      }
      if (end) break;
      if (++t == ntiles) {
        t = 0;
        u += gridDim.x;
        end = u >= total_units;
        if (!end) unit_info();
      }
      pg = end ? -1 : fetch_page(in_unit);
      if (end) in_unit = false;
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- QK^T issue
    wait_prev();
    // The whole warp runs this loop with warp-uniform values; elect.sync
    // picks the issuing lane inside mma_bf16_warp / commit_warp.
    // e4m3: one MMA per K-step against [q_hi; q_lo] (N = 2 HQ: the lo term's
    // head blocks follow the hi term's at the same 8-head stride)
    const uint32_t id_qk = kE4 ? tc::idesc_e4m3(64, 2 * HQ, false, false) : tc::idesc_bf16(64, HQ, false, false);
    // descriptor bases; the start-address field is addr >> 4 in the low bits,
    // so a byte offset o is added as o >> 4 (all addresses stay below 256 KiB).
    // Q: 16-byte block rows, the next 8 heads (kQBytes / 2 / (HQ / 8)) apart
    // within a term.
    const uint64_t qk_a0 = tc::smem_desc(smem_u32(sm.tiles[0]), 128, T::kBlk * 128);
    const uint64_t qk_b0 = tc::smem_desc(smem_u32(sm.q[0]), 128, kE4 ? 32 * 128 : 64 * 128);
    int uidx = -1, qb = 0;
    for (uint32_t n = 0;; ++n) {
      const int b = n % NB;
      if (!warp_wait(&sm.full[b], (n / NB) & 1, st)) break;
      const TileDesc d = sm.ring[n % kRing];
      if (d.flags & kEnd) break;
      if (d.flags & kFirst) {
        ++uidx;
        qb = uidx % QB;
        if (!warp_wait(&sm.q_ready[qb], (uidx / QB) & 1, st)) break;
      }
      // S^T buffer n & 1 is free once the softmax of tile n - 2 has read it
      if (n >= 2 && !warp_wait(&sm.p_ready[n & 1], ((n >> 1) - 1) & 1, st)) break;
      tc::fence_after();
      const uint64_t a_tile = qk_a0 + ((b * kTileBytes) >> 4);
      const uint64_t q_base = qk_b0 + ((qb * SM::kQBytes) >> 4);
      const uint32_t d_s = tmem + kSCols * (n & 1);
#pragma unroll
      for (int ks = 0; ks < T::kKSteps; ++ks) {
        const uint64_t ad = a_tile + ((T::k_cb(ks) * 128) >> 4);
        const uint64_t bd = q_base + ((2 * ks * 128) >> 4);
        if constexpr (kE4) {
          tc::mma_e4m3_warp(d_s, ad, bd, id_qk, ks > 0);
        } else {
          tc::mma_bf16_warp(d_s, ad, bd, id_qk, ks > 0);
        }
      }
      tc::commit_warp(&sm.s_ready[n & 1]);
      if (d.flags & kLast) tc::commit_warp(&sm.q_free[qb]);  // Q buffer qb may be replaced once this completes
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ P.V issue
    wait_prev();
    const uint32_t id_pv = kE4 ? tc::idesc_e4m3(128, NP, true, true) : tc::idesc_bf16(128, NP, true, true);
    const uint64_t pv_a0 = tc::smem_desc(smem_u32(sm.tiles[0]), T::kBlk * 128, 128);
    // P^T: 8-token block rows (NP / 8 or NP / 16 head blocks of 16 bytes) apart
    const uint64_t pv_b0 = tc::smem_desc(smem_u32(sm.p[0]), (kE4 ? NP / 16 : NP / 8) * 128, 128);
    int ui = -1;
    for (uint32_t n = 0;; ++n) {
      const int b = n % NB;
      if (!warp_wait(&sm.full[b], (n / NB) & 1, st)) break;
      const TileDesc d = sm.ring[n % kRing];
      if (d.flags & kEnd) break;
      if (d.flags & kFirst) ++ui;
      if (!warp_wait(&sm.p_ready[n & 1], (n >> 1) & 1, st)) break;
      const int ob = ui & 1;
      if ((d.flags & kFirst) && ui >= 2 && !warp_wait(&sm.o_free[ob], ((ui >> 1) - 1) & 1, st)) break;
      tc::fence_after();
      const uint64_t a_tile = pv_a0 + ((b * kTileBytes) >> 4);
      const uint64_t b_p = pv_b0 + (((n & 1) * SM::kPBytes) >> 4);
      if constexpr (kE4) {
        // K = 32 tokens per MMA: pages 2j and 2j + 1; O^T += V^T (P_hi + P_lo)^T
#pragma unroll
        for (int j = 0; j < kTilePages / 2; ++j) {
          const uint64_t bd = b_p + ((4 * j * (NP / 16) * 128) >> 4);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint64_t ad = a_tile + ((2 * j * T::kPageBytes + (T::kVcb + 8 * blk) * 128) >> 4);
            const uint32_t d_o = tmem + kOBase + 128 * ob + 32 * blk;
            tc::mma_e4m3_warp(d_o, ad, bd, id_pv, !((d.flags & kFirst) && j == 0));
            tc::mma_e4m3_warp(d_o, ad, bd + ((64 * NP) >> 4), id_pv, true);
          }
          tc::commit_warp(&sm.slot_empty[b][2 * j]);  // the producer may refill these page slots
          tc::commit_warp(&sm.slot_empty[b][2 * j + 1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kTilePages; ++j) {
          const uint64_t bd = b_p + ((2 * j * (NP / 8) * 128) >> 4);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint64_t ad = a_tile + ((j * T::kPageBytes + (T::kVcb + 16 * blk) * 128) >> 4);
            tc::mma_bf16_warp(tmem + kOBase + 128 * ob + 32 * blk, ad, bd, id_pv, !((d.flags & kFirst) && j == 0));
          }
          tc::commit_warp(&sm.slot_empty[b][j]);  // the producer may refill this page slot
        }
      }
      tc::commit_warp(&sm.pfree[n & 1]);
      if (d.flags & kLast) tc::commit_warp(&sm.o_done[ob]);
    }
  } else if (warp == 6 && kE4) {
    // ------------------------------------------------- q loader, e4m3 pool
    wait_prev();
    // Unit k's q goes to the Q buffer once the last QK^T of unit k - 1 has
    // completed.  Each head is scaled by an exact power of two 2^e, chosen so
    // that its largest |q| lands in [128, 256), and split into two e4m3
    // terms, hi = e4m3(q 2^e) and lo = e4m3(q 2^e - hi); 2^-e goes to the
    // softmax, which scales the logits back.
    int k = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++k) {
      const int q_row = a.cu_q_rows[plan_seq(sm.ub, a.batch, u)];
      const int qb = k % SM::kQBuf;
      // stage the bf16 rows in shared memory: all copies in flight at once
      const uint16_t* gsrc = a.q + static_cast<int64_t>(q_row) * HQ * 512;
      __syncwarp();  // the previous unit's reads of the stage are done
      for (int c = lane; c < HQ * 64; c += 32) {
        const int h = c >> 6, c8 = c & 63;
        cp_async16(sm.qstage + h * SM::kStageRow + c8 * 16, gsrc + h * 512 + c8 * 8);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncwarp();
      auto srow = [&](int h) { return reinterpret_cast<const uint16_t*>(sm.qstage + h * SM::kStageRow); };
      // pass 1: largest |q| of each head (lane h keeps head h's)
      float my_scale = 1.f;
#pragma unroll 4
      for (int h = 0; h < HQ; ++h) {
        float x[8], y[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(srow(h) + 16 * lane), x);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(srow(h) + 16 * lane + 8), y);
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(x[i]), fabsf(y[i])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == h) {
          // e = 7 - floor(log2 m), clamped so that 2^e and 2^-e are normal floats
          const int ex = m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 : 7;
          const int e = min(125, max(-125, 7 - ex));
          my_scale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
          sm.qscale[k & 3][h] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        }
      }
      // the Q buffer is free once the last QK^T that read it has completed
      if (k >= SM::kQBuf && !warp_wait(&sm.q_free[qb], ((k / SM::kQBuf) - 1) & 1, st)) break;
      // pass 2: lane (h & 7, cb >> 2 ... ) converts 16 dims of one head; the 8
      // heads of a block go to 8 different 16-byte bank groups
      uint8_t* qhi = sm.q[qb];
      uint8_t* qlo = sm.q[qb] + HQ * 512;
#pragma unroll 1
      for (int hb = 0; hb < HQ / 8; ++hb) {
        const int h = 8 * hb + (lane & 7);
        const float sc = __shfl_sync(0xffffffffu, my_scale, h);
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const int cb = 4 * j + (lane >> 3);
          float x[16];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(srow(h) + 16 * cb), *reinterpret_cast<float(*)[8]>(x));
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(srow(h) + 16 * cb + 8), *reinterpret_cast<float(*)[8]>(x + 8));
          uint32_t whi[4], wlo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t hw = 0, lw = 0;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const float a0 = x[4 * i + 2 * jj] * sc, a1 = x[4 * i + 2 * jj + 1] * sc;
              const __nv_fp8x2_storage_t hi2 = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
              const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi2, __NV_E4M3)));
              const __nv_fp8x2_storage_t lo2 =
                  __nv_cvt_float2_to_fp8x2(make_float2(a0 - hf.x, a1 - hf.y), __NV_SATFINITE, __NV_E4M3);
              hw |= static_cast<uint32_t>(hi2) << (16 * jj);
              lw |= static_cast<uint32_t>(lo2) << (16 * jj);
            }
            whi[i] = hw;
            wlo[i] = lw;
          }
          const int off = ((h >> 3) * 32 + cb) * 128 + (h & 7) * 16;
          *reinterpret_cast<uint4*>(qhi + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
          *reinterpret_cast<uint4*>(qlo + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.q_ready[qb]);
        mbar_arrive(&sm.qs_ready[k & 3]);
        const int un = u + gridDim.x;
        if (un < total_units)
          prefetch_l2(a.q + static_cast<int64_t>(a.cu_q_rows[plan_seq(sm.ub, a.batch, un)]) * HQ * 512, HQ * 1024);
      }
      if (kApp) {  // after the unit's q is published: unit 0's row, then one unit ahead
        if (k == 0) append_unit_row<LAYOUT>(a, sm.ub, &sm.app_done, 0, total_units);
        append_unit_row<LAYOUT>(a, sm.ub, &sm.app_done, k + 1, total_units);
      }
    }
  } else if (warp == 6) {
    // -------------------------------------------------------------- q loader
    wait_prev();
    // Unit k's rows overwrite Q once the last QK^T of unit k - 1 has
    // completed (q_free); by then they are usually in L2 already.
    int k = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++k) {
      const int q_row = a.cu_q_rows[plan_seq(sm.ub, a.batch, u)];
      if (k > 0 && !warp_wait(&sm.q_free[0], (k - 1) & 1, st)) break;
      const uint16_t* src = a.q + static_cast<int64_t>(q_row) * HQ * 512;
      for (int c = lane; c < HQ * 64; c += 32) {
        const int h = c >> 6, cb = c & 63;
        cp_async16(sm.q[0] + (((h >> 3) * 64 + cb) * 128 + (h & 7) * 16), src + h * 512 + cb * 8);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.q_ready[0]);
        const int un = u + gridDim.x;
        if (un < total_units)
          prefetch_l2(a.q + static_cast<int64_t>(a.cu_q_rows[plan_seq(sm.ub, a.batch, un)]) * HQ * 512, HQ * 1024);
      }
      if (kApp) {  // after the unit's q is published: unit 0's row, then one unit ahead
        if (k == 0) append_unit_row<LAYOUT>(a, sm.ub, &sm.app_done, 0, total_units);
        append_unit_row<LAYOUT>(a, sm.ub, &sm.app_done, k + 1, total_units);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------- softmax + epilogue
    wait_prev();
    if (early) publish_plan(a, sm.ub, tid, 128);
    const bool active = lane < 16;
    const int t = 16 * warp + lane;  // token of the tile (active lanes)
    const int j = warp;              // page of the tile
    float m_run[HQ], l_acc[HQ];
#pragma unroll
    for (int h = 0; h < HQ; ++h) {
      m_run[h] = -INFINITY;
      l_acc[h] = 0.f;
    }
    int uidx = -1;
    for (uint32_t n = 0;; ++n) {
      const int b = n % NB;
      if (!mbar_wait(&sm.full[b], (n / NB) & 1, st)) break;
      const TileDesc d = sm.ring[n % kRing];
      if (d.flags & kEnd) break;
      const bool first = d.flags & kFirst;
      if (first) ++uidx;
      // e4m3: the unit's per-head descale of q is published with qs_ready
      if (kE4 && first && !mbar_wait(&sm.qs_ready[uidx & 3], (uidx >> 2) & 1, st)) break;
      if (!mbar_wait(&sm.s_ready[n & 1], (n >> 1) & 1, st)) break;
      tc::fence_after();
      uint32_t r[32];
      const uint32_t s_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16) + kSCols * (n & 1);
      tc::ld32(s_addr, r);
      if constexpr (kE4) {
        // logit = S(q_hi) + S(q_lo): columns h and HQ + h
        if constexpr (HQ == 32) {
          uint32_t r2[32];
          tc::ld32(s_addr + 32, r2);
          tc::wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) + __uint_as_float(r2[h]));
        } else {
          tc::wait_ld();
#pragma unroll
          for (int h = 0; h < HQ; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) + __uint_as_float(r[HQ + h]));
        }
      } else {
        tc::wait_ld();
      }
      const int tabs = d.tok0 + t;
      const bool pvalid = (d.flags >> (8 + j)) & 1;
      const bool valid = active && pvalid && tabs < d.L;
      float s[HQ];
      bool need = false;
#pragma unroll
      for (int h = 0; h < HQ; ++h) {
        const float sc = kE4 ? sm.qscale[uidx & 3][h] * a.scale_log2 : a.scale_log2;
        s[h] = valid ? __uint_as_float(r[h]) * sc : -INFINITY;
        need |= s[h] > m_run[h] + kLazyThreshold;
      }
      // A thread asking for a new max tags the flag of this tile's parity
      // with the tile; the other parity's flag may meanwhile be written for
      // the next tile (whose QK^T can complete before this softmax ends), and
      // this parity is not written again before every thread has passed the
      // barrier below on the next tile.
      if (need) sm.flag[n & 1] = static_cast<int32_t>(n + 1);
      softmax_bar();
      if (first || sm.flag[n & 1] == static_cast<int32_t>(n + 1)) {
        // ---- slow path: tile max per head, maybe rescale
        float x[HQ];
#pragma unroll
        for (int h = 0; h < HQ; ++h) x[h] = s[h];
        const float wmax = head_reduce<HQ, true>(x, lane);
        if (lane < HQ) sm.red[warp][lane] = wmax;
        softmax_bar();
        if (tid < HQ) {
          const float mx = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
          const float mo = first ? -INFINITY : sm.mvec[tid];
          sm.mvec[tid] = (first || mx > mo + kLazyThreshold) ? fmaxf(mo, mx) : mo;
        }
        softmax_bar();
        float alpha[HQ];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < HQ; ++h) {
          const float mn = sm.mvec[h];
          alpha[h] = (first || m_run[h] == -INFINITY) ? 0.f : ex2(m_run[h] - mn);
          rescale |= !first && mn != m_run[h];
          m_run[h] = mn;
          l_acc[h] = first ? 0.f : l_acc[h] * alpha[h];
        }
        if (rescale) {
          // O^T *= alpha per head column, once P.V of the previous tile is done
          if (!mbar_wait(&sm.pfree[(n - 1) & 1], ((n - 1) >> 1) & 1, st)) break;
          tc::fence_after();
          const uint32_t ob = uidx & 1;
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t ad = tmem + (static_cast<uint32_t>(32 * warp) << 16) + kOBase + 128 * ob + 32 * blk;
            uint32_t o[32];
            tc::ld32(ad, o);
            tc::wait_ld();
#pragma unroll
            for (int h = 0; h < HQ; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tc::st32(ad, o);
          }
          tc::wait_st();
        }
      }
      // ---- P^T (bf16) for this tile; wait until P.V two tiles back released the buffer
      if (n >= 2 && !mbar_wait(&sm.pfree[n & 1], ((n >> 1) - 1) & 1, st)) break;
      if (active && kE4) {
        // P = P_hi + P_lo, two e4m3 terms (P <= 2^8 under the lazy max); l
        // sums exactly the weights the contraction uses
        uint8_t* phi = sm.p[n & 1] + ((t >> 3) * (NP / 16)) * 128 + (t & 7) * 16;
        uint8_t* plo = phi + 64 * NP;
#pragma unroll
        for (int hb = 0; hb < NP / 16; ++hb) {
          uint32_t whi[4], wlo[4];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            uint32_t hw = 0, lw = 0;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int h0 = hb * 16 + 4 * k4 + 2 * jj;
              const int i0 = h0 < HQ ? h0 : 0, i1 = h0 + 1 < HQ ? h0 + 1 : 0;
              const float p0 = (valid && h0 < HQ) ? ex2(s[i0] - m_run[i0]) : 0.f;
              const float p1 = (valid && h0 + 1 < HQ) ? ex2(s[i1] - m_run[i1]) : 0.f;
              const __nv_fp8x2_storage_t hi2 = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
              const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi2, __NV_E4M3)));
              const __nv_fp8x2_storage_t lo2 =
                  __nv_cvt_float2_to_fp8x2(make_float2(p0 - hf.x, p1 - hf.y), __NV_SATFINITE, __NV_E4M3);
              const float2 lf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo2, __NV_E4M3)));
              if (h0 < HQ) l_acc[i0] += hf.x + lf.x;
              if (h0 + 1 < HQ) l_acc[i1] += hf.y + lf.y;
              hw |= static_cast<uint32_t>(hi2) << (16 * jj);
              lw |= static_cast<uint32_t>(lo2) << (16 * jj);
            }
            whi[k4] = hw;
            wlo[k4] = lw;
          }
          *reinterpret_cast<uint4*>(phi + hb * 128) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
          *reinterpret_cast<uint4*>(plo + hb * 128) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
        }
        if (pvalid && tabs >= d.L) {
          uint8_t* row = sm.tiles[b][j] + (lane >> 3) * T::kBlk * 128 + (lane & 7) * 16;
          for (int cb = 0; cb < T::kBlk; ++cb) *reinterpret_cast<uint4*>(row + cb * 128) = make_uint4(0, 0, 0, 0);
        }
      } else if (active) {
        uint8_t* pdst = sm.p[n & 1] + ((t >> 3) * (NP / 8)) * 128 + (t & 7) * 16;
#pragma unroll
        for (int hb = 0; hb < HQ / 8; ++hb) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int h0 = hb * 8 + 2 * k;
            const float p0 = valid ? ex2(s[h0] - m_run[h0]) : 0.f;
            const float p1 = valid ? ex2(s[h0 + 1] - m_run[h0 + 1]) : 0.f;
            __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            l_acc[h0] += __low2float(pb);
            l_acc[h0 + 1] += __high2float(pb);
            w[k] = *reinterpret_cast<uint32_t*>(&pb);
          }
          *reinterpret_cast<uint4*>(pdst + hb * 128) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (pvalid && tabs >= d.L) {
          // token past the end of the sequence in a valid page: clear its row
          // so whatever the pool holds there cannot reach P.V
          uint8_t* row = sm.tiles[b][j] + (lane >> 3) * T::kBlk * 128 + (lane & 7) * 16;
          for (int cb = 0; cb < T::kBlk; ++cb) *reinterpret_cast<uint4*>(row + cb * 128) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc::fence_before();
      mbar_arrive(&sm.p_ready[n & 1]);

      if (d.flags & kLast) {
        // ---- epilogue: unnormalised partial (m, l, o) of this unit
        const uint32_t ob = uidx & 1;
        if (!mbar_wait(&sm.o_done[ob], (uidx >> 1) & 1, st)) break;
        tc::fence_after();
        float* po = a.part_o + static_cast<int64_t>(d.unit) * HQ * 512;
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t o[32];
          tc::ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kOBase + 128 * ob + 32 * blk, o);
          tc::wait_ld();
          const int dim = 128 * blk + 32 * warp + lane;
#pragma unroll
          for (int h = 0; h < HQ; ++h) po[h * 512 + dim] = __uint_as_float(o[h]);
        }
        float x[HQ];
#pragma unroll
        for (int h = 0; h < HQ; ++h) x[h] = l_acc[h];
        const float wl = head_reduce<HQ, false>(x, lane);
        if (lane < HQ) sm.red[warp][lane] = wl;
        softmax_bar();
        if (tid < HQ) {
          const float l = ((sm.red[0][tid] + sm.red[1][tid]) + sm.red[2][tid]) + sm.red[3][tid];
          a.part_ml[static_cast<int64_t>(d.unit) * HQ + tid] = make_float2(sm.mvec[tid], l);
        }
        softmax_bar();
        tc::fence_before();
        mbar_arrive(&sm.o_free[ob]);
      }
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
cudaError_t launch_layout(const LocalArgs& a, cudaStream_t stream) {
  auto kern = a.k_new ? global_decode_kernel<LAYOUT, HQ, true> : global_decode_kernel<LAYOUT, HQ, false>;
  const size_t smem = sizeof(GSmem<LAYOUT, HQ>);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid_ctas()), dim3(kThreads), smem, stream, a);
  if (e != cudaSuccess) return e;
  // Dropping the merged partials from L2 unwritten pays for the folded pool
  // (24.7 vs 26.9 us per serving call) but not for the full control (427 vs
  // 415 us per long-context call), measured.
  return launch_combine(a, HQ, 512, global_max_chunks(a.max_pages), LAYOUT != GW_LAYOUT_GLOBAL_FULL, stream);
}

template <int LAYOUT>
cudaError_t launch_hq(const LocalArgs& a, cudaStream_t stream) {
  switch (a.num_q_heads) {
    case 8: return launch_layout<LAYOUT, 8>(a, stream);
    case 16: return launch_layout<LAYOUT, 16>(a, stream);
    case 32: return launch_layout<LAYOUT, 32>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_global_decode(int layout, const LocalArgs& a, cudaStream_t stream) {
  if (layout == GW_LAYOUT_GLOBAL_FOLDED_E4M3) return launch_hq<GW_LAYOUT_GLOBAL_FOLDED_E4M3>(a, stream);
  return layout == GW_LAYOUT_GLOBAL_FOLDED ? launch_hq<GW_LAYOUT_GLOBAL_FOLDED>(a, stream)
                                           : launch_hq<GW_LAYOUT_GLOBAL_FULL>(a, stream);
}

}  // namespace gw
