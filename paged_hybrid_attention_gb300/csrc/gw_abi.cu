// C-ABI entry points: host-side validation, workspace carving and dispatch.
//
// Nothing here allocates, frees or synchronises.  Each entry point checks its
// arguments, records a message naming itself on failure, and enqueues kernels
// on the caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "gw_internal.h"

namespace gw {
namespace {

thread_local char g_err[512] = "";

gw_status fail(gw_status code, const char* fn, const char* fmt, ...) {
  int n = std::snprintf(g_err, sizeof(g_err), "%s: ", fn);
  if (n < 0) n = 0;
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err + n, sizeof(g_err) - static_cast<size_t>(n), fmt, ap);
  va_end(ap);
  return code;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pool description checks shared by every entry point.
// `need_base` is false for the size queries, which may run before the pool
// memory exists.
gw_status check_pool(const gw_kv_pool* p, const char* fn, bool need_base = true) {
  if (!p) return fail(GW_ERR_INVALID_ARG, fn, "pool is NULL");
  if (need_base && (!p->base || !aligned(p->base, 256)))
    return fail(GW_ERR_INVALID_ARG, fn, "pool base is NULL or not 256-byte aligned");
  if (p->num_pages < 1) return fail(GW_ERR_INVALID_ARG, fn, "num_pages must be >= 1");
  if (p->page_size != 16) return fail(GW_ERR_INVALID_ARG, fn, "page_size must be 16 (got %d)", p->page_size);
  if (p->dtype != GW_KV_BF16 && p->dtype != GW_KV_E4M3) return fail(GW_ERR_INVALID_ARG, fn, "unknown dtype %d", p->dtype);
  if (p->layout == GW_LAYOUT_LOCAL) {
    if (p->head_dim != 256 || p->rot_dim != 256)
      return fail(GW_ERR_INVALID_ARG, fn, "local pool needs head_dim 256 and rot_dim 256");
    if (p->kv_heads < 1 || p->kv_heads > 64) return fail(GW_ERR_INVALID_ARG, fn, "kv_heads must be in [1, 64]");
  } else if (p->layout == GW_LAYOUT_GLOBAL_FOLDED || p->layout == GW_LAYOUT_GLOBAL_FULL ||
             p->layout == GW_LAYOUT_GLOBAL_FOLDED_E4M3) {
    if (p->head_dim != 512 || p->rot_dim != 128)
      return fail(GW_ERR_INVALID_ARG, fn, "global pool needs head_dim 512 and rot_dim 128");
    if (p->kv_heads != 1) return fail(GW_ERR_INVALID_ARG, fn, "global pool has exactly one KV head");
    if (p->layout == GW_LAYOUT_GLOBAL_FOLDED_E4M3) {
      if (p->dtype != GW_KV_E4M3)
        return fail(GW_ERR_INVALID_ARG, fn, "layout GLOBAL_FOLDED_E4M3 needs dtype e4m3");
    } else if (p->dtype != GW_KV_BF16) {
      return fail(GW_ERR_UNSUPPORTED, fn,
                  "e4m3 KV supports only local (sliding) layers; the opt-in e4m3 global pool is layout "
                  "GLOBAL_FOLDED_E4M3");
    }
  } else {
    return fail(GW_ERR_INVALID_ARG, fn, "unknown layout %d", p->layout);
  }
  return GW_OK;
}

size_t page_bytes(const gw_kv_pool* p) {
  if (p->layout == GW_LAYOUT_LOCAL) return static_cast<size_t>(p->kv_heads) * 2 * 16 * 256 * (p->dtype == GW_KV_BF16 ? 2 : 1);
  if (p->layout == GW_LAYOUT_GLOBAL_FOLDED_E4M3) return 16 * 640;
  return p->layout == GW_LAYOUT_GLOBAL_FOLDED ? 16 * 640 * 2 : 16 * 1024 * 2;
}

gw_status cuda_status(cudaError_t e, const char* fn) {
  if (e == cudaSuccess) return GW_OK;
  return fail(GW_ERR_CUDA, fn, "CUDA error %d (%s)", static_cast<int>(e), cudaGetErrorString(e));
}

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

gw_status set_error(gw_status code, const char* fn, const char* fmt, ...) {
  int n = std::snprintf(g_err, sizeof(g_err), "%s: ", fn);
  if (n < 0) n = 0;
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err + n, sizeof(g_err) - static_cast<size_t>(n), fmt, ap);
  va_end(ap);
  return code;
}

thread_local int g_max_ctas = 0;
thread_local bool g_early_launch = true;
thread_local bool g_early_inputs = false;

bool early_launch() { return g_early_launch; }
bool early_inputs() { return g_early_inputs; }

int grid_ctas() {
  const int n = num_sms();
  return g_max_ctas > 0 && g_max_ctas < n ? g_max_ctas : n;
}

int num_sms() {
  static int cached = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached = n > 0 ? n : 1;
  });
  return cached;
}

WsLayout ws_layout(int layout, int dtype, int kv_heads, int num_q_heads, int batch, int max_seq_len, int window) {
  WsLayout w{};
  int64_t units;
  if (layout == GW_LAYOUT_LOCAL) {
    const int chunk = dtype == GW_KV_BF16 ? kLocalChunkPagesBf16 : kLocalChunkPagesE4m3;
    const int64_t span = window < max_seq_len ? window : max_seq_len;
    const int64_t pages = ceil_div(span, 16) + 1;
    units = static_cast<int64_t>(batch) * kv_heads * ceil_div(pages, chunk);
    w.heads_per_unit = num_q_heads / kv_heads;
  } else {
    // global_chunks(L) <= min(kGlobalMaxChunks, ceil(pages(L) / 16)) for every L
    const int64_t c16 = ceil_div(ceil_div(max_seq_len, 16), kGlobalChunkPagesMin);
    units = static_cast<int64_t>(batch) * (c16 < kGlobalMaxChunks ? c16 : kGlobalMaxChunks);
    w.heads_per_unit = num_q_heads;
  }
  const int D = layout == GW_LAYOUT_LOCAL ? 256 : 512;
  w.max_units = units;
  w.reserved = 0;
  w.unit_base = 256;
  w.ml = w.unit_base + round_up(static_cast<size_t>(batch + 1) * 4, 256);
  w.o = w.ml + round_up(static_cast<size_t>(units) * w.heads_per_unit * 8, 256);
  w.prompt_base = w.o + round_up(static_cast<size_t>(units) * w.heads_per_unit * D * 4, 256);
  w.total = w.prompt_base + round_up(static_cast<size_t>(batch + 1) * 4, 256);
  return w;
}

}  // namespace gw

using namespace gw;

extern "C" {

const char* gw_last_error(void) { return g_err; }

int32_t gw_version(void) { return 1; }

size_t gw_pool_page_bytes(const gw_kv_pool* pool) {
  if (check_pool(pool, "gw_pool_page_bytes", false) != GW_OK) return 0;
  return page_bytes(pool);
}

gw_status gw_kv_append(const gw_kv_pool* pool, const void* k, const void* v, int32_t num_rows, const int32_t* slot,
                       const int32_t* pos, const float* rope_cs, int32_t max_pos, int32_t* dev_status,
                       void* stream) {
  const char* fn = "gw_kv_append";
  g_err[0] = 0;
  gw_status s = check_pool(pool, fn);
  if (s != GW_OK) return s;
  if (num_rows < 0) return fail(GW_ERR_INVALID_ARG, fn, "num_rows < 0");
  if (num_rows == 0) return GW_OK;
  if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return fail(GW_ERR_INVALID_ARG, fn, "k/v NULL or not 16-byte aligned");
  if (!slot || !pos || !aligned(slot, 4) || !aligned(pos, 4)) return fail(GW_ERR_INVALID_ARG, fn, "slot/pos NULL or misaligned");
  if (!rope_cs || !aligned(rope_cs, 16)) return fail(GW_ERR_INVALID_ARG, fn, "rope_cs NULL or not 16-byte aligned");
  if (max_pos < 1) return fail(GW_ERR_INVALID_ARG, fn, "max_pos must be >= 1");
  if (dev_status && !aligned(dev_status, 4)) return fail(GW_ERR_INVALID_ARG, fn, "dev_status misaligned");
  AppendArgs a{};
  a.pool = static_cast<uint8_t*>(pool->base);
  a.num_pages = pool->num_pages;
  a.kv_heads = pool->kv_heads;
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.num_rows = num_rows;
  a.slot = slot;
  a.pos = pos;
  a.rope_cs = rope_cs;
  a.max_pos = max_pos;
  a.early_inputs = g_early_inputs ? 1 : 0;
  a.status = dev_status;
  return cuda_status(launch_append(pool->layout, pool->dtype, a, static_cast<cudaStream_t>(stream)), fn);
}

gw_status gw_rope_cs(float* rope_cs, double theta, int32_t rot_dim, int32_t head_dim, int32_t max_pos,
                     void* stream) {
  const char* fn = "gw_rope_cs";
  g_err[0] = 0;
  if (!rope_cs || !aligned(rope_cs, 16)) return fail(GW_ERR_INVALID_ARG, fn, "rope_cs NULL or not 16-byte aligned");
  if (!(theta > 0.0) || !std::isfinite(theta)) return fail(GW_ERR_INVALID_ARG, fn, "theta must be finite and > 0");
  if (head_dim < 2 || rot_dim < 2 || rot_dim > head_dim || rot_dim % 2)
    return fail(GW_ERR_INVALID_ARG, fn, "need an even rot_dim in [2, head_dim] (rot_dim %d, head_dim %d)", rot_dim,
                head_dim);
  if (max_pos < 1) return fail(GW_ERR_INVALID_ARG, fn, "max_pos must be >= 1");
  return cuda_status(launch_rope_cs(rope_cs, theta, rot_dim, head_dim, max_pos, static_cast<cudaStream_t>(stream)),
                     fn);
}

size_t gw_attn_workspace_bytes(const gw_kv_pool* pool, int32_t num_q_heads, int32_t batch, int32_t max_seq_len,
                               int32_t max_q_rows, int32_t window) {
  (void)max_q_rows;
  if (check_pool(pool, "gw_attn_workspace_bytes", false) != GW_OK) return 0;
  if (num_q_heads < 1 || batch < 0 || max_seq_len < 0) return 0;
  if (pool->layout == GW_LAYOUT_LOCAL && window < 1) return 0;
  if (num_q_heads % pool->kv_heads) return 0;
  const int ms = max_seq_len > 0 ? max_seq_len : 1;
  return ws_layout(pool->layout, pool->dtype, pool->kv_heads, num_q_heads, batch, ms,
                   pool->layout == GW_LAYOUT_LOCAL ? window : 0)
      .total;
}

// The step's K/V rows of a gw_append_decode_attn_* call.
struct FusedAppend {
  const void* k;
  const void* v;
  const float* rope_cs;
  int32_t max_pos;
};

static gw_status attn_common(const char* fn, bool local, const gw_kv_pool* pool, const void* q, void* out,
                             int32_t num_q_heads, int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                             const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                             int32_t window, float scale, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream, bool validate_only = false,
                             float* lse = nullptr, const FusedAppend* app = nullptr) {
  g_err[0] = 0;
  gw_status s = check_pool(pool, fn);
  if (s != GW_OK) return s;
  if (app) {
    if (!app->k || !app->v || !aligned(app->k, 16) || !aligned(app->v, 16))
      return fail(GW_ERR_INVALID_ARG, fn, "k/v NULL or not 16-byte aligned");
    if (!app->rope_cs || !aligned(app->rope_cs, 16))
      return fail(GW_ERR_INVALID_ARG, fn, "rope_cs NULL or not 16-byte aligned");
    if (app->max_pos < 1) return fail(GW_ERR_INVALID_ARG, fn, "max_pos must be >= 1");
  }
  if (local && pool->layout != GW_LAYOUT_LOCAL) return fail(GW_ERR_INVALID_ARG, fn, "pool layout is not LOCAL");
  if (!local && pool->layout == GW_LAYOUT_LOCAL) return fail(GW_ERR_INVALID_ARG, fn, "pool layout is not GLOBAL");
  if (batch < 0) return fail(GW_ERR_INVALID_ARG, fn, "batch < 0");
  if (batch == 0) return GW_OK;
  if (num_q_heads < 1 || num_q_heads % pool->kv_heads)
    return fail(GW_ERR_INVALID_ARG, fn, "num_q_heads (%d) must be a positive multiple of kv_heads (%d)", num_q_heads,
                pool->kv_heads);
  const int group = num_q_heads / pool->kv_heads;
  if (local && group != 1 && group != 2 && group != 4 && group != 8)
    return fail(GW_ERR_UNSUPPORTED, fn, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", group);
  if (!local && num_q_heads != 8 && num_q_heads != 16 && num_q_heads != 32)
    return fail(GW_ERR_UNSUPPORTED, fn, "num_q_heads must be 8, 16 or 32 (got %d)", num_q_heads);
  if (local && window < 1) return fail(GW_ERR_INVALID_ARG, fn, "window must be >= 1");
  if (batch > kMaxBatch)
    return fail(GW_ERR_UNSUPPORTED, fn, "batch (%d) exceeds %d sequences per call", batch, kMaxBatch);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(GW_ERR_INVALID_ARG, fn, "scale must be finite and > 0");
  if (max_pages_per_seq < 1) return fail(GW_ERR_INVALID_ARG, fn, "max_pages_per_seq must be >= 1");
  if (max_q_rows < 1) return fail(GW_ERR_INVALID_ARG, fn, "max_q_rows must be >= 1");
  if (!local && pool->dtype == GW_KV_E4M3 && max_q_rows > 1)
    return fail(GW_ERR_UNSUPPORTED, fn, "prompt rows (max_q_rows %d > 1) on an e4m3 global pool: the global "
                "prompt-row kernel reads bf16 pages only", max_q_rows);
  if (!q || !out || !aligned(q, 16) || !aligned(out, 16)) return fail(GW_ERR_INVALID_ARG, fn, "q/out NULL or not 16-byte aligned");
  if (!cu_q_rows || !seq_lens || !block_table || !aligned(cu_q_rows, 4) || !aligned(seq_lens, 4) ||
      !aligned(block_table, 4))
    return fail(GW_ERR_INVALID_ARG, fn, "cu_q_rows/seq_lens/block_table NULL or misaligned");
  if (dev_status && !aligned(dev_status, 4)) return fail(GW_ERR_INVALID_ARG, fn, "dev_status misaligned");
  if (!workspace || !aligned(workspace, 256)) return fail(GW_ERR_INVALID_ARG, fn, "workspace NULL or not 256-byte aligned");
  const int64_t max_len64 = static_cast<int64_t>(max_pages_per_seq) * 16;
  const int max_len = max_len64 > 0x7fffffff ? 0x7fffffff : static_cast<int>(max_len64);
  const WsLayout w = ws_layout(pool->layout, pool->dtype, pool->kv_heads, num_q_heads, batch, max_len,
                               local ? window : 0);
  if (workspace_bytes < w.total)
    return fail(GW_ERR_WORKSPACE, fn, "workspace_bytes %zu < %zu needed", workspace_bytes, w.total);
  if (validate_only) return GW_OK;

  LocalArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.num_pages = pool->num_pages;
  a.kv_heads = pool->kv_heads;
  a.num_q_heads = num_q_heads;
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.batch = batch;
  a.cu_q_rows = cu_q_rows;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.max_pages = max_pages_per_seq;
  a.window = local ? window : 0x7fffffff;
  a.scale_log2 = scale * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.unit_base = reinterpret_cast<int32_t*>(ws + w.unit_base);
  a.part_ml = reinterpret_cast<float2*>(ws + w.ml);
  a.part_o = reinterpret_cast<float*>(ws + w.o);
  a.prompt_base = reinterpret_cast<int32_t*>(ws + w.prompt_base);
  a.max_units = w.max_units;
  a.status = dev_status;
  a.early_inputs = g_early_inputs ? 1 : 0;
  a.lse = lse;
  if (app) {
    a.k_new = static_cast<const uint16_t*>(app->k);
    a.v_new = static_cast<const uint16_t*>(app->v);
    a.rope_cs = app->rope_cs;
    a.max_pos = app->max_pos;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (local) {
    e = launch_local_decode(pool->dtype, group, a, st);
    if (e == cudaSuccess && max_q_rows > 1) e = launch_local_prompt(pool->dtype, group, a, max_q_rows, st);
  } else {
    e = launch_global_decode(pool->layout, a, st);
    if (e == cudaSuccess && max_q_rows > 1) e = launch_global_prompt(pool->layout, a, max_q_rows, st);
  }
  return cuda_status(e, fn);
}

gw_status gw_decode_attn_local(const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                               const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                               int32_t max_pages_per_seq, int32_t max_q_rows, int32_t window, float scale,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return attn_common("gw_decode_attn_local", true, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens, block_table,
                     max_pages_per_seq, max_q_rows, window, scale, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"

namespace gw {
gw_status validate_local_call(const char* fn, const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads,
                              int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                              const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                              int32_t window, float scale, size_t workspace_bytes, int32_t* dev_status) {
  // Any 256-byte aligned non-null address stands in for the workspace: only
  // its size is checked, and nothing is launched.
  return attn_common(fn, true, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens, block_table, max_pages_per_seq,
                     max_q_rows, window, scale, reinterpret_cast<void*>(static_cast<uintptr_t>(256)), workspace_bytes,
                     dev_status, nullptr, true);
}
}  // namespace gw

extern "C" {

gw_status gw_append_decode_attn_local(const gw_kv_pool* pool, const void* k, const void* v, const float* rope_cs,
                                      int32_t max_pos, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                                      const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                                      int32_t max_pages_per_seq, int32_t window, float scale, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const FusedAppend app{k, v, rope_cs, max_pos};
  return attn_common("gw_append_decode_attn_local", true, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens,
                     block_table, max_pages_per_seq, 1, window, scale, workspace, workspace_bytes, dev_status, stream,
                     false, nullptr, &app);
}

gw_status gw_append_decode_attn_global(const gw_kv_pool* pool, const void* k, const void* v, const float* rope_cs,
                                       int32_t max_pos, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                                       const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                                       int32_t max_pages_per_seq, float scale, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const FusedAppend app{k, v, rope_cs, max_pos};
  return attn_common("gw_append_decode_attn_global", false, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens,
                     block_table, max_pages_per_seq, 1, 0, scale, workspace, workspace_bytes, dev_status, stream,
                     false, nullptr, &app);
}

gw_status gw_decode_attn_global(const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads, int32_t batch,
                                const int32_t* cu_q_rows, const int32_t* seq_lens, const int32_t* block_table,
                                int32_t max_pages_per_seq, int32_t max_q_rows, float scale, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return attn_common("gw_decode_attn_global", false, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens,
                     block_table, max_pages_per_seq, max_q_rows, 0, scale, workspace, workspace_bytes, dev_status,
                     stream);
}

gw_status gw_decode_attn_global_lse(const gw_kv_pool* pool, const void* q, void* out, float* lse,
                                    int32_t num_q_heads, int32_t batch, const int32_t* cu_q_rows,
                                    const int32_t* seq_lens, const int32_t* block_table, int32_t max_pages_per_seq,
                                    float scale, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                    void* stream) {
  const char* fn = "gw_decode_attn_global_lse";
  if (!lse || !aligned(lse, 4)) {
    g_err[0] = 0;
    return fail(GW_ERR_INVALID_ARG, fn, "lse NULL or misaligned");
  }
  return attn_common(fn, false, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens, block_table,
                     max_pages_per_seq, 1, 0, scale, workspace, workspace_bytes, dev_status, stream, false, lse);
}

gw_status gw_merge_lse(int32_t n_parts, const void* const* o_parts, const float* const* lse_parts, void* out,
                       float* lse_out, int32_t rows, int32_t num_heads, int32_t head_dim, void* stream) {
  const char* fn = "gw_merge_lse";
  g_err[0] = 0;
  if (n_parts < 1 || n_parts > kMaxMergeParts)
    return fail(GW_ERR_INVALID_ARG, fn, "n_parts (%d) outside [1, %d]", n_parts, kMaxMergeParts);
  if (rows < 0 || num_heads < 1) return fail(GW_ERR_INVALID_ARG, fn, "rows < 0 or num_heads < 1");
  if (head_dim != 256 && head_dim != 512) return fail(GW_ERR_INVALID_ARG, fn, "head_dim must be 256 or 512");
  if (!o_parts || !lse_parts) return fail(GW_ERR_INVALID_ARG, fn, "o_parts/lse_parts NULL");
  if (!out || !aligned(out, 16)) return fail(GW_ERR_INVALID_ARG, fn, "out NULL or not 16-byte aligned");
  if (lse_out && !aligned(lse_out, 4)) return fail(GW_ERR_INVALID_ARG, fn, "lse_out misaligned");
  MergeArgs m{};
  for (int r = 0; r < n_parts; ++r) {
    if (!o_parts[r] || !aligned(o_parts[r], 16) || !lse_parts[r] || !aligned(lse_parts[r], 4))
      return fail(GW_ERR_INVALID_ARG, fn, "part %d: o NULL or not 16-byte aligned, or lse NULL or misaligned", r);
    m.o[r] = static_cast<const uint16_t*>(o_parts[r]);
    m.lse[r] = lse_parts[r];
  }
  if (rows == 0) return GW_OK;
  m.n_parts = n_parts;
  m.rows = rows;
  m.heads = num_heads;
  m.head_dim = head_dim;
  m.out = static_cast<uint16_t*>(out);
  m.lse_out = lse_out;
  return cuda_status(launch_merge_lse(m, static_cast<cudaStream_t>(stream)), fn);
}

gw_status gw_set_max_ctas(int32_t max_ctas) {
  g_err[0] = 0;
  if (max_ctas < 0) return fail(GW_ERR_INVALID_ARG, "gw_set_max_ctas", "max_ctas (%d) < 0", max_ctas);
  g_max_ctas = max_ctas;
  return GW_OK;
}

gw_status gw_set_early_launch(int32_t on) {
  g_err[0] = 0;
  g_early_launch = on != 0;
  return GW_OK;
}

gw_status gw_set_early_inputs(int32_t on) {
  g_err[0] = 0;
  g_early_inputs = on != 0;
  return GW_OK;
}

gw_status gw_bw_probe(const void* buf, size_t bytes, int32_t* dev_status, void* stream) {
  const char* fn = "gw_bw_probe";
  g_err[0] = 0;
  if (!buf || !aligned(buf, 16)) return fail(GW_ERR_INVALID_ARG, fn, "buf NULL or not 16-byte aligned");
  if (bytes < 8192) return fail(GW_ERR_INVALID_ARG, fn, "bytes (%zu) < 8192", bytes);
  if (dev_status && !aligned(dev_status, 4)) return fail(GW_ERR_INVALID_ARG, fn, "dev_status misaligned");
  return cuda_status(launch_bw_probe(buf, static_cast<int64_t>(bytes / 8192), dev_status,
                                     static_cast<cudaStream_t>(stream)),
                     fn);
}

gw_status gw_bw_probe_tma(const void* buf, size_t bytes, int32_t* dev_status, void* stream) {
  const char* fn = "gw_bw_probe_tma";
  g_err[0] = 0;
  if (!buf || !aligned(buf, 256)) return fail(GW_ERR_INVALID_ARG, fn, "buf NULL or not 256-byte aligned");
  if (bytes < 16384) return fail(GW_ERR_INVALID_ARG, fn, "bytes (%zu) < 16384", bytes);
  if (bytes / 16384 > (static_cast<size_t>(1) << 22))  // tensor-map rows stay below 2^31
    return fail(GW_ERR_INVALID_ARG, fn, "bytes (%zu) above 2^36", bytes);
  if (dev_status && !aligned(dev_status, 4)) return fail(GW_ERR_INVALID_ARG, fn, "dev_status misaligned");
  return cuda_status(launch_bw_probe_tma(buf, static_cast<int64_t>(bytes / 16384), dev_status,
                                         static_cast<cudaStream_t>(stream)),
                     fn);
}

gw_status gw_wait_selftest(int32_t* dev_status, int32_t* result, int64_t limit_ns, void* stream) {
  const char* fn = "gw_wait_selftest";
  g_err[0] = 0;
  if (!dev_status || !aligned(dev_status, 4)) return fail(GW_ERR_INVALID_ARG, fn, "dev_status NULL or misaligned");
  if (!result || !aligned(result, 4)) return fail(GW_ERR_INVALID_ARG, fn, "result NULL or misaligned");
  if (limit_ns < 1000 || limit_ns > 1000000000)
    return fail(GW_ERR_INVALID_ARG, fn, "limit_ns (%lld) outside [1e3, 1e9]", static_cast<long long>(limit_ns));
  return cuda_status(launch_wait_selftest(dev_status, result, limit_ns, static_cast<cudaStream_t>(stream)), fn);
}

}  // extern "C"
