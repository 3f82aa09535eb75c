// Internal interface between the C-ABI layer (gw_abi.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gw.h"

namespace gw {

// ---- split-KV plan constants ------------------------------------------------
// A local decode work unit is (sequence, KV head, chunk of kLocalChunkPages
// logical pages of that sequence's window); a global unit is (sequence, chunk
// of global_chunk_pages(L) pages).  Chunks depend only on the sequence's own
// length, so a row's arithmetic never depends on the rest of the batch.
constexpr int kLocalChunkPagesBf16 = 8;
constexpr int kLocalChunkPagesE4m3 = 8;
// Global chunks start at 32 pages and double until a sequence has at most
// kGlobalMaxChunks of them (long contexts get long chunks, so the partials
// stay a small fraction of the KV bytes).
constexpr int kGlobalChunkPagesMin = 32;
constexpr int kGlobalMaxChunks = 128;

// The decode kernels keep the batch's split plan in shared memory.
constexpr int kMaxBatch = 4096;


__host__ __device__ __forceinline__ int local_chunks(int L, int window, int chunk) {
  const int first = L > window ? L - window : 0;
  const int p0 = first / 16, p1 = (L - 1) / 16;
  return (p1 - p0 + chunk) / chunk;
}

// An upper bound on local_chunks(L, window, chunk) over L <= 16 * max_pages.
__host__ __device__ __forceinline__ int local_max_chunks(int max_pages, int window, int chunk) {
  const int span = (window - 1) / 16 + 1;  // p1 - p0 once L > window
  const int d = max_pages - 1 < span ? max_pages - 1 : span;
  return (d + chunk) / chunk;
}

// An upper bound on global_chunks(L) over L <= 16 * max_pages.
__host__ __device__ __forceinline__ int global_max_chunks(int max_pages) {
  const int c = (max_pages + kGlobalChunkPagesMin - 1) / kGlobalChunkPagesMin;
  return c < kGlobalMaxChunks ? c : kGlobalMaxChunks;
}

__host__ __device__ __forceinline__ int global_chunk_pages(int L) {
  const int pages = (L + 15) / 16;
  int cpg = kGlobalChunkPagesMin;
  while ((pages + cpg - 1) / cpg > kGlobalMaxChunks) cpg *= 2;
  return cpg;
}

__host__ __device__ __forceinline__ int global_chunks(int L) {
  const int cpg = global_chunk_pages(L);
  return ((L + 15) / 16 + cpg - 1) / cpg;
}

// Workspace layout (offsets from the 256-byte aligned workspace base):
//   [0, 256)          reserved
//   [256, ub_end)     int32 unit_base[batch + 1], rounded up to 256 bytes
//   [ub_end, ml_end)  float2 (m, l) per (unit, head of the unit)
//   [ml_end, o_end)   float  o[unit][head of the unit][head_dim]
//   [o_end, ...)      int32 prompt_base[batch + 1] (prompt-row tile offsets)
struct WsLayout {
  size_t reserved, unit_base, ml, o, prompt_base, total;
  int64_t max_units;
  int heads_per_unit;
};

WsLayout ws_layout(int layout, int dtype, int kv_heads, int num_q_heads, int batch, int max_seq_len,
                   int window);

struct LocalArgs {
  const uint8_t* pool;
  int64_t num_pages;
  int32_t kv_heads;
  int32_t num_q_heads;
  const uint16_t* q;  // bf16 bits
  uint16_t* out;      // bf16 bits
  int32_t batch;
  const int32_t* cu_q_rows;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t window;  // local; ignored for global
  float scale_log2;  // softmax scale * log2(e)
  int32_t* unit_base;
  float2* part_ml;
  float* part_o;
  int64_t max_units;
  int32_t* status;
  int32_t* prompt_base;  // tile offsets of the prompt-row kernels
  float* lse;            // optional: natural-log log-sum-exp per (decode row, q head)
  // Fused append (gw_append_decode_attn_*): the K/V row of each decode row,
  // at position seq_len - 1, written by the decode kernel; k_new null: none.
  const uint16_t* k_new;
  const uint16_t* v_new;
  const float* rope_cs;
  int32_t max_pos;
  int32_t early_inputs;  // gw_set_early_inputs: plan before the wait on the previous kernel
};

struct AppendArgs {
  uint8_t* pool;
  int64_t num_pages;
  int32_t kv_heads;
  const uint16_t* k;
  const uint16_t* v;
  int32_t num_rows;
  const int32_t* slot;
  const int32_t* pos;
  const float* rope_cs;
  int32_t max_pos;
  int32_t* status;
  int32_t early_inputs;  // gw_set_early_inputs: slot, pos and RoPE rows read before the wait
};

int num_sms();
// CTAs of a persistent attention kernel: one per SM, or the calling thread's
// gw_set_max_ctas cap if smaller.
int grid_ctas();
// Whether this thread's launches may start before their predecessor in the
// stream has finished (programmatic dependent launch); gw_set_early_launch.
bool early_launch();
// Whether the calling thread's calls may read their index inputs before the
// previous kernel of their stream has finished; gw_set_early_inputs.
bool early_inputs();

// Every host-side check of gw_decode_attn_local, workspace size included,
// with errors reported under the name `fn`; launches nothing.
gw_status validate_local_call(const char* fn, const gw_kv_pool* pool, const void* q, void* out, int32_t num_q_heads,
                              int32_t batch, const int32_t* cu_q_rows, const int32_t* seq_lens,
                              const int32_t* block_table, int32_t max_pages_per_seq, int32_t max_q_rows,
                              int32_t window, float scale, size_t workspace_bytes, int32_t* dev_status);

// Records `fmt` (printf-style) as the calling thread's gw_last_error message,
// prefixed by `fn`, and returns `code`.
gw_status set_error(gw_status code, const char* fn, const char* fmt, ...);

// Log-sum-exp merge of each decode row's partials into bf16 `out`; units of
// heads_per_unit q heads, planned as in a.unit_base, at most max_chunks
// chunks per sequence; with `discard`, the merged partials' L2 lines are
// dropped unwritten.
cudaError_t launch_combine(const LocalArgs& a, int heads_per_unit, int head_dim, int max_chunks, bool discard,
                           cudaStream_t st);

cudaError_t launch_append(int layout, int dtype, const AppendArgs& a, cudaStream_t st);

// Up to kMaxMergeParts attention results of the same rows over disjoint key
// sets, merged by their log-sum-exp (gw_merge_lse).
constexpr int kMaxMergeParts = 16;
struct MergeArgs {
  const uint16_t* o[kMaxMergeParts];  // bf16 [rows][heads][head_dim]
  const float* lse[kMaxMergeParts];   // [rows][heads], natural log
  int32_t n_parts, rows, heads, head_dim;
  uint16_t* out;
  float* lse_out;
};
cudaError_t launch_merge_lse(const MergeArgs& m, cudaStream_t st);
// (cos, sin) table of gw_rope_cs: float32 [max_pos][rot_dim / 2][2].
cudaError_t launch_rope_cs(float* out, double theta, int rot_dim, int head_dim, int max_pos, cudaStream_t st);
cudaError_t launch_bw_probe(const void* buf, int64_t chunks, int32_t* status, cudaStream_t st);
cudaError_t launch_bw_probe_tma(const void* buf, int64_t pages, int32_t* status, cudaStream_t st);
cudaError_t launch_wait_selftest(int32_t* status, int32_t* result, int64_t limit_ns, cudaStream_t st);
// TMA descriptor of a LOCAL pool: rows of 256 elements in 128-byte chunks
// (4 chunks of 64 bf16, or 2 chunks of 128 e4m3); row = ((page * kv_heads +
// head) * 2 + {K, V}) * 16 + token; box {one chunk, 1, 16 rows}, 128-byte
// swizzle.
constexpr int kPageTokens = 16;
// Tensor map of a LOCAL pool: boxes of one 128-byte chunk of `box_rows` rows
// (16: a page head's K or V; 32: its K and V together), 128-byte swizzled.
cudaError_t make_local_kv_map(const LocalArgs& a, CUtensorMap* map, int dtype = GW_KV_BF16, int box_rows = 16);
cudaError_t launch_local_decode(int dtype, int group, const LocalArgs& a, cudaStream_t st);
// tcgen05 decode kernel (kind::f8f6f4) for e4m3 LOCAL pools, plus the combine
cudaError_t launch_local_decode_e4m3_tc(int group, const LocalArgs& a, cudaStream_t st);
cudaError_t launch_global_decode(int layout, const LocalArgs& a, cudaStream_t st);
cudaError_t launch_local_prompt(int dtype, int group, const LocalArgs& a, int max_q_rows, cudaStream_t st);
// tcgen05 prompt-row kernel for local layers (bf16 or e4m3 pools); expects
// a.prompt_base planned with 128 / group queries per tile
cudaError_t launch_local_prompt_tc(int dtype, int group, const LocalArgs& a, cudaStream_t st);
// tcgen05 prompt-row kernel for global layers; expects a.prompt_base planned
// with 2 tiles (output-dim halves) per block of 128 / num_q_heads queries
cudaError_t launch_global_prompt_tc(int layout, const LocalArgs& a, cudaStream_t st);
cudaError_t launch_global_prompt(int layout, const LocalArgs& a, int max_q_rows, cudaStream_t st);

}  // namespace gw
