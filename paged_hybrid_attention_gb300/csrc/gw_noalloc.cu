// Local decode attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at the point where they
// run attention: code replayed inside an already-captured CUDA graph whose
// memory plan is frozen, allocator-less embedding runtimes, or hosts that
// forbid device allocation after start-up.  gw_decode_attn_local needs a
// caller-supplied workspace for its split-KV partials; this entry point runs
// the same computation with that workspace carved from a fixed, file-scope
// device array instead, so the call itself allocates nothing.
//
// The array is kStaticScratchBytes (32 MiB) and lives on every GPU that loads
// this library's module, until the process exits.  A call whose workspace
// requirement (gw_attn_workspace_bytes) exceeds it is rejected.
#include <cstdio>
#include <mutex>

#include "gw_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;

// Device-side scratch shared by every call of gw_decode_attn_local_noalloc.
// In host code this name is only a stand-in for the symbol, not a device
// address: the address is obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, resolved once per
// device (with that device current) and cached.
gw_status scratch_for_current_device(const char* fn, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gw::set_error(GW_ERR_CUDA, fn, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return gw::set_error(GW_ERR_UNSUPPORTED, fn, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return gw::set_error(GW_ERR_CUDA, fn, "cudaGetSymbolAddress of the static scratch failed: %s",
                           cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GW_OK;
}

}  // namespace

extern "C" gw_status gw_decode_attn_local_noalloc(const gw_kv_pool* pool, const void* q, void* out,
                                                  int32_t num_q_heads, int32_t batch, const int32_t* cu_q_rows,
                                                  const int32_t* seq_lens, const int32_t* block_table,
                                                  int32_t max_pages_per_seq, int32_t max_q_rows, int32_t window,
                                                  float scale, int32_t* dev_status, void* stream) {
  const char* fn = "gw_decode_attn_local_noalloc";
  if (batch > 0 && max_pages_per_seq > 0) {
    const int64_t max_len64 = static_cast<int64_t>(max_pages_per_seq) * 16;
    const int32_t max_len = max_len64 > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(max_len64);
    const size_t need = gw_attn_workspace_bytes(pool, num_q_heads, batch, max_len, max_q_rows, window);
    if (need > kStaticScratchBytes)
      return gw::set_error(GW_ERR_WORKSPACE, fn,
                           "this call needs %zu bytes of split-KV scratch; the static scratch holds %zu", need,
                           kStaticScratchBytes);
  }
  void* scratch = nullptr;
  gw_status s = scratch_for_current_device(fn, &scratch);
  if (s != GW_OK) return s;
  s = gw_decode_attn_local(pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens, block_table, max_pages_per_seq,
                           max_q_rows, window, scale, scratch, kStaticScratchBytes, dev_status, stream);
  if (s != GW_OK) {
    char msg[512];
    std::snprintf(msg, sizeof(msg), "%s", gw_last_error());
    return gw::set_error(s, fn, "%s", msg);
  }
  return GW_OK;
}

extern "C" size_t gw_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }
