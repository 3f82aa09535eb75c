// Local decode attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at the point where they
// run attention: embedding runtimes that have no device allocator of their
// own, and hosts that forbid device allocation once serving has started (a
// fixed memory budget decided at start-up).  gw_decode_attn_local needs a
// caller-supplied workspace for its split-KV partials; this entry point runs
// the same computation with that workspace carved from a fixed, file-scope
// device array instead, so the call itself allocates nothing.
//
// The array is kStaticScratchBytes (32 MiB) and lives on every GPU that loads
// this library's module, until the process exits.  A call whose workspace
// requirement (gw_attn_workspace_bytes) exceeds it is rejected.
#include <cstdio>
#include <mutex>

#include <cuda.h>

#include "gw_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;

// Device-side scratch shared by every call of gw_decode_attn_local_noalloc.
// In host code this name is only a stand-in for the symbol, not a device
// address: the address is obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kStaticScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn resolve_ctx_get_current() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<CtxGetCurrentFn>(fn);
}

// Cached address of the scratch per device, tagged with the context it was
// resolved in: after a device reset the module is loaded again, possibly at
// another address, in a new context, and the address is looked up again.
constexpr int kMaxDevices = 64;
struct Cached {
  CUcontext ctx;
  void* addr;
};
std::mutex g_mu;
Cached g_scratch[kMaxDevices] = {};

// Device address of the scratch on the current device (with that device
// current).
gw_status scratch_for_current_device(const char* fn, void** out) {
  static const CtxGetCurrentFn ctx_get_current = resolve_ctx_get_current();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gw::set_error(GW_ERR_CUDA, fn, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return gw::set_error(GW_ERR_UNSUPPORTED, fn, "device ordinal %d >= %d", dev, kMaxDevices);
  if (!ctx_get_current) return gw::set_error(GW_ERR_CUDA, fn, "cuCtxGetCurrent is not available");
  // Before the runtime's first call on this device no context may be current
  // (ctx stays NULL); cudaGetSymbolAddress then initialises the device's
  // primary context, which is read again afterwards.
  CUcontext ctx = nullptr;
  if (ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_scratch[dev].addr || g_scratch[dev].ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return gw::set_error(GW_ERR_CUDA, fn, "cudaGetSymbolAddress of the static scratch failed: %s",
                           cudaGetErrorString(e));
    if (ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx)
      return gw::set_error(GW_ERR_CUDA, fn, "cannot read the current CUDA context");
    g_scratch[dev] = Cached{ctx, p};
  }
  *out = g_scratch[dev].addr;
  return GW_OK;
}

}  // namespace

extern "C" gw_status gw_decode_attn_local_noalloc(const gw_kv_pool* pool, const void* q, void* out,
                                                  int32_t num_q_heads, int32_t batch, const int32_t* cu_q_rows,
                                                  const int32_t* seq_lens, const int32_t* block_table,
                                                  int32_t max_pages_per_seq, int32_t max_q_rows, int32_t window,
                                                  float scale, int32_t* dev_status, void* stream) {
  const char* fn = "gw_decode_attn_local_noalloc";
  // The same checks, in the same order, as gw_decode_attn_local, with the
  // static scratch's size as the workspace size: an invalid call gets the
  // same status as there, and a call needing more scratch GW_ERR_WORKSPACE.
  gw_status s = gw::validate_local_call(fn, pool, q, out, num_q_heads, batch, cu_q_rows, seq_lens, block_table,
                                        max_pages_per_seq, max_q_rows, window, scale, kStaticScratchBytes,
                                        dev_status);
  if (s != GW_OK || batch == 0) return s;
  void* scratch = nullptr;
  s = scratch_for_current_device(fn, &scratch);
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
