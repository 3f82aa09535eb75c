// Device helpers shared by the gw kernels (sm_103a).
//
// Thin inline-PTX wrappers for the Blackwell asynchronous-copy machinery the
// kernels use (mbarrier, cp.async.bulk), bounded waits, and the bf16 / e4m3
// unpacking used on the KV load path.
#pragma once

#include <atomic>
#include <mutex>
#include <cstdint>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gw_internal.h"

namespace gw {

constexpr int kPage = 16;
// A bounded wait gives up after this many nanoseconds of the global timer and
// raises GW_DEV_TIMEOUT; legitimate waits are microseconds.
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and records
// GW_DEV_TIMEOUT) if the phase never completes; the caller then abandons its
// work instead of spinning forever.
// (`limit_ns` other than kWaitNs only in the wait self-test.)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status,
                                          uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, GW_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Orders this thread's earlier global writes (generic proxy) before later
// asynchronous-proxy accesses, such as a tensor copy of the same bytes.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void st_release_shared(int32_t* p, int32_t v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t ld_acquire_shared(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Bounded wait until the shared-memory counter *p, raised by another warp of
// the CTA, reaches `target`.  Returns false (and records GW_DEV_TIMEOUT) if
// it never does.
__device__ __forceinline__ bool wait_counter(const int32_t* p, int32_t target, int32_t* status) {
  if (ld_acquire_shared(p) >= target) return true;
  const uint64_t t0 = global_ns();
  while (ld_acquire_shared(p) < target) {
    if (global_ns() - t0 > kWaitNs) {
      if (status) atomicOr(status, GW_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// One-dimensional bulk copy global -> shared, completion counted on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Prefetch [src, src + bytes) into L2 (no completion tracking); 16-byte
// aligned address, size a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 policy for data read many times in a short span (prompt-row K/V tiles).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data read exactly once (KV pages): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Invalidate the 128-byte L2 line at p (128-byte aligned) without writing it
// back: scratch data that has been read for the last time.
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- unpacking of stored KV elements to fp32 --------------------------------
__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---- programmatic dependent launch ---------------------------------------
// Every gw kernel is launched with programmatic stream serialisation allowed,
// so its CTAs may be scheduled while the previous kernel of the stream is
// still running.  pdl_wait() blocks until that kernel has completed and its
// memory is visible; each kernel calls it before touching any memory the
// caller or an earlier kernel may still be writing.  pdl_trigger() lets the
// next kernel's CTAs be scheduled early (they still wait in pdl_wait()).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early_launch() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
inline cudaError_t set_smem_once(const void* kern, size_t bytes) {
  struct Entry {
    const void* fn;
    uint64_t devices;
  };
  static std::mutex mu;
  static Entry table[64];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  std::lock_guard<std::mutex> lock(mu);
  Entry* ent = nullptr;
  for (int i = 0; i < used; ++i)
    if (table[i].fn == kern) ent = &table[i];
  if (ent && bit && (ent->devices & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (!ent && used < 64) {
    table[used] = Entry{kern, 0};
    ent = &table[used++];
  }
  if (ent) ent->devices |= bit;
  return cudaSuccess;
}

}  // namespace gw
