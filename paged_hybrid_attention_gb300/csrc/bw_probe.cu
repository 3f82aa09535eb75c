// gw_bw_probe: the read bandwidth the decode kernels' copy pipeline can reach.
// gw_bw_probe_tma: the same for the tensor-map pipeline of the bf16 kernel.
// gw_wait_selftest: the bounded-wait path of the kernels, made to run out.
//
// Not part of the method: a measurement aid for the roofline.  It streams a
// buffer through exactly the pipeline shape of the local decode kernel - one
// persistent CTA per SM, 8 warps, each with a private 2-stage ring of 8 KiB
// stages filled by two 4 KiB cp.async.bulk copies - and does no arithmetic,
// so its rate is the ceiling that pipeline can reach on this GPU.
#include "common.cuh"
#include "tma.cuh"

namespace gw {
namespace {

constexpr int kProbeWarps = 8;
constexpr int kProbeStages = 2;
constexpr int kProbeStage = 8192;

struct __align__(128) ProbeWarp {
  uint8_t stage[kProbeStages][kProbeStage];
  uint64_t bar[kProbeStages];
};

__global__ void __launch_bounds__(kProbeWarps * 32, 1) bw_probe_kernel(const uint8_t* buf, int64_t chunks,
                                                                          int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ProbeWarp& sm = reinterpret_cast<ProbeWarp*>(smem_raw)[warp];
  if (lane == 0) {
    for (int i = 0; i < kProbeStages; ++i) mbar_init(&sm.bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_trigger();
  const uint64_t pol = policy_evict_first();
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kProbeWarps;
  int64_t next = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x;  // SM-minor, as the decode kernel
  uint32_t issued = 0, consumed = 0;
  auto issue = [&]() {
    const int st = issued % kProbeStages;
    if (lane == 0) {
      const uint8_t* src = buf + next * kProbeStage;
      mbar_arrive_expect_tx(&sm.bar[st], kProbeStage);
      bulk_g2s(sm.stage[st], src, kProbeStage / 2, &sm.bar[st], pol);
      bulk_g2s(sm.stage[st] + kProbeStage / 2, src + kProbeStage / 2, kProbeStage / 2, &sm.bar[st], pol);
    }
    ++issued;
    next += n_warps;
  };
  while (next < chunks && issued - consumed < kProbeStages) issue();
  uint32_t acc = 0;
  while (consumed < issued) {
    const int st = consumed % kProbeStages;
    if (!mbar_wait(&sm.bar[st], (consumed / kProbeStages) & 1, status)) {
      for (uint32_t k = consumed + 1; k < issued; ++k)
        mbar_wait(&sm.bar[k % kProbeStages], (k / kProbeStages) & 1, nullptr);
      return;
    }
    acc ^= *reinterpret_cast<const uint32_t*>(sm.stage[st] + lane * 16);
    __syncwarp();
    ++consumed;
    while (next < chunks && issued - consumed < kProbeStages) issue();
  }
  // never true for a pool of finite bf16 data; keeps the reads observable
  if (acc == 0x7FC00001u && status) atomicOr(status, 0);
}

// gw_bw_probe_tma: the copy pipeline of the bf16 local decode kernel (one
// persistent CTA per SM, 6 warps, each with a 2-stage ring of 16 KiB stages;
// a stage is one 16-token page head, K then V, brought by 8 tensor-map boxes
// of 2 KiB that land 128-byte swizzled), streaming the buffer viewed as a
// LOCAL pool of one KV head: stage i is page i.  No arithmetic.
constexpr int kTmaWarps = 6;
constexpr int kTmaStages = 2;
constexpr int kTmaStage = 16384;

struct __align__(1024) TmaProbeWarp {
  uint8_t stage[kTmaStages][kTmaStage];
  uint64_t bar[kTmaStages];
};

__global__ void __launch_bounds__(kTmaWarps * 32, 1) bw_probe_tma_kernel(int64_t pages, int32_t* status,
                                                                           const __grid_constant__ CUtensorMap map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TmaProbeWarp& sm = reinterpret_cast<TmaProbeWarp*>(smem_raw)[warp];
  if (lane == 0) {
    for (int i = 0; i < kTmaStages; ++i) mbar_init(&sm.bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_trigger();
  const uint64_t pol = policy_evict_first();
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kTmaWarps;
  int64_t next = static_cast<int64_t>(warp) * gridDim.x + blockIdx.x;
  uint32_t issued = 0, consumed = 0;
  auto issue = [&]() {
    const int st = issued % kTmaStages;
    if (lane == 0) mbar_arrive_expect_tx(&sm.bar[st], kTmaStage);
    __syncwarp();
    if (lane < 4)  // one 4 KB box per 64-dim chunk: the page head's K and V rows
      tma_rows(smem_u32(sm.stage[st]) + lane * 4096, &map, lane, static_cast<int>(next * 2 * kPage), &sm.bar[st],
               pol);
    ++issued;
    next += n_warps;
  };
  while (next < pages && issued - consumed < kTmaStages) issue();
  uint32_t acc = 0;
  while (consumed < issued) {
    const int st = consumed % kTmaStages;
    if (!mbar_wait(&sm.bar[st], (consumed / kTmaStages) & 1, status)) {
      for (uint32_t k = consumed + 1; k < issued; ++k)
        mbar_wait(&sm.bar[k % kTmaStages], (k / kTmaStages) & 1, nullptr);
      return;
    }
    acc ^= *reinterpret_cast<const uint32_t*>(sm.stage[st] + lane * 16);
    __syncwarp();
    ++consumed;
    while (next < pages && issued - consumed < kTmaStages) issue();
  }
  if (acc == 0x7FC00001u && status) atomicOr(status, 0);
}

// gw_wait_selftest: one warp, one mbarrier of arrival count 1.  Phase 0 is
// completed by an arrival, then waited on (must succeed); phase 1 is never
// arrived on, so its wait must give up after limit_ns, raise GW_DEV_TIMEOUT
// and return.  result = {phase-0 wait succeeded, phase-1 wait gave up,
// microseconds spent in the phase-1 wait}.
__global__ void wait_selftest_kernel(int32_t* status, int32_t* result, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_arrive(&bar);
  __syncwarp();
  const bool ok0 = __all_sync(0xffffffffu, mbar_wait(&bar, 0, status, limit_ns));
  const uint64_t t0 = global_ns();
  const bool ok1 = __all_sync(0xffffffffu, mbar_wait(&bar, 1, status, limit_ns));
  const uint64_t dt = global_ns() - t0;
  if (threadIdx.x == 0) {
    result[0] = ok0 ? 1 : 0;
    result[1] = ok1 ? 0 : 1;
    result[2] = static_cast<int32_t>(dt / 1000 < 0x7fffffffull ? dt / 1000 : 0x7fffffffull);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* status, int32_t* result, int64_t limit_ns, cudaStream_t st) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, st, status, result,
                    static_cast<uint64_t>(limit_ns));
}

cudaError_t launch_bw_probe_tma(const void* buf, int64_t pages, int32_t* status, cudaStream_t st) {
  LocalArgs a{};
  a.pool = static_cast<const uint8_t*>(buf);
  a.num_pages = pages;
  a.kv_heads = 1;
  CUtensorMap map;
  cudaError_t e = make_local_kv_map(a, &map, GW_KV_BF16, 32);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(TmaProbeWarp) * kTmaWarps;
  e = set_smem_once(reinterpret_cast<const void*>(bw_probe_tma_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(bw_probe_tma_kernel, dim3(num_sms()), dim3(kTmaWarps * 32), smem, st, pages, status, map);
}

cudaError_t launch_bw_probe(const void* buf, int64_t chunks, int32_t* status, cudaStream_t st) {
  const size_t smem = sizeof(ProbeWarp) * kProbeWarps;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(bw_probe_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(bw_probe_kernel, dim3(num_sms()), dim3(kProbeWarps * 32), smem, st,
                    static_cast<const uint8_t*>(buf), chunks, status);
}

}  // namespace gw
