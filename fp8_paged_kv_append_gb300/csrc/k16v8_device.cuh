// Device-side building blocks shared by the k16v8 kernels (sm_103a):
// mbarrier + bulk-async (TMA engine) copies, bounded waits, number-format
// conversions, and the host-side status helpers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "k16v8.h"

namespace k16v8 {

constexpr int kPage = K16V8_PAGE_SIZE;   // tokens per page
constexpr int kHeadDim = K16V8_HEAD_DIM;  // d
constexpr int kGroup = K16V8_GQA_GROUP;   // query heads per KV head
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Upper bound on polls of one mbarrier phase before a kernel gives up and
// flags K16V8_DEVERR_TIMEOUT.  try_wait suspends the thread for a
// hardware-defined interval per poll, so this is far beyond any real copy.
constexpr uint32_t kMaxPolls = 1u << 24;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint32_t max_polls = kMaxPolls) {
  for (uint32_t i = 0; i < max_polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Poll limit of the one wait that the bounded-wait test hooks make expire
// (a copy that is deliberately never issued): short, so the error path is
// reached at once.
constexpr uint32_t kTestPolls = 64;
constexpr uint32_t kTestSpins = 1u << 12;  // the same for a spinning (test_wait) role

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with an explicit suspend-time hint (ns) for latency-critical
// hand-offs.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded spin on test_wait (no suspension): for waits on the critical path
// of a pipeline.  The bound is far beyond any real copy or MMA.
constexpr uint32_t kMaxSpins = 1u << 28;
__device__ __forceinline__ bool mbar_spin_bounded(uint64_t *bar, uint32_t parity,
                                                  uint32_t max_spins = kMaxSpins) {
  for (uint32_t i = 0; i < max_spins; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return false;
}

// One contiguous global->shared copy on the bulk-async engine, completing
// `bytes` of transaction count on `bar`.  dst, src 16-B aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (the stream is read once).
__device__ __forceinline__ void bulk_g2s_evict_first(void *dst, const void *src, uint32_t bytes,
                                                     uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Start fetching `bytes` (a multiple of 16, 16-byte aligned) into L2.  Nothing
// reaches the SM, so it is safe on data that another kernel may still write:
// L2 is where the GPU's writes meet.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> two E4M3FN bytes, round-to-nearest-even, saturating finite
// values (hardware cvt).  Result: lo byte <- x0, hi byte <- x1.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}

// Two E4M3FN bytes -> half2 (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  __half2 h;
  *reinterpret_cast<uint32_t *>(&h) = r;
  return h;
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible (a no-op without the launch
// attribute), and allow the next grid to begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_error(int32_t *dev_error, int32_t bit) {
  if (dev_error) atomicOr(dev_error, bit);
}

}  // namespace k16v8

// Host-side helper: translate the result of a launch into a status.
static inline int32_t k16v8_launch_status() {
  return cudaGetLastError() == cudaSuccess ? K16V8_OK : K16V8_ERR_CUDA;
}

// SM count of the current device, cached per device (host only).
static inline int k16v8_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = sms;
  return sms;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous grid of the stream drains; every k16v8 kernel executes
// griddepcontrol.wait before it reads anything, so ordering is unchanged.
template <typename... KArgs, typename... Args>
static inline int32_t k16v8_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                       size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess
             ? K16V8_OK
             : K16V8_ERR_CUDA;
}

static inline bool k16v8_aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}
