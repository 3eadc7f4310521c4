// pkv_device.cuh -- device helpers shared by the libpkv kernels (sm_103a).
//
// Inline PTX for the pieces the kernels build on: shared-memory mbarriers with
// transaction counting (the tiled TMA copies of pkv_tc.cuh complete on them),
// 16-byte cp.async copies, bounded waits that report a timeout instead of
// hanging, and the first-error-wins status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Geometry the kernels are specialised for.
constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;
constexpr int kQHeads = 16;
constexpr int kKVHeads = 8;
constexpr int kGroup = kQHeads / kKVHeads;                 // query heads per KV head
constexpr int kTileBytes = kPageSize * kHeadDim * 2;        // one (page, KV head) tile of K or V: 4 KiB
constexpr int kRowBytes = kHeadDim * 2;                     // one K or V row: 256 B

// A wait that has not completed after this many SM clock cycles (about one
// second at the GB300's clocks) gives up and reports PKV_ERR_DEVICE_TIMEOUT.
constexpr long long kWaitLimitCycles = 2000000000LL;

constexpr float kLog2e = 1.4426950408889634f;

// ----------------------------------------------------------------------------
// status word
// ----------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor in the stream is finishing.
// grid_dependency_wait() blocks until the predecessor grid has completed and
// its memory is visible; every kernel here calls it before touching any
// argument buffer. allow_dependents() lets the successor start launching.
// Both are no-ops for a normal launch.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Launch with programmatic stream serialisation allowed.
template <typename Kernel, typename... Args>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ----------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA copies).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy global writes before its later
// async-proxy (TMA copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the barrier's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete. Returns false (and leaves the
// barrier alone) if it has not completed within `limit` SM clock cycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit = kWaitLimitCycles) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// 16-byte asynchronous copy global -> shared (cp.async, generic proxy); the
// issuing thread waits with cp_async_wait_all (a compiler memory barrier), the
// other threads after a CTA barrier.
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gmem_src));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------------------
// loads and conversions
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// bf16 pair (element 2i in the low half, 2i+1 in the high half) -> two floats, exactly.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// 2^x on the MUFU unit (x = -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace pkv
