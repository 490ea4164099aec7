// Device helpers shared by the layer's kernels (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/moe_layer.h"

namespace moe {

constexpr float kF16MaxFinite = 65504.0f;

// fp32 -> binary16 for stage outputs: round to nearest even, saturating at +-65504.
__device__ __forceinline__ __half f2h_sat(float v) {
  v = fminf(fmaxf(v, -kF16MaxFinite), kF16MaxFinite);
  return __float2half_rn(v);
}

// Two fp32 -> a binary16 pair (lo, hi), each as f2h_sat (round to nearest even,
// saturating at +-65504), in one conversion.
__device__ __forceinline__ __half2 f2h2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = r;
  return h;
}

__device__ __forceinline__ int clamp127(int v) { return max(-127, min(127, v)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max of non-negative values; every thread gets the result.
// `red` must hold blockDim.x / 32 floats.
__device__ __forceinline__ float block_max_nonneg(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0f;
  r = warp_max(r);
  __syncthreads();  // red may be reused by the caller
  return r;
}

// ---------------------------------------------------------------------------------
// mbarrier / TMA (inline PTX)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up (returns false) after about two
// seconds of wall time, which only a barrier that can never complete reaches.
// The clock is read only after a few hundred unsuccessful polls.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *count >= target, a count that other CTAs of the same grid raise
// (the fused SwiGLU's per-expert item counters): acquire loads between short sleeps;
// gives up (returns false) after limit_ns of wall time.
__device__ __forceinline__ bool count_wait_bounded(const int32_t* count, int target,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  if (ld_acquire(count) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(256);
    if (ld_acquire(count) >= target) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// 2-D tiled TMA load of box {x: inner, y: outer} at coordinates (x, y) into smem,
// completing `bar`'s transaction count.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Four rows y.x..y.w of a 2-D tensor map whose box is one row high, `x` the first
// column: lands as four consecutive box rows at smem_dst (the map's swizzle applies
// as for a four-row tiled box at that address).
__device__ __forceinline__ void tma_gather4(void* smem_dst, const void* tmap, int32_t x, int4 y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y.x), "r"(y.y), "r"(y.z), "r"(y.w), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy of `bytes` contiguous global bytes into this CTA's shared memory,
// completing `bar`'s transaction count.  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes of this CTA's shared memory to global
// memory, in the thread's current bulk async-group.  Both addresses 16-byte aligned,
// bytes a multiple of 16; the shared source must have been written before a
// fence_proxy_async_smem() and a barrier with the writers.
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(gdst)),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until this thread's committed bulk stores have read their shared source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Status word at the start of a layer / GEMM workspace.
__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace moe
