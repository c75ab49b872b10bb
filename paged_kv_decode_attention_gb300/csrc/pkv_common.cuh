// pkv_common.cuh -- shared device helpers of libpkv (sm_103a).
//
// Inline-PTX wrappers for the pieces the kernels build on: mbarrier-tracked
// bulk (TMA) copies from global into shared memory, bounded barrier waits,
// BF16 unpacking and the base-2 exponential.  Every spin-wait here gives up
// after kWaitLimitNs of wall time and reports failure to its caller, which
// records PKV_DEVERR_TIMEOUT in the device error word instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;                       // tokens per physical block
constexpr int kHeadDim = 128;                        // dims per head
constexpr int kGroup = 4;                            // query heads per KV head
constexpr int kTileBytes = kBlockSize * kHeadDim * 2;  // one (block, kv head) tile: 4 KiB
// q8_0 tile of one (block, kv head): int8 codes [16][128], then the FP16
// scale of every 32-value group, [16][4]: 64 groups of 34 bytes.
constexpr int kQ8CodeBytes = kBlockSize * kHeadDim;                  // 2048
constexpr int kQ8TileBytes = kQ8CodeBytes + kBlockSize * kHeadDim / 32 * 2;  // 2176
// FP8 (E4M3) tile of one (block, kv head): codes [16][128], no scale.
constexpr int kFp8TileBytes = kBlockSize * kHeadDim;  // 2048
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // 2 s: a healthy wait takes microseconds

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy, TMA, tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy
// (bulk copy, TMA) reads of the same memory, issued after a synchronisation.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the same condition (for a thread that polls several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete; false once limit_ns
// of wall time has passed without it.
__device__ __forceinline__ bool mbar_wait_limited(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// The kernels' wait: bounded by kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_limited(bar, parity, kWaitLimitNs);
}

// L2 policy for data read exactly once (streamed KV tiles).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// BF16 pair (low half = element 0) to two floats: BF16 is the top half of binary32.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two floats to a BF16 pair, round to nearest even (hardware conversion).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x (hardware approximation; 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void report(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// q8_0 quantisation of one 128-value row by one warp ("Chapter 8: Inference
// Optimization" §8.4.2, Fig. 8-23: groups of 32 values share one FP16
// scale, 8-bit codes).  Lane l holds values 4l .. 4l+3 (two BF16 pairs), so
// lanes 8g .. 8g+7 hold group g.  Per group d = max|x| / 127 and code =
// round-half-away-from-zero(x * (1/d)), every step one IEEE-rounded FP32
// operation (a zero group gets d = 0 and codes 0).  Returns the lane's 4
// codes (byte k = value 4l + k) and sets d, the group's scale before its
// FP16 rounding (the stored scale is __float2half_rn(d)).
__device__ __forceinline__ uint32_t q8_0_quantize_lane(uint2 w, float& d) {
  const float x0 = bf16_lo(w.x), x1 = bf16_hi(w.x), x2 = bf16_lo(w.y), x3 = bf16_hi(w.y);
  float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  d = __fdiv_rn(amax, 127.0f);
  const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
  const int c0 = static_cast<int>(roundf(__fmul_rn(x0, id)));
  const int c1 = static_cast<int>(roundf(__fmul_rn(x1, id)));
  const int c2 = static_cast<int>(roundf(__fmul_rn(x2, id)));
  const int c3 = static_cast<int>(roundf(__fmul_rn(x3, id)));
  return (static_cast<uint32_t>(c0) & 0xffu) | ((static_cast<uint32_t>(c1) & 0xffu) << 8) |
         ((static_cast<uint32_t>(c2) & 0xffu) << 16) | (static_cast<uint32_t>(c3) << 24);
}

}  // namespace pkv

namespace pkv {

// ---- thread-block clusters (distributed shared memory) ----
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier: every thread of every CTA in the cluster; release /
// acquire order shared-memory writes before / reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_to_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Hint: bring the 128-byte line holding `p` into this SM's L1.
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

// ---- programmatic dependent launch ----
// Wait until the grids this one depends on have completed and their writes
// are visible (a no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid in the stream launch its CTAs (they still wait in
// pdl_wait before touching this grid's results).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// BF16 pair to a float2 (element 0 in .x).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

}  // namespace pkv
