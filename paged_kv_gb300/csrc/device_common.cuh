// Device helpers shared by the sm_103a kernels: mbarrier and bulk-copy
// primitives (inline PTX), streaming loads, the order-preserving float key,
// and warp-level scans.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Orders mbarrier initialisation before later arrivals and bulk-copy
// completions on it.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrives (count 1) on `bar` with release semantics at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar))
               : "memory");
}

// Arrives on `bar` and adds `bytes` to the transaction count it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` transaction bytes on `bar`.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Tests phase `parity` of this CTA's mbarrier (acquire at CTA scope).  May
// suspend briefly; true once the phase is complete.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Global nanosecond timer (bounds every wait).
__device__ __forceinline__ long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return static_cast<long long>(t);
}

// ----------------------------------------------------------------- loads

// 16-byte streaming load that does not allocate in L1 (each logit is read
// from HBM exactly once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ----------------------------------------------------------------- float helpers

// Maximum that propagates NaN (PTX max.NaN), so one reduction both finds the
// row maximum and detects a NaN anywhere in the row.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 2^x with the hardware approximation (MUFU.EX2), subnormal results flushed.
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Order-preserving map from a float to uint32: a > b  <=>  key(a) > key(b)
// for non-NaN a, b.  -0 is folded onto +0 first (x + 0 is +0 for x = -0), so
// equal values have equal keys.
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(u);
}

// ----------------------------------------------------------------- cp.async

// 16-byte asynchronous copy global -> shared (L2 only, no L1 allocation).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// Waits until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ----------------------------------------------------------------- warp

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Warp sum of 64-bit unsigned values in three 32-bit reductions (fields of
// 24, 24 and 16 bits, whose lane sums cannot overflow).  Exact whenever the
// total fits in 64 bits.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
  const uint32_t lo = __reduce_add_sync(kFull, static_cast<uint32_t>(v & 0xffffffull));
  const uint32_t mid = __reduce_add_sync(kFull, static_cast<uint32_t>((v >> 24) & 0xffffffull));
  const uint32_t hi = __reduce_add_sync(kFull, static_cast<uint32_t>(v >> 48));
  return (static_cast<unsigned long long>(hi) << 48) + (static_cast<unsigned long long>(mid) << 24) +
         lo;
}

// Inclusive prefix over lanes: lane l gets v_0 + ... + v_l.  Used by code
// that runs once per row, where instruction fetch sets the pace: a loop
// keeps one copy of the step's code.
template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v, int lane) {
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Inclusive suffix over lanes: lane l gets v_l + ... + v_31.
template <typename T>
__device__ __forceinline__ T warp_suffix_scan(T v, int lane) {
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_down_sync(kFull, v, o);
    if (lane + o < 32) v += n;
  }
  return v;
}

}  // namespace pkv
