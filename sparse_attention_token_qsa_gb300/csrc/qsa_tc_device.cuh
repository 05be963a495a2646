// Device helpers of the tcgen05 kernels that stream key tiles with TMA: the
// mbarrier operations, bounded waits, the 2-D tile copy, the 128-byte
// swizzled K-major shared-memory descriptor, the MMA, its commit, the TMEM
// load of a lane's four head columns, and a NaN-keeping relu.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <stdint.h>

namespace qsa {

// A wait's hardware suspend hint, in ns: the wait ends early when its phase
// completes.
constexpr uint32_t kTcSuspendNs = 500;

__device__ __forceinline__ uint32_t sm32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}

// Bounded wait on a phase: a non-blocking test, then sleeps of up to
// kTcSuspendNs that end early when the phase completes.  Gives up (raising
// the abort flag) once `limit` cycles have passed, or when another role
// already gave up.
__device__ inline bool tc_wait(uint32_t mb, uint32_t parity, long long limit,
                        volatile int32_t *abort_flag) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mb), "r"(parity)
        : "memory");
    if (ok) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (clock64() - t0 > limit) {
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(mb), "r"(parity), "r"(kTcSuspendNs)
        : "memory");
    if (ok) return true;
  }
}

// The same wait made warp-uniform: lane 0 waits, the verdict is broadcast.
__device__ __forceinline__ bool tc_warp_wait(uint32_t mb, uint32_t parity, long long limit,
                                             volatile int32_t *abort_flag) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(mb, parity, limit, abort_flag) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, descriptor version 1 (sm_100 family).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// This thread's TMEM lane, four consecutive columns (the four heads).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3])
               :
               : "memory");
}

// relu that keeps NaN (max.NaN returns NaN when either input is NaN)
__device__ __forceinline__ float relu_nan(float d) {
  float r;
  asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(d));
  return r;
}

}  // namespace qsa
