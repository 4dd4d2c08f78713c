// mbarrier.cuh — shared-memory barrier helpers of libvsf's pipelined
// kernels (sm_103a inline PTX): initialisation, arrivals with transaction
// bytes, and bounded waits. Included inside a namespace by each translation
// unit that uses it.
//
// Every wait is bounded in wall-clock time (the global timer). A timeout is
// sticky per CTA: the first wait that runs out sets bit 1 of the caller's
// device error word and the CTA's shared stop flag, and from then on every
// wait of that CTA returns false at once, so a broken pipeline ends within a
// few limits instead of one limit per wait. mbar_drain ignores the flag; it
// is for the copies a CTA must see land before it exits.
#pragma once

constexpr uint32_t kSuspendNs = 1u << 20;        // sleep limit of one barrier test
constexpr uint64_t kWaitNs = 2000000000ull;       // bound of one wait: 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One potentially blocking test of the phase with the given parity: the
// thread may sleep until the phase completes or kSuspendNs pass, so a
// waiting warp issues a few instructions per wait instead of spinning.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity. Returns false at once if
// the CTA's stop flag is set, or after limit_ns (kWaitNs unless given) of
// wall-clock time (global timer), having then set the stop flag and bit 1 of
// the error word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err,
                                          volatile uint32_t* stop, uint64_t limit_ns = kWaitNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (*stop == 0u) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      *stop = 1u;
      atomicOr(err, 2u);
      return false;
    }
  }
  return false;
}

// The same at cluster scope (acquire), for barriers that peers arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, unsigned* err,
                                                  volatile uint32_t* stop) {
  if (mbar_try_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (*stop == 0u) {
    if (mbar_try_cluster(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) {
      *stop = 1u;
      atomicOr(err, 2u);
      return false;
    }
  }
  return false;
}

// Wait for an issued copy to land, ignoring the stop flag, until the global
// timer passes `deadline`; used once per slot before the CTA exits.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t deadline,
                                           unsigned* err) {
  while (!mbar_try(bar, parity)) {
    if (global_ns() > deadline) {
      atomicOr(err, 2u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

