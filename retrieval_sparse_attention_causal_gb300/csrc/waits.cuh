// Bounded waits on mbarriers for the warp-specialised tcgen05 kernels, and a tensor-map
// prefetch.  Every wait gives up after a limit, records the wait site in the error word and
// raises the CTA's abort flag, so that a protocol fault can neither hang a kernel nor let a
// role run on stale data.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "tc.cuh"

namespace gca {

constexpr uint32_t kWaitLimit = 1u << 21;

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Bounded wait for phase `parity` of `bar` that gives up early once the CTA's abort flag
// is raised; on running out it records `site` (with CTA, tile, slot) and raises the flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag, ErrWord* err,
                                              int site, int tile, int slot) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (tc::mbar_try(bar, parity)) return true;
    if ((it & 15) == 15 && *reinterpret_cast<volatile int*>(abort_flag)) return false;
  }
  flag_timeout(err, site, blockIdx.x, tile, slot);
  atomicExch(abort_flag, 1);
  return false;
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One probe of phase `parity` of `bar` that lets the hardware park the thread until the
// phase completes, for at most `hint_ns` (so that a waiting warp takes no issue slots
// from the warps that work).
__device__ __forceinline__ bool mbar_try_park(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(tc::su32(bar)), "r"(parity), "r"(hint_ns));
  return done != 0;
}

// Bounded wait with parking, for kernels with many waiting warps: gives up once the CTA's
// abort flag is raised, or after kParkLimitNs of global time, recording `site` (with CTA,
// tile, slot) and raising the flag.
constexpr uint64_t kParkLimitNs = 2000000000ull;
__device__ __forceinline__ bool park_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag, ErrWord* err,
                                              int site, int tile, int slot) {
  if (tc::mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_park(bar, parity, 20000)) return true;
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (global_ns() - t0 > kParkLimitNs) break;
  }
  flag_timeout(err, site, blockIdx.x, tile, slot);
  atomicExch(abort_flag, 1);
  return false;
}

// The same bounded wait without parking (for the warp whose wake-up latency is on the
// critical path).
__device__ __forceinline__ bool spin_or_abort(uint64_t* bar, uint32_t parity, int* abort_flag, ErrWord* err,
                                              int site, int tile, int slot) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (tc::mbar_try(bar, parity)) return true;
    if ((it & 15) == 15) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (global_ns() - t0 > kParkLimitNs) break;
    }
  }
  flag_timeout(err, site, blockIdx.x, tile, slot);
  atomicExch(abort_flag, 1);
  return false;
}


}  // namespace gca
