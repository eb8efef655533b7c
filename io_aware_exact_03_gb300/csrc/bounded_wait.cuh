// Bounded mbarrier waits, shared by every kernel of the library.
//
// No wait inside a kernel can run forever: a waiting role gives up after
// `limit_ns` of global time, sets the CTA's abort flag and the kernel file's
// device status word (read back by attn_check_status as ATTN_ERR_TIMEOUT), and
// returns false; every other role sees the flag at its next wait and returns
// false too, so the CTA drains what it issued, frees TMEM and exits normally.
#pragma once

#include <stdint.h>

#include "attn_internal.h"
#include "tc_ptx.cuh"

namespace attn {
namespace {

// Slow path: poll, checking the abort flag and the clock every 32 polls.
__device__ __noinline__ bool bounded_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned long long limit_ns, unsigned* status) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Wait for the phase of parity `parity` of mbarrier `bar` to complete.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long limit_ns, unsigned* status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return bounded_wait_slow(bar, parity, abort_flag, limit_ns, status);
}

// Drain-only wait (used while aborting): bounded, never raises the flag.
__device__ __forceinline__ void bounded_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > limit_ns) return;
    }
}

}  // namespace
}  // namespace attn
