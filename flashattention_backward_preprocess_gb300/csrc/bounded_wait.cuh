// bounded_wait.cuh -- mbarrier waits with a time limit, shared by the main
// backward kernel and the wait self-test.  A wait that runs out raises the
// CTA's abort flag, records kErrTimeout in the device error word and returns
// false, so the kernel can unwind (wait for its own copies / MMAs in flight,
// free TMEM) instead of hanging the GPU.
#pragma once

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {

constexpr uint64_t kWaitLimitNs = 10ull * 1000 * 1000 * 1000;  // 10 s

// Bounded wait.  Returns false (and raises the CTA abort flag and the device
// error word) if the phase did not complete in time or another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err, uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (++spins % 64 == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform bounded wait: every lane waits (each gets the acquire), the
// warp then agrees, so a timeout seen by one lane makes the whole warp leave.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err, uint64_t limit_ns = kWaitLimitNs) {
    const bool ok = wait_bar(bar, parity, abort_flag, err, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait until a counter in global memory, advanced by other CTAs of the same launch
// (release stores), reaches `want`; acquire ordering on success.  Polls every ~100 ns.
// The CTAs waited for took lower start-order tickets, so they are already running.
__device__ __forceinline__ bool wait_counter(const unsigned int* ctr, unsigned int want,
                                             volatile int* abort_flag, unsigned int* err,
                                             uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::ld_acquire_gpu(ctr) >= want) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        __nanosleep(100);
        if (ptx::ld_acquire_gpu(ctr) >= want) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// Wait used while shutting down after an abort: bounded, no flag checks.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > kWaitLimitNs) return;
    }
}

}  // namespace fa
