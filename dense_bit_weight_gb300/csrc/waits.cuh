// waits.cuh -- bounded mbarrier waits shared by the TMA-fed kernels.
//
// Every wait on a copy or on another warp ends: after about a second without
// progress the waiting thread raises its CTA's abort flag and the device error
// word (GEMM_ERR_DEVICE_TIMEOUT) and returns false, so the kernel can drain
// its own copies and exit with the context still usable.
#pragma once

#include <stdint.h>

#include "../../include/dbw_gemm.h"
#include "ptx.cuh"

namespace dbw {

constexpr uint64_t kTimeoutNs = 1000000000ull;

// Bounded wait on an mbarrier phase.  The thread is suspended in hardware
// between polls (woken as soon as the phase completes), and every poll checks
// the CTA's abort flag and the 1-second limit; on expiry it raises the abort
// flag and the device error word and returns false.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         int *d_error)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
        if (ptx::mbar_try_wait_suspend(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1u;
            atomicExch(d_error, (int)GEMM_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// The same wait by every lane of a converged warp, with a warp-uniform result
// (a lane that timed out makes the whole warp give up), so the warp can go on
// to .sync.aligned tensor-memory operations and elected MMA issue together.
// (Polling from lane 0 alone and broadcasting the outcome measured slower.)
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              int *d_error)
{
    const bool ok = wait_bar(bar, parity, abort_flag, d_error);
    return __all_sync(0xffffffffu, ok);
}

// Consume a probe taken earlier with mbar_test_wait: if any lane saw the phase
// incomplete, the warp falls back to the bounded blocking wait.
__device__ __forceinline__ bool settle_warp(bool probe, uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                            int *d_error)
{
    if (__all_sync(0xffffffffu, probe)) return true;
    return wait_bar_warp(bar, parity, abort_flag, d_error);
}

// One arrival for the whole (converged) warp, after every lane's prior
// accesses: the barrier counts warps, not threads.
__device__ __forceinline__ void arrive_warp(uint32_t bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
}

// A barrier among several warps built on an mbarrier whose count is the
// number of warps: every warp arrives once, then waits for the phase with the
// bounded wait, so a warp that gave up elsewhere can never leave the others
// stuck (a named barrier, bar.sync, has no time limit).  `phase` is the
// caller's running parity of this barrier.  Returns false on expiry or abort.
__device__ __forceinline__ bool group_sync_warp(uint32_t bar, uint32_t &phase, volatile uint32_t *abort_flag,
                                                int *d_error)
{
    arrive_warp(bar);
    const bool ok = wait_bar_warp(bar, phase, abort_flag, d_error);
    phase ^= 1u;
    return ok;
}

// Wait without looking at the abort flag (used when draining before exit).
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait_suspend(bar, parity, 100000u))
        if (ptx::global_timer_ns() - t0 > kTimeoutNs) return;
}

}  // namespace dbw
