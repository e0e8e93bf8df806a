// pkv_pipeline.cuh -- pieces of the warp-specialised tcgen05 decode kernels'
// pipelines: an mbarrier wait that is bounded and gives up once any role of
// the CTA has aborted, and a barrier over the 128 softmax threads that also
// ORs a predicate.
#pragma once

#include <cstdint>

#include "pkv_device.cuh"

namespace pkv {

// Bounded wait for the phase of `bar` with the given parity.  Gives up
// (false) when another role has set *abort_flag, or after limit_ns, in
// which case it raises PKV_DEV_TIMEOUT and sets *abort_flag for the others.
__device__ __forceinline__ bool pipe_wait(uint32_t bar, uint32_t parity, uint32_t *status,
                                          volatile int *abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - start > limit_ns) {
            raise_status(status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// Named barrier `id` over `threads` threads (whole warps); every participant
// gets the OR of their predicates.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; "
        "selp.u32 %0, 1, 0, q; }"
        : "=r"(r) : "r"(uint32_t(pred)), "r"(id), "r"(threads) : "memory");
    return r != 0;
}

// Named barrier 1 over the 128 softmax threads; every participant gets the
// OR of their predicates.
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, 128, p; "
        "selp.u32 %0, 1, 0, q; }"
        : "=r"(r) : "r"(uint32_t(pred)) : "memory");
    return r != 0;
}

}  // namespace pkv
