// Bounded waits and the device status word shared by every kernel.
//
// No kernel of this library waits without a limit. A wait that runs past its
// limit records AP_ERR_DEVICE_TIMEOUT and the site that gave up in the status
// word (first error wins), raises the CTA's abort flag so the other roles stop
// too, and returns false; the kernel then drains the copies it issued (again
// with a limit) and returns normally. No trap, no assert, no endless loop.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace ap {

// Status word layout: bits 0..7 the ap_status code, bits 8..15 the site.
enum WaitSite : uint32_t {
    SITE_RING_PRODUCER_EMPTY = 1,
    SITE_RING_CONSUMER_FULL = 2,
    SITE_RING_DRAIN = 3,
    SITE_EX_LOADER_CREDIT = 4,
    SITE_EX_PUSHER_LOADED = 5,
    SITE_EX_RECEIVER_FULL = 6,
    SITE_EX_DRAIN = 7,
    SITE_RING_TENSOR_ALIGN = 8,
    SITE_MASKED_CODE = 9,
    SITE_CHECK_PRODUCER = 10,
    SITE_CHECK_CONSUMER = 11,
    SITE_EX_PUSHER_CREDIT = 12,
};

constexpr uint32_t kStatusTimeout = 9;  // AP_ERR_DEVICE_TIMEOUT
constexpr uint32_t kStatusAlign = 3;    // AP_ERR_ALIGN
constexpr uint32_t kStatusShape = 2;    // AP_ERR_SHAPE

__device__ __forceinline__ void raise_timeout(uint32_t* status, uint32_t site, volatile int* abort_flag) {
    atomicCAS(status, 0u, kStatusTimeout | (site << 8));
    if (abort_flag) *abort_flag = 1;
}

enum WaitResult : int { WAIT_OK = 0, WAIT_TIMEOUT = 1, WAIT_ABORTED = 2 };

// Wait for the phase with `parity` of the CTA-local barrier `bar`. Gives up
// with WAIT_TIMEOUT after `timeout_ns`, or with WAIT_ABORTED as soon as the
// CTA's abort flag is set (nullptr: ignore the flag).
template <bool kClusterScope>
__device__ __forceinline__ int wait_phase(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile int* abort_flag) {
    auto probe = [&]() {
        return kClusterScope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (probe()) return WAIT_OK;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (probe()) return WAIT_OK;
        if (abort_flag != nullptr && *abort_flag) return WAIT_ABORTED;
        if (ptx::globaltimer_ns() - t0 > timeout_ns) return WAIT_TIMEOUT;
    }
}

// A drain: before a kernel leaves, it waits for the copies it issued, so that
// none is still reading or writing a CTA's shared memory when the CTA exits.
// After an abort (a wait elsewhere gave up) the barrier of such a copy may
// never complete: its receiver no longer consumes, or fault injection
// inflated the bytes it expects, although the bytes themselves still land.
// The drain then stops at once and holds the thread for a grace period far
// longer than an issued copy takes to finish, instead of waiting out the full
// limit for every remaining copy. Returns false when the drain should stop.
constexpr uint64_t kDrainGraceNs = 100000;

template <bool kClusterScope>
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns, uint32_t* status,
                                           uint32_t site, volatile int* abort_flag) {
    const int w = wait_phase<kClusterScope>(bar, parity, timeout_ns, abort_flag);
    if (w == WAIT_OK) return true;
    if (w == WAIT_TIMEOUT) raise_timeout(status, site, abort_flag);
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < kDrainGraceNs) {
    }
    return false;
}

}  // namespace ap
