// Bounded waits of the tcgen05 kernels: every mbarrier wait gives up after a
// bound, records a timeout in the library's status word and makes the CTA abort.
#pragma once

#include <stdint.h>

#include "qwp_internal.h"
#include "qwp_ptx.cuh"

namespace qwp {

struct Ctl {
    uint32_t *abort;  // shared-memory flag
    uint32_t *status;
    uint64_t timeout_cycles;  // main-loop waits
    uint64_t drain_cycles;    // waits for the CTA's own work in flight
};

// Bounded wait on phase `parity` of `bar`.  False if it timed out or the CTA is
// aborting (this CTA or, through the status word, any other); a timeout
// records `where` in the status word.  The loop mostly sits in try_wait (which
// suspends the thread in hardware, often until the phase completes, so a wait
// takes few polls).  The bound is kept in SM clock cycles (clock64, a cheap
// register read, looked at after every unsuccessful poll); the global status
// word is read every 64 polls.  Waits that do not honour an abort (a CTA
// waiting for its own copies and MMAs in flight before it exits) always allow
// the default bound.
// kLazy waits sleep between polls (roles off the critical path, which should
// not take issue slots from the warps that are on it).
template <bool kCluster = false, bool kLazy = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &ctl,
                                         uint32_t where, bool honour_abort = true) {
    auto poll = [&] { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = clock64();
    const uint64_t limit = honour_abort ? ctl.timeout_cycles : ctl.drain_cycles;
    for (uint32_t it = 1;; ++it) {
        if (kLazy) __nanosleep(256);
        if (poll()) return true;
        if (honour_abort && *reinterpret_cast<volatile uint32_t *>(ctl.abort)) return false;
        if (static_cast<uint64_t>(clock64()) - t0 > limit) {
            *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;
            atomicCAS(ctl.status, 0u, 0x100u | where);
            return false;
        }
        if ((it & 63u) == 0 && honour_abort &&
            (*reinterpret_cast<volatile uint32_t *>(ctl.status) & kStatusTimeoutMask)) {
            *reinterpret_cast<volatile uint32_t *>(ctl.abort) = 1u;  // another CTA failed
            return false;
        }
    }
}

// A wait on a barrier that peers of the cluster arrive on (acquire at cluster
// scope), by the epilogue warps (lazy).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, const Ctl &ctl, uint32_t where) {
    return wait_bar<true, true>(bar, parity, ctl, where);
}

__device__ __forceinline__ bool aborted(const Ctl &ctl) {
    return *reinterpret_cast<volatile uint32_t *>(ctl.abort) != 0;
}

// A wait bound in SM clock cycles: at 2.1 cycles per ns (above GB300's highest SM
// clock, 2.07 GHz) a bound never ends sooner than its time in ns; at a lower
// clock it lasts proportionally longer.
inline uint64_t ns_to_cycles(uint64_t ns) { return ns * 21 / 10 + 1; }

}  // namespace qwp
