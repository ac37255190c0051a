// Bounded mbarrier waits shared by the tcgen05 kernels.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moge {
namespace ptx {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s per wait

// Wait for the phase of the given parity.  Gives up (returns false) when the CTA-wide abort
// flag is raised by another role, or after kWaitTimeoutNs, in which case it raises the flag
// itself and records MOGE_ERR_TIMEOUT in the workspace status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         uint32_t *status, uint64_t timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 31) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > timeout_ns || n > (1u << 30)) {
                *abort_flag = 1;
                raise_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// wait_bar with cluster-scope acquire (a phase completed by another CTA of the cluster).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                 uint32_t *status, uint64_t timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_acq_cluster(bar, parity)) return true;
        if ((n & 31) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > timeout_ns || n > (1u << 30)) {
                *abort_flag = 1;
                raise_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: used at exit for copies and MMAs already issued.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint32_t *status) {
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 0; !mbar_try_wait(bar, parity); ++n) {
        if ((n & 31) == 31 && (globaltimer() - t0 > kWaitTimeoutNs || n > (1u << 30))) {
            raise_status(status, kStatusTimeout);
            return;
        }
    }
}

}  // namespace ptx
}  // namespace moge
