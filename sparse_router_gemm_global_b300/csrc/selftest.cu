// Self-test of the failure detection of the bounded waits (no counterpart on the pages).
//
// Every wait of the tcgen05 kernels on an mbarrier gives up after a time limit: it then raises
// the CTA's abort flag (which ends the other roles' waits at once) and records MOGE_ERR_TIMEOUT
// in the workspace status word instead of hanging the GPU.  This kernel exercises exactly that
// routine (wait_bar) on barriers that nothing ever completes: warp 0 waits with the given limit
// and times out; warp 1 waits on another barrier with no limit of its own and must leave through
// the abort flag.  Nothing faults, traps or waits for longer than the limit.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_wait.cuh"

namespace moge {
namespace {

__global__ void bounded_wait_selftest_kernel(uint32_t *status, uint64_t timeout_ns, uint32_t *result) {
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bar[1]), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort_v = &abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0 && warp < 2) {
        // phase 0 of a barrier that expects one arrival nobody makes never completes
        const bool ok = warp == 0 ? ptx::wait_bar(ptx::smem_u32(&bar[0]), 0, abort_v, status, timeout_ns)
                                  : ptx::wait_bar(ptx::smem_u32(&bar[1]), 0, abort_v, status, 4 * timeout_ns);
        result[warp] = ok ? 1u : 0u;  // both must give up: 0
    }
    __syncthreads();
    if (threadIdx.x == 0) result[2] = (uint32_t)abort_flag;
}

}  // namespace
}  // namespace moge

extern "C" moge_status_t moge_selftest_bounded_wait(void *ws, uint64_t timeout_ns, uint32_t *result,
                                                    moge_stream_t stream) {
    using namespace moge;
    if (!ws || !result || ((uintptr_t)ws & 255u) != 0 || ((uintptr_t)result & 15u) != 0)
        return MOGE_ERR_INVALID_ARGUMENT;
    if (timeout_ns == 0 || timeout_ns > 1000000000ull) return MOGE_ERR_INVALID_ARGUMENT;  // at most 1 s
    bounded_wait_selftest_kernel<<<1, 64, 0, (cudaStream_t)stream>>>((uint32_t *)ws, timeout_ns, result);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOGE_OK : MOGE_ERR_CUDA;
}
