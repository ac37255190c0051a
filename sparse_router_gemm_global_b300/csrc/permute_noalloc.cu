// moge_permute_noalloc: the permutation with its scratch in a static device array, for
// callers that have no workspace to hand over.
//
// Some callers of this library cannot allocate device memory: a serving runtime whose memory
// pool already owns all of HBM and hands a plugin only its input and output buffers, or a
// latency-critical loop that must not call cudaMalloc (which can synchronise the device).
// For them the per-chunk expert counts live in g_permute_scratch below instead of the caller's
// workspace.  The array is a file-scope __device__ variable, so every GPU that loads this
// library holds it (kNoAllocScratchBytes) until the process exits.
//
// Host code may not use the array's name as a device address (on the host it names a
// stand-in object); its device address is taken with cudaGetSymbolAddress once per device,
// with that device current, on the first call made on that device.
#include <mutex>

#include "common.cuh"

namespace moge {
namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;  // chunks * N int32 counts
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

std::mutex g_mutex;
int32_t *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device (nullptr on failure).
int32_t *scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = static_cast<int32_t *>(ptr);
    }
    return g_scratch_ptr[dev];
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace moge

extern "C" moge_status_t moge_permute_noalloc(const moge_config_t *cfg, const int32_t *topk_idx, const void *x,
                                              int32_t *counts, int32_t *offsets, int32_t *pair_row,
                                              int32_t *row_token, void *x_perm, moge_stream_t stream) {
    using namespace moge;
    if (!cfg) return MOGE_ERR_INVALID_ARGUMENT;
    const moge_config_t &c = *cfg;
    if (c.T < 0 || c.N < 1 || c.M < 1 || c.N % c.M != 0) return MOGE_ERR_INVALID_ARGUMENT;
    if (c.k_per_group < 1 || c.k_per_group > c.N / c.M) return MOGE_ERR_INVALID_ARGUMENT;
    const int64_t K = c.M * c.k_per_group;
    if (c.N > 1024 || K > 1024 || c.T > ((int64_t)1 << 31) / K - 1) return MOGE_ERR_UNSUPPORTED;
    const bool gather = x && x_perm;
    if (gather) {
        if (c.d < 1) return MOGE_ERR_INVALID_ARGUMENT;
        if (c.act_dtype != MOGE_F32 && c.act_dtype != MOGE_BF16) return MOGE_ERR_UNSUPPORTED;
        if (c.d % (c.act_dtype == MOGE_BF16 ? 8 : 4) != 0) return MOGE_ERR_UNSUPPORTED;
        if (!row_token) return MOGE_ERR_INVALID_ARGUMENT;
    }
    if (!topk_idx || !counts || !offsets) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)topk_idx, x, (const void *)counts, (const void *)offsets,
                          (const void *)pair_row, (const void *)row_token, (const void *)x_perm})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    // the static array bounds the problem size: one int32 count per (token chunk, expert)
    const int64_t chunks = cdiv(c.T > 0 ? c.T : 1, kPermuteChunk);
    if ((size_t)(chunks * c.N) * sizeof(int32_t) > kNoAllocScratchBytes) return MOGE_ERR_UNSUPPORTED;
    int32_t *scratch = scratch_on_current_device();
    if (!scratch) return MOGE_ERR_CUDA;
    // Every count the scan reads is written earlier in the same call, so nothing in the array
    // has to start at zero; calls that overlap on the GPU share the array and race.
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_permute(topk_idx, c.T, K, c.N, counts, offsets, pair_row, row_token, scratch,
                                   nullptr, st);
    if (e == cudaSuccess && gather)
        e = pair_row ? launch_scatter_rows(x, pair_row, c.T, K, 0, 0, c.d, c.act_dtype, x_perm, st)
                     : launch_gather_rows(x, row_token, offsets, c.N, c.T * K, c.d, c.act_dtype, x_perm, st);
    return e == cudaSuccess ? MOGE_OK : MOGE_ERR_CUDA;
}
