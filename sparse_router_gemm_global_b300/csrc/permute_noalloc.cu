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
// stand-in object); its device address is taken with cudaGetSymbolAddress once per CUDA context,
// with that context current, on the first call made in it.  The cache is keyed on the current
// driver context (cuCtxGetCurrent, looked up through the runtime like the tensor-map encoder),
// so a caller that makes its own context current on a device gets that context's address, not
// the primary context's.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "validate.cuh"

namespace moge {
namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;  // chunks * N int32 counts
constexpr int kMaxContexts = 64;

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

std::mutex g_mutex;
struct CachedAddress {
    CUcontext ctx;
    int32_t *ptr;
};
CachedAddress g_cache[kMaxContexts] = {};
int g_cached = 0;

// Device address of g_permute_scratch in the current context (nullptr on failure).
int32_t *scratch_in_current_context() {
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ctx)
        for (int i = 0; i < g_cached; ++i)
            if (g_cache[i].ctx == ctx) return g_cache[i].ptr;
    // first call in this context; with no context current yet, the lookup itself makes the
    // current device's primary context current (as every runtime call does), then it is read
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess || !ptr) return nullptr;
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return nullptr;
    if (g_cached < kMaxContexts) g_cache[g_cached++] = {ctx, static_cast<int32_t *>(ptr)};
    return static_cast<int32_t *>(ptr);
}

}  // namespace
}  // namespace moge

extern "C" moge_status_t moge_permute_noalloc(const moge_config_t *cfg, const int32_t *topk_idx, const void *x,
                                              int32_t *counts, int32_t *offsets, int32_t *pair_row,
                                              int32_t *row_token, void *x_perm, moge_stream_t stream) {
    using namespace moge;
    // the same checks as moge_permute
    moge_status_t s = check_permute_args(cfg, topk_idx, x, counts, offsets, pair_row, row_token, x_perm);
    if (s != MOGE_OK) return s;
    const moge_config_t &c = *cfg;
    const int64_t K = c.M * c.k_per_group;
    const bool gather = x && x_perm;
    // the static array bounds the problem size: one int32 count per (token chunk, expert)
    const int64_t chunks = cdiv(c.T > 0 ? c.T : 1, kPermuteChunk);
    if ((size_t)(chunks * c.N) * sizeof(int32_t) > kNoAllocScratchBytes) return MOGE_ERR_UNSUPPORTED;
    int32_t *scratch = scratch_in_current_context();
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
