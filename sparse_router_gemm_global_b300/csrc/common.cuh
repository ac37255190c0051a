// Shared device/host helpers of the MoGE CUDA library (internal header).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "moge.h"

namespace moge {

// Kernel launch counter and per-thread stage events (instrumentation, api.cu).
void count_launches(int n);
void mark_stage(int stage, cudaStream_t s);

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch.  The layer's kernels are launched so that each may start (its
// prologue: barriers, TMEM, descriptor prefetch) while the previous kernel in the stream
// finishes; every such kernel calls pdl_wait() before it touches memory written by earlier
// work, and pdl_trigger() right after, which lets its own successor be scheduled.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Status word bits (first 4 bytes of the workspace).
enum : uint32_t {
    kStatusTimeout = 1u << 0,   // a bounded mbarrier wait gave up
    kStatusBadIndex = 1u << 1,  // an expert id outside [0, N) was skipped
};

__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

__host__ __device__ constexpr int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// First row and row count of expert e's segment [offsets[e], offsets[e+1]), clamped to the
// buffer's rows [0, rows): offsets that no permutation wrote (decreasing, negative or past the
// end) never lead a kernel to a row outside its buffers, nor to more tiles than the rows hold.
__device__ __forceinline__ void expert_segment(const int32_t *offsets, int e, int rows, int &begin, int &count) {
    begin = min(max(offsets[e], 0), rows);
    count = min(max(offsets[e + 1], begin), rows) - begin;
}

// SwiGLU activation silu(a) * u with silu(a) = a / (1 + exp(-a)).
// swiglu_fast uses the hardware exp2 approximation and the approximate division (a few fp32
// ulps; the bf16 tensor-core path rounds its output to bf16 anyway, and an IEEE division here
// costs the GEMM epilogue several times the instructions); swiglu_precise uses expf and an IEEE
// division (all-fp32 path).
__device__ __forceinline__ float swiglu_fast(float a, float u) { return __fdividef(a, 1.0f + __expf(-a)) * u; }
__device__ __forceinline__ float swiglu_precise(float a, float u) { return a / (1.0f + expf(-a)) * u; }

// ---------------------------------------------------------------------------------------------
// Workspace layout (every region 256-byte aligned).  Computed identically on every call.
// ---------------------------------------------------------------------------------------------
struct WsLayout {
    size_t status, logits, idx, gate, counts, offsets, pair_row, row_token, chunk_counts, x_perm, h, y_perm, total;
};

constexpr int kPermuteChunk = 256;   // tokens per permutation block

// The first kStatusPageBytes of the workspace must be zero before first use: the status word
// sits at byte 0 and the small-batch router's self-resetting counter at kTicketOffset.
constexpr int kStatusPageBytes = 4096;
constexpr int kTicketOffset = 256;
// Tile counters of the CTA-pair grouped GEMM launches (next tile, finished CTAs), one 256-byte
// slot per GEMM of the layer; each launch returns its pair to zero before it ends.
constexpr int kSchedGateUpOffset = 512;
constexpr int kSchedDownOffset = 768;
constexpr int kRouterTileRows = 128;
constexpr int kDesignSMs = 148;  // B300 SM count: sizes the router's split of the reduction

// Number of slices the tensor-core router splits its reduction over d into, so that small
// batches still spread over more SMs (1 = no split).  The slices of a tile form one thread-block
// cluster and are added in order through distributed shared memory: at most 8 (the portable
// cluster size), each at least 8 k-blocks of 64.  Deterministic in (T, d, N).
inline int router_kslices(int64_t T, int64_t d, int64_t N) {
    const int64_t mtiles = cdiv(T, kRouterTileRows), kblocks = cdiv(d, 64);
    if (T <= 0) return 1;
    int64_t s = kDesignSMs / mtiles;
    if (s > kblocks / 8) s = kblocks / 8;
    if (s > 8) s = 8;
    return s < 1 ? 1 : (int)s;
}

// Batches of at most kSmallRouteMaxT tokens are routed (and, inside the layer, permuted) by one
// CUDA-core launch (route_small.cu) when its shared-memory staging fits kSmallRouteMaxSmem.
constexpr int kSmallRouteMaxT = 64;
constexpr size_t kSmallRouteMaxSmem = 160 * 1024;
static_assert(kSmallRouteMaxT <= kPermuteChunk, "the small router permutes its tokens in one block");

// Tile plan of the bf16 grouped GEMM for `rows` (token, expert) rows over `experts` experts of a
// batch of T tokens.  Weights-as-M tiles stream each expert's weights at full MMA height with
// the expert's token rows as the MMA's N (16/32/64/128 per tile, several tiles for a larger
// expert); they suit batches whose experts hold few rows, where 256-row tokens-as-M tiles would
// be mostly padding.  With at most 32 tokens the GEMM gathers the token rows from x itself
// (TMA gather4, at most 8 copies per k-block); otherwise the rows are first copied to x_perm.
enum FfnTiles { kTilesSwap16 = 16, kTilesSwap32 = 32, kTilesSwap64 = 64, kTilesSwap128 = 128, kTilesPair = 256 };
constexpr int64_t kSwap64MaxMeanRows = 48;  // 64-token weights-as-M tiles while rows / experts <= this
constexpr int64_t kSwapMaxMeanRows = 104;   // 128-token weights-as-M tiles while rows / experts <= this
struct FfnPlan {
    int tiles;
    bool gather_in_gemm;
};
inline FfnPlan ffn_plan(int64_t T, int64_t rows, int64_t experts) {
    if (T <= 16) return {kTilesSwap16, true};
    if (T <= 32) return {kTilesSwap32, true};
    if (rows <= kSwap64MaxMeanRows * experts) return {kTilesSwap64, false};
    if (rows <= kSwapMaxMeanRows * experts) return {kTilesSwap128, false};
    return {kTilesPair, false};
}

// Whether the layer's gate/up GEMM reads the token rows from x itself (no x_perm); fp32 layers
// always read x_perm.
inline bool gathers_in_gemm(const moge_config_t &c, int64_t S = 0) {
    const int64_t rows = c.T * c.M * c.k_per_group + S * c.T;
    return c.act_dtype == MOGE_BF16 && ffn_plan(c.T, rows, c.N + S).gather_in_gemm;
}

// S shared experts (every token visits each of them; rows P + s*T + t) extend the expert index
// space to N + S and the rows to P + S*T.
inline WsLayout ws_layout(const moge_config_t &c, int64_t S = 0) {
    const int64_t K = c.M * c.k_per_group;
    const int64_t P = c.T * K;
    const int64_t rows = P + S * c.T;
    const size_t es = (c.act_dtype == MOGE_BF16) ? 2 : 4;
    const int64_t chunks = cdiv(c.T > 0 ? c.T : 1, kPermuteChunk);
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (size_t)round_up((int64_t)bytes, 256); return o; };
    L.status = take(kStatusPageBytes);
    L.logits = take((size_t)c.T * c.N * 4);
    L.idx = take((size_t)P * 4);
    L.gate = take((size_t)P * 4);
    L.counts = take((size_t)c.N * 4);
    L.offsets = take((size_t)(c.N + S + 1) * 4);
    L.pair_row = take((size_t)P * 4);
    L.row_token = take((size_t)rows * 4);
    L.chunk_counts = take((size_t)chunks * c.N * 4);
    // layers whose gate/up GEMM gathers token rows itself store no permuted copy of x
    L.x_perm = take(gathers_in_gemm(c, S) ? 0 : (size_t)rows * c.d * es);
    L.h = take((size_t)rows * c.I * es);
    L.y_perm = take((size_t)rows * c.d * es);
    L.total = off;
    return L;
}

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per (kernel, device) and
// size: the largest size set so far is remembered, so steady-state launches (and launches
// inside a CUDA graph capture) make no attribute call.  Defined in api.cu.
cudaError_t set_max_smem_impl(const void *kernel, size_t bytes);
template <typename Kernel> cudaError_t set_max_smem(Kernel kernel, size_t bytes) {
    return set_max_smem_impl(reinterpret_cast<const void *>(kernel), bytes);
}

// ---------------------------------------------------------------------------------------------
// Launchers (defined in the .cu files).  All return cudaGetLastError() after launching.
// ---------------------------------------------------------------------------------------------
cudaError_t launch_route_select(const float *logits, int64_t T, int64_t N, int64_t M, int64_t kpg,
                                bool global, int32_t *idx, float *gate, cudaStream_t s);
// cuTensorMapEncodeTiled from the driver (nullptr if unavailable); defined in ffn_tc.cu.
void *tensor_map_encoder();

// Fused tensor-core router (bf16, N <= 256): scores, softmax and selection in one launch.
cudaError_t launch_router_tc(const void *x, const void *w_r, const float *bias, int64_t T, int64_t d, int64_t N,
                             int64_t M, int64_t kpg, bool global, float *logits_out, int32_t *idx, float *gate,
                             uint32_t *status, cudaStream_t s);
// Small-batch router (any dtype): scores, softmax, selection and, when counts != nullptr, the
// permutation of all T tokens (+ group loads and imbalance score) in one launch.
bool route_small_fits(int64_t T, int64_t N, int64_t K, int64_t M, bool permute);
cudaError_t launch_route_small(const void *x, const void *w_r, const float *bias, int64_t T, int64_t d, int64_t N,
                               int64_t M, int64_t kpg, bool global, int dtype, float *scores, float *logits_out,
                               int32_t *idx, float *gate, uint32_t *ticket, uint32_t *status, int32_t *counts,
                               int32_t *offsets, int32_t *pair_row, int32_t *row_token, int32_t *group_load,
                               float *score, cudaStream_t s);
// Monte-Carlo imbalance study (imbalance_study.cu): N <= kStudyMaxExperts.
constexpr int64_t kStudyMaxExperts = 256;
size_t imbalance_study_smem_bytes(int64_t N, int64_t M);
cudaError_t launch_imbalance_study(int64_t T, int64_t N, int64_t M, int64_t kpg, int64_t batches, uint64_t seed,
                                   const float *bias, int32_t *loads_grouped, int32_t *loads_global,
                                   float *is_grouped, float *is_global, cudaStream_t s);
cudaError_t launch_router_logits_simt(const void *x, const void *w_r, const float *bias, int64_t T,
                                      int64_t d, int64_t N, int dtype, float *logits, cudaStream_t s);
cudaError_t launch_permute(const int32_t *idx, int64_t T, int64_t K, int64_t N, int32_t *counts,
                           int32_t *offsets, int32_t *pair_row, int32_t *row_token, int32_t *chunk_counts,
                           uint32_t *status, cudaStream_t s, int64_t M = 1, int32_t *group_load = nullptr,
                           float *score = nullptr);
cudaError_t launch_gather_rows(const void *x, const int32_t *row_token, const int32_t *offsets,
                               int64_t N, int64_t P, int64_t d, int dtype, void *x_perm, cudaStream_t s);
// x_perm[pair_row[t,k]] = x[t] (k < K) and x_perm[shared_base + s*T + t] = x[t] (s < S).
cudaError_t launch_scatter_rows(const void *x, const int32_t *pair_row, int64_t T, int64_t K, int64_t S,
                                int64_t shared_base, int64_t d, int dtype, void *x_perm, cudaStream_t s);
cudaError_t launch_imbalance(const int32_t *counts, int64_t T, int64_t N, int64_t M, int32_t *group_load,
                             float *score, cudaStream_t s);
// y[t] = sum_k gate[t,k] * y_perm[pair_row[t,k]] + sum_{s<S} y_perm[shared_base + s*T + t]
//        (+ residual[t] when residual is not null)
cudaError_t launch_combine(const void *y_perm, const int32_t *pair_row, const float *gate, int64_t T,
                           int64_t K, int64_t d, int dtype, void *y, cudaStream_t s, int64_t S = 0,
                           int64_t shared_base = 0, const void *residual = nullptr);
// Rows of S shared experts after the P routed rows: offsets[N+1+s] = P + (s+1)*T and
// row_token[P + s*T + t] = t (offsets[N] = P is the permutation's).
cudaError_t launch_shared_rows(int64_t T, int64_t N, int64_t S, int64_t P, int32_t *offsets, int32_t *row_token,
                               cudaStream_t s);
cudaError_t launch_ffn_simt(const void *x_perm, const int32_t *offsets, int64_t N, int64_t P, int64_t d,
                            int64_t I, int dtype, const void *w_gate, const void *w_up, const void *w_down,
                            void *h, void *y_perm, cudaStream_t s);

}  // namespace moge
