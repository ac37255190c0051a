// C ABI of the MoGE layer forward: argument validation, workspace carving and launches.
// Every check runs on the host before anything is enqueued; see include/moge.h.
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <map>
#include <mutex>

#include "common.cuh"
#include "ffn_tc.cuh"
#include "validate.cuh"

using namespace moge;

namespace {
std::atomic<uint64_t> g_launches{0};
thread_local void *const *t_stage_events = nullptr;
}  // namespace

namespace moge {
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t set_max_smem_impl(const void *kernel, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> done;  // (kernel, device) -> bytes set
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(kernel, dev);
    const auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess) done[key] = bytes;
    return err;
}
void mark_stage(int stage, cudaStream_t s) {
    if (t_stage_events && stage >= 0 && stage <= MOGE_NUM_STAGES && t_stage_events[stage])
        cudaEventRecord((cudaEvent_t)t_stage_events[stage], s);
}
}  // namespace moge

namespace {

constexpr int64_t kMaxExperts = kAbiMaxExperts;

moge_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOGE_OK;
    static bool verbose = getenv("MOGE_VERBOSE") != nullptr;
    if (verbose) fprintf(stderr, "moge: CUDA error %s\n", cudaGetErrorString(e));
    return MOGE_ERR_CUDA;
}

moge_status_t check_ws(const moge_config_t *c, void *ws, size_t ws_bytes, int64_t S = 0) {
    if (!ws || ((uintptr_t)ws & 255u) != 0) return MOGE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*c, S).total) return MOGE_ERR_WORKSPACE;
    return MOGE_OK;
}

constexpr int64_t kMaxShared = 64;

template <typename T> T *at(void *ws, size_t off) { return (T *)((char *)ws + off); }

moge_status_t route_impl(const moge_config_t *c, moge_route_mode_t mode, const void *x, const void *w_router,
                         const float *bias, float *logits, int32_t *idx, float *gate, void *ws,
                         cudaStream_t st) {
    const WsLayout L = ws_layout(*c);
    const float *scores = logits;
    const bool global = mode == MOGE_ROUTE_GLOBAL_TOPK;
    const int64_t K = c->M * c->k_per_group;
    if (x && route_small_fits(c->T, c->N, K, c->M, false))  // few tokens: CUDA cores, one launch
        return cuda_status(launch_route_small(x, w_router, bias, c->T, c->d, c->N, c->M, c->k_per_group, global,
                                              c->act_dtype, at<float>(ws, L.logits), logits, idx, gate,
                                              at<uint32_t>(ws, kTicketOffset), at<uint32_t>(ws, L.status),
                                              nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, st));
    if (x && c->act_dtype == MOGE_BF16 && c->N <= 256)  // scores, softmax and selection in one launch
        return cuda_status(launch_router_tc(x, w_router, bias, c->T, c->d, c->N, c->M, c->k_per_group, global,
                                            logits, idx, gate, at<uint32_t>(ws, L.status), st));
    if (x) {
        float *dst = logits ? logits : at<float>(ws, L.logits);
        cudaError_t e = launch_router_logits_simt(x, w_router, bias, c->T, c->d, c->N, c->act_dtype, dst, st);
        if (e != cudaSuccess) return cuda_status(e);
        scores = dst;
    }
    return cuda_status(launch_route_select(scores, c->T, c->N, c->M, c->k_per_group,
                                           mode == MOGE_ROUTE_GLOBAL_TOPK, idx, gate, st));
}

// act = x_perm (row_token == nullptr) or x gathered through row_token (bf16 only).  With S shared
// experts the expert index space is N + S and the rows P + S*T.
moge_status_t ffn_impl(const moge_config_t *c, const void *act, const int32_t *row_token, const int32_t *offsets,
                       const void *wg, const void *wu, const void *wd, void *y_perm, void *ws, cudaStream_t st,
                       int64_t S = 0) {
    const WsLayout L = ws_layout(*c, S);
    const int64_t rows = c->T * c->M * c->k_per_group + S * c->T;
    const int64_t experts = c->N + S;
    void *h = at<void>(ws, L.h);
    uint32_t *status = at<uint32_t>(ws, L.status);
    if (c->act_dtype == MOGE_BF16)
        return cuda_status(launch_ffn_tc(act, row_token, offsets, experts, rows, c->T, c->d, c->I, wg, wu, wd, h,
                                         y_perm, status, st));
    const void *x_perm = act;
    return cuda_status(launch_ffn_simt(x_perm, offsets, experts, rows, c->d, c->I, c->act_dtype, wg, wu, wd, h,
                                       y_perm, st));
}

// The whole layer with S >= 0 shared experts (weights of N + S experts; S = 0 is the MoGE layer)
// and an optional residual stream added to the output (residual == nullptr: none).
moge_status_t layer_impl(const moge_config_t *cfg, int64_t S, const void *x, const void *residual,
                         const void *w_router, const float *bias, const void *w_gate, const void *w_up,
                         const void *w_down, void *y, const moge_aux_t *aux, void *ws, size_t ws_bytes,
                         moge_stream_t stream) {
    moge_status_t s = check_layer(cfg);
    if (s != MOGE_OK) return s;
    if (S < 0 || S > kMaxShared) return MOGE_ERR_INVALID_ARGUMENT;
    if (cfg->N + S > kMaxExperts) return MOGE_ERR_UNSUPPORTED;
    if (!w_router || !w_gate || !w_up || !w_down) return MOGE_ERR_INVALID_ARGUMENT;
    if (cfg->T > 0 && (!x || !y)) return MOGE_ERR_INVALID_ARGUMENT;  // an empty batch may pass NULL
    moge_aux_t a = aux ? *aux : moge_aux_t{};
    for (const void *p : {x, residual, w_router, (const void *)bias, w_gate, w_up, w_down, (const void *)y,
                          (const void *)a.logits, (const void *)a.topk_idx, (const void *)a.topk_gate,
                          (const void *)a.counts, (const void *)a.offsets, (const void *)a.group_load,
                          (const void *)a.score})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    if ((s = check_ws(cfg, ws, ws_bytes, S)) != MOGE_OK) return s;
    const WsLayout L = ws_layout(*cfg, S);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t K = cfg->M * cfg->k_per_group;
    const int64_t P = cfg->T * K;
    if (cfg->T == 0) {  // empty batch: only the counts/offsets/score outputs exist
        if (a.counts || a.offsets || a.score || a.group_load) {
            int32_t *counts = a.counts ? a.counts : at<int32_t>(ws, L.counts);
            int32_t *offsets = a.offsets ? a.offsets : at<int32_t>(ws, L.offsets);
            return cuda_status(launch_permute(nullptr, 0, K, cfg->N, counts, offsets, nullptr, nullptr, nullptr,
                                              nullptr, st, cfg->M, a.group_load, a.score));
        }
        return MOGE_OK;
    }
    int32_t *idx = a.topk_idx ? a.topk_idx : at<int32_t>(ws, L.idx);
    float *gate = a.topk_gate ? a.topk_gate : at<float>(ws, L.gate);
    int32_t *counts = a.counts ? a.counts : at<int32_t>(ws, L.counts);
    // the expert offsets live in the workspace whenever shared experts extend them past N + 1
    int32_t *offsets = (a.offsets && S == 0) ? a.offsets : at<int32_t>(ws, L.offsets);
    int32_t *pair_row = at<int32_t>(ws, L.pair_row);
    int32_t *row_token = at<int32_t>(ws, L.row_token);
    void *x_perm = at<void>(ws, L.x_perm);
    void *y_perm = at<void>(ws, L.y_perm);

    mark_stage(MOGE_STAGE_ROUTE, st);
    cudaError_t e = cudaSuccess;
    if (route_small_fits(cfg->T, cfg->N, K, cfg->M, true)) {
        // few tokens: routing and permutation in one launch; the permutation stage is empty
        e = launch_route_small(x, w_router, bias, cfg->T, cfg->d, cfg->N, cfg->M, cfg->k_per_group, false,
                               cfg->act_dtype, at<float>(ws, L.logits), a.logits, idx, gate,
                               at<uint32_t>(ws, kTicketOffset), at<uint32_t>(ws, L.status), counts, offsets,
                               pair_row, row_token, a.group_load, a.score, st);
        if (e != cudaSuccess) return cuda_status(e);
        mark_stage(MOGE_STAGE_PERMUTE, st);
    } else {
        if ((s = route_impl(cfg, MOGE_ROUTE_GROUPED, x, w_router, bias, a.logits, idx, gate, ws, st)) != MOGE_OK)
            return s;
        mark_stage(MOGE_STAGE_PERMUTE, st);  // the permutation also writes the imbalance outputs
        e = launch_permute(idx, cfg->T, K, cfg->N, counts, offsets, pair_row, row_token,
                           at<int32_t>(ws, L.chunk_counts), at<uint32_t>(ws, L.status), st, cfg->M, a.group_load,
                           a.score);
    }
    if (e == cudaSuccess) e = launch_shared_rows(cfg->T, cfg->N, S, P, offsets, row_token, st);
    if (e == cudaSuccess && a.offsets && S > 0)
        e = cudaMemcpyAsync(a.offsets, offsets, (size_t)(cfg->N + 1) * 4, cudaMemcpyDeviceToDevice, st);
    // bf16 with at most 32 tokens: the gate/up GEMM gathers the token rows itself (TMA gather4
    // through row_token) and the gather stage is empty; otherwise rows are first copied to x_perm
    // and loaded as tiles.
    const bool gather_in_gemm = gathers_in_gemm(*cfg, S);
    mark_stage(MOGE_STAGE_GATHER, st);
    if (e == cudaSuccess && !gather_in_gemm)
        e = launch_scatter_rows(x, pair_row, cfg->T, K, S, P, cfg->d, cfg->act_dtype, x_perm, st);
    if (e != cudaSuccess) return cuda_status(e);
    mark_stage(MOGE_STAGE_GATE_UP, st);  // the FFN marks MOGE_STAGE_DOWN between its two GEMMs
    s = gather_in_gemm ? ffn_impl(cfg, x, row_token, offsets, w_gate, w_up, w_down, y_perm, ws, st, S)
                       : ffn_impl(cfg, x_perm, nullptr, offsets, w_gate, w_up, w_down, y_perm, ws, st, S);
    if (s != MOGE_OK) return s;
    mark_stage(MOGE_STAGE_COMBINE, st);
    e = launch_combine(y_perm, pair_row, gate, cfg->T, K, cfg->d, cfg->act_dtype, y, st, S, P, residual);
    mark_stage(MOGE_STAGE_IMBALANCE, st);  // empty: computed with the permutation
    mark_stage(MOGE_NUM_STAGES, st);
    return cuda_status(e);
}

}  // namespace

extern "C" {

int moge_abi_version(void) { return MOGE_ABI_VERSION; }

const char *moge_status_string(moge_status_t s) {
    switch (s) {
        case MOGE_OK: return "ok";
        case MOGE_ERR_INVALID_ARGUMENT: return "invalid argument";
        case MOGE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOGE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOGE_ERR_CUDA: return "CUDA error";
        case MOGE_ERR_TIMEOUT: return "bounded device wait timed out";
    }
    return "unknown status";
}

size_t moge_workspace_bytes(const moge_config_t *cfg) {
    if (check_routing(cfg) != MOGE_OK) return 0;
    moge_config_t c = *cfg;
    if (c.d < 0 || c.I < 0) return 0;
    if (c.act_dtype != MOGE_BF16) c.act_dtype = MOGE_F32;
    return ws_layout(c).total;
}

moge_status_t moge_reset_device_status(void *ws, moge_stream_t stream) {
    if (!ws) return MOGE_ERR_INVALID_ARGUMENT;
    return cuda_status(cudaMemsetAsync(ws, 0, kStatusPageBytes, (cudaStream_t)stream));
}

moge_status_t moge_query_device_status(const void *ws, moge_stream_t stream) {
    if (!ws) return MOGE_ERR_INVALID_ARGUMENT;
    uint32_t word = 0;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemcpy(&word, ws, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    return (word & kStatusTimeout) ? MOGE_ERR_TIMEOUT : MOGE_OK;
}

moge_status_t moge_route(const moge_config_t *cfg, moge_route_mode_t mode, const void *x, const void *w_router,
                         const float *bias, float *logits, int32_t *topk_idx, float *topk_gate, void *ws,
                         size_t ws_bytes, moge_stream_t stream) {
    moge_status_t s = x ? check_layer(cfg) : check_routing(cfg);
    if (s != MOGE_OK) return s;
    if (mode != MOGE_ROUTE_GROUPED && mode != MOGE_ROUTE_GLOBAL_TOPK) return MOGE_ERR_INVALID_ARGUMENT;
    if (!topk_idx || !topk_gate) return MOGE_ERR_INVALID_ARGUMENT;
    if (!x && !logits) return MOGE_ERR_INVALID_ARGUMENT;
    if (x && !w_router) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)x, w_router, (const void *)bias, (const void *)logits,
                          (const void *)topk_idx, (const void *)topk_gate})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    if ((s = check_ws(cfg, ws, ws_bytes)) != MOGE_OK) return s;
    return route_impl(cfg, mode, x, w_router, bias, logits, topk_idx, topk_gate, ws, (cudaStream_t)stream);
}

moge_status_t moge_permute(const moge_config_t *cfg, const int32_t *topk_idx, const void *x, int32_t *counts,
                           int32_t *offsets, int32_t *pair_row, int32_t *row_token, void *x_perm, void *ws,
                           size_t ws_bytes, moge_stream_t stream) {
    const bool gather = x && x_perm;
    moge_status_t s = check_permute_args(cfg, topk_idx, x, counts, offsets, pair_row, row_token, x_perm);
    if (s != MOGE_OK) return s;
    if ((s = check_ws(cfg, ws, ws_bytes)) != MOGE_OK) return s;
    const WsLayout L = ws_layout(*cfg);
    const int64_t K = cfg->M * cfg->k_per_group;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_permute(topk_idx, cfg->T, K, cfg->N, counts, offsets, pair_row, row_token,
                                   at<int32_t>(ws, L.chunk_counts), at<uint32_t>(ws, L.status), st);
    if (e == cudaSuccess && gather)  // token-major copy when the slot -> row map is an output
        e = pair_row ? launch_scatter_rows(x, pair_row, cfg->T, K, 0, 0, cfg->d, cfg->act_dtype, x_perm, st)
                     : launch_gather_rows(x, row_token, offsets, cfg->N, cfg->T * K, cfg->d, cfg->act_dtype,
                                          x_perm, st);
    return cuda_status(e);
}

moge_status_t moge_expert_ffn(const moge_config_t *cfg, const void *x_perm, const int32_t *offsets,
                              const void *w_gate, const void *w_up, const void *w_down, void *y_perm, void *ws,
                              size_t ws_bytes, moge_stream_t stream) {
    moge_status_t s = check_layer(cfg);
    if (s != MOGE_OK) return s;
    if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !y_perm) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {x_perm, (const void *)offsets, w_gate, w_up, w_down, (const void *)y_perm})
        if (!aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    if ((s = check_ws(cfg, ws, ws_bytes)) != MOGE_OK) return s;
    return ffn_impl(cfg, x_perm, nullptr, offsets, w_gate, w_up, w_down, y_perm, ws, (cudaStream_t)stream);
}

moge_status_t moge_combine(const moge_config_t *cfg, const void *y_perm, const int32_t *pair_row,
                           const float *topk_gate, void *y, moge_stream_t stream) {
    moge_status_t s = check_layer(cfg);
    if (s != MOGE_OK) return s;
    if (!y_perm || !pair_row || !topk_gate || !y) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {y_perm, (const void *)pair_row, (const void *)topk_gate, (const void *)y})
        if (!aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    const int64_t K = cfg->M * cfg->k_per_group;
    return cuda_status(launch_combine(y_perm, pair_row, topk_gate, cfg->T, K, cfg->d, cfg->act_dtype, y,
                                      (cudaStream_t)stream));
}

moge_status_t moge_imbalance_score(const moge_config_t *cfg, const int32_t *counts, int32_t *group_load,
                                   float *score, moge_stream_t stream) {
    moge_status_t s = check_routing(cfg);
    if (s != MOGE_OK) return s;
    if (!counts || !score) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)counts, (const void *)group_load, (const void *)score})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    return cuda_status(launch_imbalance(counts, cfg->T, cfg->N, cfg->M, group_load, score, (cudaStream_t)stream));
}

moge_status_t moge_layer_forward(const moge_config_t *cfg, const void *x, const void *w_router, const float *bias,
                                 const void *w_gate, const void *w_up, const void *w_down, void *y,
                                 const moge_aux_t *aux, void *ws, size_t ws_bytes, moge_stream_t stream) {
    return layer_impl(cfg, 0, x, nullptr, w_router, bias, w_gate, w_up, w_down, y, aux, ws, ws_bytes, stream);
}

size_t moge_workspace_bytes_shared(const moge_config_t *cfg, int64_t n_shared) {
    if (n_shared < 0 || n_shared > kMaxShared || check_routing(cfg) != MOGE_OK) return 0;
    moge_config_t c = *cfg;
    if (c.d < 0 || c.I < 0) return 0;
    if (c.act_dtype != MOGE_BF16) c.act_dtype = MOGE_F32;
    return ws_layout(c, n_shared).total;
}

moge_status_t moge_layer_forward_shared(const moge_config_t *cfg, int64_t n_shared, const void *x,
                                        const void *w_router, const float *bias, const void *w_gate,
                                        const void *w_up, const void *w_down, void *y, const moge_aux_t *aux,
                                        void *ws, size_t ws_bytes, moge_stream_t stream) {
    return layer_impl(cfg, n_shared, x, nullptr, w_router, bias, w_gate, w_up, w_down, y, aux, ws, ws_bytes,
                      stream);
}

moge_status_t moge_layer_forward_residual(const moge_config_t *cfg, int64_t n_shared, const void *x,
                                          const void *residual, const void *w_router, const float *bias,
                                          const void *w_gate, const void *w_up, const void *w_down, void *y,
                                          const moge_aux_t *aux, void *ws, size_t ws_bytes, moge_stream_t stream) {
    if (!residual && cfg && cfg->T > 0) return MOGE_ERR_INVALID_ARGUMENT;
    return layer_impl(cfg, n_shared, x, residual, w_router, bias, w_gate, w_up, w_down, y, aux, ws, ws_bytes,
                      stream);
}

moge_status_t moge_imbalance_study(const moge_config_t *cfg, int64_t batches, uint64_t seed, const float *bias,
                                   int32_t *loads_grouped, int32_t *loads_global, float *is_grouped,
                                   float *is_global, moge_stream_t stream) {
    moge_status_t s = check_routing(cfg);
    if (s != MOGE_OK) return s;
    if (batches < 0 || !loads_grouped || !loads_global) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)bias, (const void *)loads_grouped, (const void *)loads_global,
                          (const void *)is_grouped, (const void *)is_global})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    if (cfg->N > kStudyMaxExperts || cfg->T > (1 << 30) || batches * cfg->M > ((int64_t)1 << 31) ||
        imbalance_study_smem_bytes(cfg->N, cfg->M) > 200 * 1024)
        return MOGE_ERR_UNSUPPORTED;
    return cuda_status(launch_imbalance_study(cfg->T, cfg->N, cfg->M, cfg->k_per_group, batches, seed, bias,
                                              loads_grouped, loads_global, is_grouped, is_global,
                                              (cudaStream_t)stream));
}

moge_status_t moge_set_stage_events(void *const *events, int n) {
    if (events && n != MOGE_NUM_STAGES + 1) return MOGE_ERR_INVALID_ARGUMENT;
    t_stage_events = events;
    return MOGE_OK;
}

uint64_t moge_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
