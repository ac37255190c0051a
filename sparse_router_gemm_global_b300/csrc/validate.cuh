// Host-side argument checks shared by every entry point (internal header).  Each returns the
// status the call reports, before anything is launched.
#pragma once

#include <stdint.h>

#include "moge.h"

namespace moge {

constexpr int64_t kAbiMaxExperts = 1024;
constexpr int64_t kAbiMaxSlots = 1024;

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Routing shape: T >= 0, 1 <= M, N % M == 0, 1 <= K' <= N/M, N <= 1024, T*K < 2^31.
inline moge_status_t check_routing(const moge_config_t *c) {
    if (!c) return MOGE_ERR_INVALID_ARGUMENT;
    if (c->T < 0 || c->N < 1 || c->M < 1 || c->N % c->M != 0) return MOGE_ERR_INVALID_ARGUMENT;
    if (c->k_per_group < 1 || c->k_per_group > c->N / c->M) return MOGE_ERR_INVALID_ARGUMENT;
    const int64_t K = c->M * c->k_per_group;
    if (c->N > kAbiMaxExperts || K > kAbiMaxSlots) return MOGE_ERR_UNSUPPORTED;
    if (c->T > ((int64_t)1 << 31) / K - 1) return MOGE_ERR_UNSUPPORTED;
    return MOGE_OK;
}

// Full layer shape: routing shape + d, I >= 1, one supported dtype, 16-byte rows.
inline moge_status_t check_layer(const moge_config_t *c) {
    moge_status_t s = check_routing(c);
    if (s != MOGE_OK) return s;
    if (c->d < 1 || c->I < 1) return MOGE_ERR_INVALID_ARGUMENT;
    if (c->act_dtype != c->weight_dtype) return MOGE_ERR_UNSUPPORTED;
    if (c->act_dtype != MOGE_F32 && c->act_dtype != MOGE_BF16) return MOGE_ERR_UNSUPPORTED;
    const int64_t vec = (c->act_dtype == MOGE_BF16) ? 8 : 4;  // elements per 16 bytes
    if (c->d % vec != 0 || c->I % vec != 0) return MOGE_ERR_UNSUPPORTED;
    if (c->d > (1 << 20) || c->I > (1 << 20)) return MOGE_ERR_UNSUPPORTED;
    return MOGE_OK;
}

// The permutation's own arguments (moge_permute and moge_permute_noalloc): the layer shape when
// rows are copied (x and x_perm given), else the routing shape; the index outputs; alignment.
inline moge_status_t check_permute_args(const moge_config_t *c, const int32_t *topk_idx, const void *x,
                                        const int32_t *counts, const int32_t *offsets, const int32_t *pair_row,
                                        const int32_t *row_token, const void *x_perm) {
    const bool gather = x && x_perm;
    moge_status_t s = gather ? check_layer(c) : check_routing(c);
    if (s != MOGE_OK) return s;
    if (!topk_idx || !counts || !offsets) return MOGE_ERR_INVALID_ARGUMENT;
    if (gather && !row_token) return MOGE_ERR_INVALID_ARGUMENT;
    for (const void *p : {(const void *)topk_idx, x, (const void *)counts, (const void *)offsets,
                          (const void *)pair_row, (const void *)row_token, x_perm})
        if (p && !aligned16(p)) return MOGE_ERR_INVALID_ARGUMENT;
    return MOGE_OK;
}

}  // namespace moge
