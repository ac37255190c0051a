// Grouped expert FFN on tcgen05 tensor cores (bf16 in, fp32 accumulation in TMEM).
#pragma once

#include "common.cuh"

namespace moge {

// Token rows: act = x [T,d] gathered through row_token [P] (the permutation's row -> token map),
// or, with row_token == nullptr, act = x_perm [P,d] already in permuted order.
// offsets [N+1] (device), w_gate/w_up [N,I,d], w_down [N,d,I], h [P,I] scratch, y_perm [P,d].
// T bounds every expert's row count (a token picks an expert at most once).
cudaError_t launch_ffn_tc(const void *act, const int32_t *row_token, const int32_t *offsets, int64_t N, int64_t P,
                          int64_t T, int64_t d, int64_t I, const void *w_gate, const void *w_up, const void *w_down,
                          void *h, void *y_perm, uint32_t *status, cudaStream_t s);

}  // namespace moge
