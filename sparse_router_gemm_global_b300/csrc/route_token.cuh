// Routing from fp32 scores: global softmax over all N experts, then top-K' inside each group
// (Pangu Pro MoE explainer, section 1 "innovative architecture"), or top-K over all experts.
// Shared by the scores-input kernel, the tensor-core router and the small-batch router.
#pragma once

#include "common.cuh"

namespace moge {

// Route rows [r0, r1) of a score tile with a whole block (scores[row * stride + e], any memory
// space; bias already added).  groups/G/per describe the selection: grouped = (M, N/M, K'), global
// = (1, N, M*K').  Experts are compared on their fp32 scores, equal scores going to the lower
// index; the gate of a selected expert is exp(l - max) / sum_e exp(l_e - max) (not
// renormalised).  Two parallel passes:
// (1) one warp per row: max and sum of exp(l - max) (compensated per lane) by butterfly
// reductions; (2) one thread per
// (row, group): every member's rank, rank(e) = #{e' in group : l[e'] > l[e] or (l[e'] == l[e] and
// e' < e)}, and e is taken iff rank(e) < per, into slot group * per + rank -- the definition of
// the group top-K' itself, with no ordering step.  Groups of up to kRegGroup members are ranked in
// registers.  row_max / row_sum: shared scratch of (r1 - r0) floats each.  Outputs of row r go to
// idx_out[r * K .. ] and gate_out[r * K ..] with K = groups * per.
constexpr int kRegGroup = 16;

__device__ __forceinline__ void route_rows_block(const float *scores, int stride, int r0, int r1, int N, int groups,
                                                 int G, int per, int32_t *idx_out, float *gate_out, float *row_max,
                                                 float *row_sum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int rows = r1 - r0;
    for (int i = warp; i < rows; i += nwarps) {
        const float *l = scores + (size_t)(r0 + i) * stride;
        float m = -__int_as_float(0x7f800000);
        for (int e = lane; e < N; e += 32) m = fmaxf(m, l[e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.f, comp = 0.f;  // per-lane Neumaier-compensated sum, then a butterfly
        for (int e = lane; e < N; e += 32) {
            const float v = expf(l[e] - m);
            const float t = s + v;
            comp += (fabsf(s) >= fabsf(v)) ? ((s - t) + v) : ((v - t) + s);
            s = t;
        }
        s += comp;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
            row_max[i] = m;
            row_sum[i] = s;
        }
    }
    __syncthreads();
    const int K = groups * per;
    for (int task = threadIdx.x; task < rows * groups; task += blockDim.x) {
        const int i = task / groups, g = task - i * groups;
        const int r = r0 + i;
        const float *l = scores + (size_t)r * stride + g * G;
        const float m = row_max[i], s = row_sum[i];
        if (G <= kRegGroup) {
            float v[kRegGroup];
#pragma unroll
            for (int j = 0; j < kRegGroup; ++j) v[j] = j < G ? l[j] : 0.f;
#pragma unroll
            for (int j = 0; j < kRegGroup; ++j) {
                if (j >= G) break;
                int rank = 0;
#pragma unroll
                for (int q = 0; q < kRegGroup; ++q)
                    if (q < G) rank += (v[q] > v[j]) || (v[q] == v[j] && q < j);
                if (rank < per) {
                    idx_out[(size_t)r * K + g * per + rank] = g * G + j;
                    gate_out[(size_t)r * K + g * per + rank] = expf(v[j] - m) / s;
                }
            }
        } else {
            for (int j = 0; j < G; ++j) {
                const float vj = l[j];
                int rank = 0;
                for (int q = 0; q < G && rank < per; ++q) {
                    const float vq = l[q];
                    rank += (vq > vj) || (vq == vj && q < j);
                }
                if (rank < per) {
                    idx_out[(size_t)r * K + g * per + rank] = g * G + j;
                    gate_out[(size_t)r * K + g * per + rank] = expf(vj - m) / s;
                }
            }
        }
    }
}

}  // namespace moge
