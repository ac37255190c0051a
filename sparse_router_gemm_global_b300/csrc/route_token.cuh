// Per-token routing from fp32 scores: global softmax over all N experts, then top-K' inside
// each group (Pangu Pro MoE explainer, section 1 "innovative architecture"), or top-K over all
// experts.  Shared by the scores-input kernel and the fused tensor-core router.
#pragma once

#include "common.cuh"

namespace moge {

// Route one token from its scores l[0..N) (any memory space).  groups/G/per describe the
// selection: grouped = (M, N/M, K'), global = (1, N, M*K').  Experts are compared on their
// fp32 scores, equal scores going to the lower index; the gate of a selected expert is
// exp(l - max) / sum_e exp(l_e - max) with a compensated fp32 sum (not renormalised).
__device__ __forceinline__ void route_token(const float *l, int N, int groups, int G, int per,
                                            int32_t *idx_out, float *gate_out) {
    float m = l[0];
    for (int e = 1; e < N; ++e) m = fmaxf(m, l[e]);
    // Neumaier-compensated sum of exp(l - m)
    float s = 0.f, comp = 0.f;
    for (int e = 0; e < N; ++e) {
        const float v = expf(l[e] - m);
        const float t = s + v;
        comp += (fabsf(s) >= fabsf(v)) ? ((s - t) + v) : ((v - t) + s);
        s = t;
    }
    s += comp;
    for (int g = 0; g < groups; ++g) {
        // walk the group's experts in rank order: each round takes the best
        // expert ranking strictly after the previously taken one
        float last_v = __int_as_float(0x7f800000);  // +inf
        int last_e = -1;
        for (int r = 0; r < per; ++r) {
            float bv = 0.f;
            int be = -1;
            for (int e = g * G; e < (g + 1) * G; ++e) {
                const float v = l[e];
                const bool after = (v < last_v) || (v == last_v && e > last_e);
                if (after && (be < 0 || v > bv)) { bv = v; be = e; }
            }
            idx_out[g * per + r] = be;
            gate_out[g * per + r] = expf(bv - m) / s;
            last_v = bv;
            last_e = be;
        }
    }
}

}  // namespace moge
