// Monte-Carlo study of the imbalance score (Pangu Pro MoE explainer, section 1: the imbalance
// score is the load of the busiest device minus that of the idlest over a batch; a Monte-Carlo
// simulation finds it almost always above zero for conventional top-K routing, while grouping
// the experts by device and taking K' per group makes it zero by construction).
//
// Each batch b of T tokens gets synthetic scores s[b,t,e] = z(i) + bias[e], i = (b*T + t)*N + e,
// where z is drawn on the device from a counter-based generator: three splitmix64 words
// (Steele, Lea and Flood, OOPSLA 2014) per element, whose twelve 16-bit fields u give the
// Irwin-Hall approximation of a standard normal, z = sum (u + 1/2)/2^16 - 6.  Every step of z
// is exact in fp32, so any implementation of that definition yields the same bits.  Each
// token is routed both ways (group top-K' and global top-K, K = M*K', ties to the lower
// index); the groups of the selected experts are counted per batch, and
//   imbalance[b] = (max_g load[b,g] - min_g load[b,g]) / T.
// Loads are integer sums (order-free atomics), so every output is exact and reproducible.
#include <algorithm>

#include "common.cuh"

namespace moge {
namespace st {

constexpr int kThreads = 128;              // tokens per block
constexpr uint64_t kStudyTensorId = 8;     // stream id of the study's scores

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float study_normal(uint64_t key, uint64_t i) {
    uint32_t S = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const uint64_t w = mix64(key + 3 * i + (uint64_t)j);
        S += (uint32_t)(w & 0xFFFFu) + (uint32_t)((w >> 16) & 0xFFFFu) + (uint32_t)((w >> 32) & 0xFFFFu) +
             (uint32_t)(w >> 48);
    }
    return (float)(2u * S + 12u) * (1.0f / 131072.0f) - 6.0f;
}

// Experts [lo, hi) of the token's scores l: add the groups of its top `per` (ranked by score,
// ties to the lower index) to the block's load counters `cnt` (group of e = e / G).
__device__ __forceinline__ void count_top(const float *l, int lo, int hi, int per, int G, int *cnt) {
    float last_v = __int_as_float(0x7f800000);  // +inf
    int last_e = -1;
    for (int r = 0; r < per; ++r) {
        float bv = 0.f;
        int be = -1;
        for (int e = lo; e < hi; ++e) {
            const float v = l[e];
            const bool after = (v < last_v) || (v == last_v && e > last_e);
            if (after && (be < 0 || v > bv)) {
                bv = v;
                be = e;
            }
        }
        atomicAdd(&cnt[be / G], 1);
        last_v = bv;
        last_e = be;
    }
}

__global__ void study_zero_kernel(int32_t *a, int32_t *b, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        a[i] = 0;
        b[i] = 0;
    }
}

__global__ void __launch_bounds__(kThreads)
study_route_kernel(uint64_t key, int64_t b0, int T, int N, int M, int kpg, const float *__restrict__ bias,
                   int32_t *__restrict__ loads_grouped, int32_t *__restrict__ loads_global) {
    extern __shared__ float sm[];  // [kThreads][N+1] scores, then 2*M block counters
    const int stride = N + 1;
    int *cnt = reinterpret_cast<int *>(sm + kThreads * stride);
    const int64_t b = b0 + blockIdx.y;
    const int t = blockIdx.x * kThreads + threadIdx.x;
    const int G = N / M;
    for (int i = threadIdx.x; i < 2 * M; i += kThreads) cnt[i] = 0;
    __syncthreads();
    if (t < T) {
        float *l = sm + threadIdx.x * stride;
        const uint64_t base = ((uint64_t)b * (uint64_t)T + (uint64_t)t) * (uint64_t)N;
        for (int e = 0; e < N; ++e) l[e] = study_normal(key, base + e) + (bias ? bias[e] : 0.f);
        for (int g = 0; g < M; ++g) count_top(l, g * G, (g + 1) * G, kpg, G, cnt);  // MoGE
        count_top(l, 0, N, M * kpg, G, cnt + M);                                     // global top-K
    }
    __syncthreads();
    for (int g = threadIdx.x; g < M; g += kThreads) {
        if (cnt[g]) atomicAdd(&loads_grouped[b * M + g], cnt[g]);
        if (cnt[M + g]) atomicAdd(&loads_global[b * M + g], cnt[M + g]);
    }
}

__global__ void study_score_kernel(const int32_t *__restrict__ loads_grouped, const int32_t *__restrict__ loads_global,
                                   int64_t batches, int M, int T, float *__restrict__ is_grouped,
                                   float *__restrict__ is_global) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batches) return;
    for (int mode = 0; mode < 2; ++mode) {
        const int32_t *ld = (mode == 0 ? loads_grouped : loads_global) + b * M;
        float *out = mode == 0 ? is_grouped : is_global;
        if (!out) continue;
        int mx = ld[0], mn = ld[0];
        for (int g = 1; g < M; ++g) {
            mx = max(mx, ld[g]);
            mn = min(mn, ld[g]);
        }
        out[b] = (float)(mx - mn) / (float)T;
    }
}

}  // namespace st

size_t imbalance_study_smem_bytes(int64_t N, int64_t M) {
    return (size_t)st::kThreads * (N + 1) * 4 + (size_t)2 * M * 4;
}

cudaError_t launch_imbalance_study(int64_t T, int64_t N, int64_t M, int64_t kpg, int64_t batches, uint64_t seed,
                                   const float *bias, int32_t *loads_grouped, int32_t *loads_global,
                                   float *is_grouped, float *is_global, cudaStream_t s) {
    using namespace st;
    if (batches == 0) return cudaSuccess;
    const int64_t n = batches * M;
    st::study_zero_kernel<<<(unsigned)std::min<int64_t>(cdiv(n, 256), 4096), 256, 0, s>>>(loads_grouped,
                                                                                          loads_global, n);
    count_launches(1);
    if (T > 0) {
        const size_t smem = imbalance_study_smem_bytes(N, M);
        cudaError_t err = set_max_smem(study_route_kernel, (int)smem);
        if (err != cudaSuccess) return err;
        const uint64_t key = mix64(seed ^ kStudyTensorId);
        constexpr int64_t kMaxGridY = 65535;
        for (int64_t b0 = 0; b0 < batches; b0 += kMaxGridY) {
            const dim3 grid((unsigned)cdiv(T, kThreads), (unsigned)std::min<int64_t>(kMaxGridY, batches - b0));
            study_route_kernel<<<grid, kThreads, smem, s>>>(key, b0, (int)T, (int)N, (int)M, (int)kpg, bias,
                                                            loads_grouped, loads_global);
            count_launches(1);
        }
    }
    if (is_grouped || is_global) {
        study_score_kernel<<<(unsigned)cdiv(batches, 256), 256, 0, s>>>(loads_grouped, loads_global, batches,
                                                                        (int)M, (int)(T > 0 ? T : 1), is_grouped,
                                                                        is_global);
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace moge
