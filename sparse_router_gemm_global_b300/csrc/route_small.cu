// Small-batch router: the whole routing of a few tokens (and optionally their permutation) in
// one launch on CUDA cores.
//
// With a few tokens the router projection is a skinny matrix-vector product bound by reading
// W_r once, so tensor cores buy nothing and one 128-token MMA tile would leave all but a
// handful of SMs idle.  Here every CTA computes the scores of kTokTile tokens x kExpTile experts
// over the full hidden size (its threads split the hidden dimension, 16-byte loads, one round of
// loads in flight, fixed summation order), writes them to the workspace and takes a ticket; the
// last CTA to finish (no CTA ever waits) adds the bias and routes every token with the whole
// block (route_rows_block: global softmax, then group top-K' -- Pangu Pro MoE explainer, section
// 1: scores for all experts, one softmax over them, a local top-K' per group) and, when asked,
// permutes all tokens in the same block (histogram, prefix sum, deterministic scatter, group
// loads and imbalance score).
#include "common.cuh"
#include "permute_block.cuh"
#include "route_token.cuh"

namespace moge {
namespace rs {

constexpr int kThreads = kPermuteChunk;  // the permutation runs on one block of kPermuteChunk threads
constexpr int kTokTile = 4;              // tokens per CTA
constexpr int kExpTile = 8;              // experts per CTA

struct Params {
    const void *x;        // [T, d]
    const void *w;        // [N, d]
    const float *bias;    // [N] or null
    int T, d, N, groups, G, per;
    float *scores;        // [T, N] raw dot products (workspace)
    float *logits;        // [T, N] scores + bias, optional output
    int32_t *idx;         // [T, K]
    float *gate;          // [T, K]
    uint32_t *ticket;     // one self-resetting counter in the workspace status page
    uint32_t *status;
    // permutation (counts == nullptr: routing only)
    int M;
    int32_t *counts, *offsets, *pair_row, *row_token, *group_load;
    float *score;
};

__device__ __forceinline__ void unpack(const uint4 &v, float (&f)[8], __nv_bfloat16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}

__device__ __forceinline__ void unpack(const uint4 &v, float (&f)[4], float) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

template <typename E>
__global__ void __launch_bounds__(kThreads) route_small_kernel(const Params p) {
    extern __shared__ float sm[];
    __shared__ float part[kThreads / 32][kTokTile * kExpTile];
    __shared__ float tmax[kSmallRouteMaxT], tsum[kSmallRouteMaxT];
    __shared__ int is_last;
    constexpr int V = 16 / sizeof(E);  // elements per 16-byte vector
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kTokTile;
    const int e0 = blockIdx.y * kExpTile;
    pdl_wait();
    pdl_trigger();

    // ---- scores of this CTA's kTokTile x kExpTile tile.  Thread i of the block owns the 16-byte
    // vectors i, i + 256, ... of the hidden dimension for every token and expert of the tile,
    // so one round of loads brings in the whole tile; partial sums are reduced over the lanes
    // (butterfly) and then over the warps in warp order.
    {
        const int nvec = p.d / V;  // d is a multiple of V (16-byte rows)
        const uint4 *xrow[kTokTile], *wrow[kExpTile];
#pragma unroll
        for (int j = 0; j < kTokTile; ++j)  // rows past T repeat the last token; never stored
            xrow[j] = reinterpret_cast<const uint4 *>(static_cast<const E *>(p.x) + (size_t)min(t0 + j, p.T - 1) * p.d);
#pragma unroll
        for (int k = 0; k < kExpTile; ++k)  // rows past N repeat the last expert; never stored
            wrow[k] = reinterpret_cast<const uint4 *>(static_cast<const E *>(p.w) + (size_t)min(e0 + k, p.N - 1) * p.d);
        float acc[kTokTile][kExpTile];
#pragma unroll
        for (int j = 0; j < kTokTile; ++j)
#pragma unroll
            for (int k = 0; k < kExpTile; ++k) acc[j][k] = 0.f;
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            uint4 xv[kTokTile], wv[kExpTile];
#pragma unroll
            for (int j = 0; j < kTokTile; ++j) xv[j] = __ldg(xrow[j] + v);
#pragma unroll
            for (int k = 0; k < kExpTile; ++k) wv[k] = __ldg(wrow[k] + v);
#pragma unroll
            for (int k = 0; k < kExpTile; ++k) {
                float wf[V];
                unpack(wv[k], wf, E());
#pragma unroll
                for (int j = 0; j < kTokTile; ++j) {
                    float xf[V];
                    unpack(xv[j], xf, E());
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[j][k] = fmaf(xf[i], wf[i], acc[j][k]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kTokTile; ++j)
#pragma unroll
            for (int k = 0; k < kExpTile; ++k) {
                float a = acc[j][k];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                acc[j][k] = a;
            }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kTokTile; ++j)
#pragma unroll
                for (int k = 0; k < kExpTile; ++k) part[warp][j * kExpTile + k] = acc[j][k];
        }
        __syncthreads();
        if (threadIdx.x < kTokTile * kExpTile) {
            const int j = threadIdx.x / kExpTile, k = threadIdx.x - j * kExpTile;
            float a = part[0][threadIdx.x];
            for (int w = 1; w < kThreads / 32; ++w) a += part[w][threadIdx.x];
            if (t0 + j < p.T && e0 + k < p.N) p.scores[(size_t)(t0 + j) * p.N + e0 + k] = a;
        }
    }

    // ---- the last CTA to finish routes (and permutes) every token
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t total = gridDim.x * gridDim.y;
        const uint32_t ticket = atomicAdd(p.ticket, 1u);
        is_last = ticket == total - 1;
        if (is_last) *p.ticket = 0u;  // every CTA has taken its ticket: ready for the next call
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    const int K = p.groups * p.per;
    float *stage = sm;                                                      // [T][N] scores
    int32_t *sidx = reinterpret_cast<int32_t *>(sm + p.T * p.N);            // [T][K]
    uint32_t *psm = reinterpret_cast<uint32_t *>(sidx + p.T * K);           // permutation scratch
    for (int i = threadIdx.x; i < p.T * p.N; i += kThreads) {
        float v = __ldcg(p.scores + i);
        if (p.bias) v += p.bias[i % p.N];
        stage[i] = v;
        if (p.logits) p.logits[i] = v;
    }
    __syncthreads();
    route_rows_block(stage, p.N, 0, p.T, p.N, p.groups, p.G, p.per, sidx, p.gate, tmax, tsum);
    __syncthreads();
    for (int i = threadIdx.x; i < p.T * K; i += kThreads) p.idx[i] = sidx[i];
    if (p.counts)
        permute_one_block(sidx, p.T, K, p.N, p.counts, p.offsets, p.pair_row, p.row_token, p.status, p.M,
                          p.group_load, p.score, psm);
}

size_t smem_bytes(int64_t T, int64_t N, int64_t K, int64_t M, bool permute) {
    size_t words = (size_t)T * N + (size_t)T * K;
    if (permute) words += (size_t)permute_block_smem_words((int)N, (int)M);
    return words * 4;
}

}  // namespace rs

bool route_small_fits(int64_t T, int64_t N, int64_t K, int64_t M, bool permute) {
    return T >= 1 && T <= kSmallRouteMaxT && rs::smem_bytes(T, N, K, M, permute) <= kSmallRouteMaxSmem;
}

cudaError_t launch_route_small(const void *x, const void *w_r, const float *bias, int64_t T, int64_t d, int64_t N,
                               int64_t M, int64_t kpg, bool global, int dtype, float *scores, float *logits_out,
                               int32_t *idx, float *gate, uint32_t *ticket, uint32_t *status, int32_t *counts,
                               int32_t *offsets, int32_t *pair_row, int32_t *row_token, int32_t *group_load,
                               float *score, cudaStream_t s) {
    using namespace rs;
    Params p{};
    p.x = x;
    p.w = w_r;
    p.bias = bias;
    p.T = (int)T;
    p.d = (int)d;
    p.N = (int)N;
    p.groups = global ? 1 : (int)M;
    p.G = global ? (int)N : (int)(N / M);
    p.per = global ? (int)(M * kpg) : (int)kpg;
    p.scores = scores;
    p.logits = logits_out;
    p.idx = idx;
    p.gate = gate;
    p.ticket = ticket;
    p.status = status;
    p.M = (int)M;
    p.counts = counts;
    p.offsets = offsets;
    p.pair_row = pair_row;
    p.row_token = row_token;
    p.group_load = group_load;
    p.score = score;
    const int64_t K = M * kpg;
    if (!route_small_fits(T, N, K, M, counts != nullptr)) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(T, N, K, M, counts != nullptr);
    const dim3 grid((unsigned)cdiv(T, kTokTile), (unsigned)cdiv(N, kExpTile));
    cudaError_t err;
    if (dtype == MOGE_BF16) {
        err = set_max_smem(route_small_kernel<__nv_bfloat16>, (int)smem);
        if (err != cudaSuccess) return err;
        err = launch_pdl(route_small_kernel<__nv_bfloat16>, grid, dim3(kThreads), smem, s, p);
    } else {
        err = set_max_smem(route_small_kernel<float>, (int)smem);
        if (err != cudaSuccess) return err;
        err = launch_pdl(route_small_kernel<float>, grid, dim3(kThreads), smem, s, p);
    }
    count_launches(1);
    return err;
}

}  // namespace moge
