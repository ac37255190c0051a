// Block-level building blocks of the permutation (histogram -> prefix sum -> deterministic
// scatter), shared by the permutation kernels and by the small-batch router, which permutes
// its tokens in the same launch.  Every function here is called by all kPermuteChunk threads
// of a block, which share the (token, slot) pairs of a chunk of kPermuteChunk tokens.
//
// Row of pair (t,k) with expert e:  offsets[e] + #{t' < t routed to e}.
// Inside a chunk, token r sets its bit in the mask of (32-token group r/32, expert) (shared
// atomicOr: order-free, so deterministic); the rank of a token among earlier tokens of its
// group is popc(mask below its bit), the rank of a group's first token is the sum of popc over
// earlier groups, and the chunk's base is the sum over earlier chunks.  A token selects each
// expert at most once, so "earlier pair with the same expert" equals "earlier token".
#pragma once

#include "common.cuh"

namespace moge {

constexpr int kChunk = kPermuteChunk;
constexpr int kWarps = kChunk / 32;

// Fill masks[w*N + e] for the chunk of tokens [t0, t0 + kChunk): bit j of masks[w*N + e] is set
// iff token t0 + 32w + j selected expert e.  The block's threads share the chunk's (token, slot)
// pairs.  Caller syncs afterwards.
__device__ __forceinline__ void build_masks(const int32_t *__restrict__ idx, int64_t t0, int64_t T, int K, int N,
                                            uint32_t *masks, uint32_t *status) {
    for (int i = threadIdx.x; i < kWarps * N; i += blockDim.x) masks[i] = 0u;
    __syncthreads();
    const int nt = (int)min((int64_t)kChunk, T - t0);
    for (int i = threadIdx.x; i < nt * K; i += blockDim.x) {
        const int r = i / K;  // token inside the chunk
        const int e = idx[(t0 + r) * K + (i - r * K)];
        if (e >= 0 && e < N) atomicOr(&masks[(r >> 5) * N + e], 1u << (r & 31));
        else raise_status(status, kStatusBadIndex);
    }
}

// Exclusive prefix sum of cnt[0..N) by warp 0 (N <= 1024): lane j owns the consecutive
// experts [j*c, (j+1)*c), c = ceil(N/32), adds them in order, the lane totals are scanned with
// shuffles.  Writes excl[e] (may alias cnt) and returns the total to lane 0 of warp 0.
__device__ __forceinline__ int warp_exclusive_scan(const int32_t *cnt, int N, int32_t *excl) {
    const int lane = threadIdx.x & 31;
    const int c = (N + 31) >> 5;
    const int e0 = min(lane * c, N), e1 = min(e0 + c, N);
    int local = 0;
    for (int e = e0; e < e1; ++e) local += cnt[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
        const int v = cnt[e];
        excl[e] = run;
        run += v;
    }
    return __shfl_sync(0xffffffffu, incl, 31);
}

// Optional imbalance score from per-expert counts in shared memory (the whole block calls it):
// group_load[g] = sum of the counts of group g's experts, score = (max - min) / T (fp32).
// `loads` is shared scratch of M ints.
__device__ __forceinline__ void block_imbalance(const int32_t *cnt, int N, int M, int64_t T, int32_t *loads,
                                                int32_t *__restrict__ group_load, float *__restrict__ score) {
    if (!group_load && !score) return;
    const int G = N / M;
    for (int g = threadIdx.x; g < M; g += blockDim.x) {
        int s = 0;
        for (int e = g * G; e < (g + 1) * G; ++e) s += cnt[e];
        loads[g] = s;
        if (group_load) group_load[g] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0 && score) {
        int mx = loads[0], mn = loads[0];
        for (int g = 1; g < M; ++g) {
            mx = max(mx, loads[g]);
            mn = min(mn, loads[g]);
        }
        *score = T > 0 ? (float)(mx - mn) / (float)T : 0.f;
    }
}

// Rows of the chunk's pairs (tokens [t0, t0 + kChunk)).  base[e] = offsets[e] + bases of
// earlier chunks.  The row of token t0 + r with expert e is base[e] + (tokens of earlier warps
// routed to e) + popc(mask of its warp below its own bit).
__device__ __forceinline__ void scatter_rows(const int32_t *__restrict__ idx, int64_t t0, int64_t T, int K, int N,
                                             const uint32_t *masks, int32_t *warp_base,
                                             const int32_t *base, int32_t *__restrict__ pair_row,
                                             int32_t *__restrict__ row_token) {
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int run = base[e];
        for (int w = 0; w < kWarps; ++w) {
            warp_base[w * N + e] = run;
            run += __popc(masks[w * N + e]);
        }
    }
    __syncthreads();
    const int nt = (int)min((int64_t)kChunk, T - t0);
    for (int i = threadIdx.x; i < nt * K; i += blockDim.x) {
        const int r = i / K;
        const int64_t pair = (t0 + r) * K + (i - r * K);
        const int e = idx[pair];
        int row = -1;
        if (e >= 0 && e < N)
            row = warp_base[(r >> 5) * N + e] + __popc(masks[(r >> 5) * N + e] & ((1u << (r & 31)) - 1u));
        if (pair_row) pair_row[pair] = row;
        if (row_token && row >= 0) row_token[row] = (int32_t)(t0 + r);
    }
}

// Shared-memory words needed by permute_one_block.
__host__ __device__ constexpr int permute_block_smem_words(int N, int M) { return 2 * kWarps * N + N + M; }

// All T <= kChunk tokens in one block: count, scan and scatter (+ imbalance).  `sm` holds
// permute_block_smem_words(N, M) words.  idx must be visible to the whole block.
__device__ __forceinline__ void permute_one_block(const int32_t *__restrict__ idx, int64_t T, int K, int N,
                                                  int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                                  int32_t *__restrict__ pair_row, int32_t *__restrict__ row_token,
                                                  uint32_t *status, int M, int32_t *__restrict__ group_load,
                                                  float *__restrict__ score, uint32_t *sm) {
    uint32_t *masks = sm;
    int32_t *warp_base = (int32_t *)(sm + kWarps * N);
    int32_t *base = warp_base + kWarps * N;
    int32_t *loads = base + N;
    build_masks(idx, 0, T, K, N, masks, status);
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < kWarps; ++w) c += __popc(masks[w * N + e]);
        base[e] = c;
    }
    __syncthreads();
    block_imbalance(base, N, M, T, loads, group_load, score);
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) counts[e] = base[e];
    __syncthreads();
    if (threadIdx.x < 32) {
        const int total = warp_exclusive_scan(base, N, base);
        __syncwarp();
        for (int e = threadIdx.x; e < N; e += 32) offsets[e] = base[e];
        if (threadIdx.x == 0) offsets[N] = total;
    }
    __syncthreads();
    scatter_rows(idx, 0, T, K, N, masks, warp_base, base, pair_row, row_token);
}

}  // namespace moge
