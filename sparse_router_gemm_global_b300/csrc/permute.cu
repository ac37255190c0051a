// Permutation of (token, slot) pairs into expert-contiguous rows:
// histogram -> prefix sum -> deterministic scatter, then the row copy into x_perm (token-major
// from pair_row, or row-major through row_token when the caller wants no pair_row).
// Tokens are cut into chunks of kPermuteChunk (one block each, one token per thread); the
// block-level steps are in permute_block.cuh.
#include <algorithm>

#include "common.cuh"
#include "permute_block.cuh"

namespace moge {

// Per-chunk expert counts: chunk_counts[chunk][e].
__global__ void permute_count_kernel(const int32_t *__restrict__ idx, int64_t T, int K, int N,
                                     int32_t *__restrict__ chunk_counts, uint32_t *status) {
    extern __shared__ uint32_t masks[];  // [kWarps][N]
    pdl_wait();
    pdl_trigger();
    build_masks(idx, (int64_t)blockIdx.x * kChunk, T, K, N, masks, status);
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < kWarps; ++w) c += __popc(masks[w * N + e]);
        chunk_counts[(int64_t)blockIdx.x * N + e] = c;
    }
}

// One block: chunk_counts -> per-chunk bases (in place), counts, offsets (+ imbalance).
__global__ void permute_scan_kernel(int32_t *__restrict__ chunk_counts, int chunks, int N,
                                    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int M,
                                    int64_t T, int32_t *__restrict__ group_load, float *__restrict__ score) {
    extern __shared__ int32_t tot[];  // [N] counts, then [M] group loads
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
        int run = 0;
        for (int c = 0; c < chunks; ++c) {
            const int v = chunk_counts[(int64_t)c * N + e];
            chunk_counts[(int64_t)c * N + e] = run;
            run += v;
        }
        tot[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // N <= 1024: a serial scan is cheap and obviously ordered
        int run = 0;
        for (int e = 0; e < N; ++e) {
            offsets[e] = run;
            run += tot[e];
        }
        offsets[N] = run;
    }
    block_imbalance(tot, N, M, T, tot + N, group_load, score);
}

__global__ void permute_scatter_kernel(const int32_t *__restrict__ idx, int64_t T, int K, int N,
                                       const int32_t *__restrict__ chunk_base,
                                       const int32_t *__restrict__ offsets, int32_t *__restrict__ pair_row,
                                       int32_t *__restrict__ row_token) {
    extern __shared__ uint32_t sm[];
    uint32_t *masks = sm;                              // [kWarps][N]
    int32_t *warp_base = (int32_t *)(sm + kWarps * N);  // [kWarps][N]
    int32_t *base = warp_base + kWarps * N;             // [N]
    pdl_wait();
    pdl_trigger();
    build_masks(idx, (int64_t)blockIdx.x * kChunk, T, K, N, masks, nullptr);
    for (int e = threadIdx.x; e < N; e += blockDim.x)
        base[e] = offsets[e] + chunk_base[(int64_t)blockIdx.x * N + e];
    __syncthreads();
    scatter_rows(idx, (int64_t)blockIdx.x * kChunk, T, K, N, masks, warp_base, base, pair_row, row_token);
}

// T <= kChunk: count, scan and scatter in one block (+ imbalance).
__global__ void permute_single_kernel(const int32_t *__restrict__ idx, int64_t T, int K, int N,
                                      int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                      int32_t *__restrict__ pair_row, int32_t *__restrict__ row_token,
                                      uint32_t *status, int M, int32_t *__restrict__ group_load,
                                      float *__restrict__ score) {
    extern __shared__ uint32_t sm[];
    pdl_wait();
    pdl_trigger();
    permute_one_block(idx, T, K, N, counts, offsets, pair_row, row_token, status, M, group_load, score, sm);
}

__global__ void zero_counts_kernel(int N, int32_t *counts, int32_t *offsets, int M, int32_t *group_load,
                                   float *score) {
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e <= N; e += blockDim.x) {
        if (e < N) counts[e] = 0;
        offsets[e] = 0;
    }
    if (group_load)
        for (int g = threadIdx.x; g < M; g += blockDim.x) group_load[g] = 0;
    if (score && threadIdx.x == 0) *score = 0.f;
}

cudaError_t launch_permute(const int32_t *idx, int64_t T, int64_t K, int64_t N, int32_t *counts,
                           int32_t *offsets, int32_t *pair_row, int32_t *row_token, int32_t *chunk_counts,
                           uint32_t *status, cudaStream_t s, int64_t M, int32_t *group_load, float *score) {
    if (T == 0) {
        cudaError_t err = launch_pdl(zero_counts_kernel, dim3(1), dim3(256), 0, s, (int)N, counts, offsets, (int)M,
                                     group_load, score);
        count_launches(1);
        return err;
    }
    const size_t smem_scatter = (size_t)permute_block_smem_words((int)N, (int)M) * 4;
    cudaError_t err;
    if (T <= kChunk) {
        err = set_max_smem(permute_single_kernel, (int)smem_scatter);
        if (err != cudaSuccess) return err;
        err = launch_pdl(permute_single_kernel, dim3(1), dim3(kChunk), smem_scatter, s, idx, T, (int)K, (int)N,
                         counts, offsets, pair_row, row_token, status, (int)M, group_load, score);
        count_launches(1);
        return err;
    }
    const int chunks = (int)cdiv(T, kChunk);
    const size_t smem_count = (size_t)kWarps * N * 4;
    err = set_max_smem(permute_count_kernel, (int)smem_count);
    if (err != cudaSuccess) return err;
    err = set_max_smem(permute_scatter_kernel, (int)smem_scatter);
    if (err != cudaSuccess) return err;
    err = launch_pdl(permute_count_kernel, dim3(chunks), dim3(kChunk), smem_count, s, idx, T, (int)K, (int)N,
                     chunk_counts, status);
    count_launches(1);
    if (err != cudaSuccess) return err;
    err = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), (size_t)(N + M) * 4, s, chunk_counts, chunks, (int)N,
                     counts, offsets, (int)M, T, group_load, score);
    count_launches(1);
    if (err != cudaSuccess) return err;
    err = launch_pdl(permute_scatter_kernel, dim3(chunks), dim3(kChunk), smem_scatter, s, idx, T, (int)K, (int)N,
                     (const int32_t *)chunk_counts, (const int32_t *)offsets, pair_row, row_token);
    count_launches(1);
    return err;
}

// ---------------------------------------------------------------------------------------------
// Row gather x_perm[r,:] = x[row_token[r],:] (moge_permute without pair_row); one warp per row,
// 16-byte vectors, each lane issuing 8 loads before their stores so that a row's reads are in
// flight together.  Only rows r < offsets[N] (the pairs that exist) are copied.  Every row of x
// is read once per expert its token selected, so x is loaded with an evict-last L2 policy and
// x_perm (written once, read back much later) is stored with the streaming hint; still, at the
// prefill shape it moved 1.51 GB against 1.14 GB algorithmic, where the token-major copy below
// moves 1.08 GB.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ int4 ld_keep(const int4 *p, uint64_t pol) {
    int4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__global__ void gather_rows_kernel(const int4 *__restrict__ x, const int32_t *__restrict__ row_token,
                                   const int32_t *__restrict__ offsets, int N, int64_t vec_per_row,
                                   int4 *__restrict__ x_perm) {
    constexpr int kBatch = 8;
    uint64_t keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    pdl_wait();
    pdl_trigger();
    const int64_t rows = offsets[N];
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const int64_t t = row_token[r];
        const int4 *src = x + t * vec_per_row;
        int4 *dst = x_perm + r * vec_per_row;
        for (int64_t v0 = lane; v0 < vec_per_row; v0 += 32 * kBatch) {
            int4 buf[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int64_t v = v0 + 32 * j;
                if (v < vec_per_row) buf[j] = ld_keep(src + v, keep);
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int64_t v = v0 + 32 * j;
                if (v < vec_per_row) __stcs(dst + v, buf[j]);
            }
        }
    }
}

cudaError_t launch_gather_rows(const void *x, const int32_t *row_token, const int32_t *offsets, int64_t N,
                               int64_t P, int64_t d, int dtype, void *x_perm, cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    const int64_t row_bytes = d * (dtype == MOGE_BF16 ? 2 : 4);
    const int64_t vec = row_bytes / 16;
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = cdiv(P, 8);  // 8 warps (rows in flight) per block
    const unsigned blocks = (unsigned)std::min<int64_t>(want, (int64_t)sms * 8);
    cudaError_t err = launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, (const int4 *)x, row_token,
                                 offsets, (int)N, vec, (int4 *)x_perm);
    count_launches(1);
    return err;
}

// ---------------------------------------------------------------------------------------------
// Token-major row copy: x_perm[pair_row[t,k],:] = x[t,:] for every slot k, and
// x_perm[shared_base + s*T + t,:] = x[t,:] for each of S shared experts.  The same rows as the
// gather above, but a warp loads one 32 x kBatch-vector chunk of a token's row once and stores it
// to all its destinations, so the copy reads x about once whatever L2 keeps.  Work item =
// (token, chunk, destination group): small batches split the K + S destinations of a token into
// `dgroups` groups so that enough warps are in flight; one warp per item.
// ---------------------------------------------------------------------------------------------
constexpr int kScatterBatch = 8;
constexpr int64_t kScatterChunkVec = 32 * kScatterBatch;
constexpr int kScatterThreads = 128;

__global__ void __launch_bounds__(kScatterThreads)
scatter_rows_kernel(const int4 *__restrict__ x, const int32_t *__restrict__ pair_row, int64_t T, int K, int S,
                    int64_t shared_base, int64_t vec_per_row, int dgroups, int4 *__restrict__ x_perm) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (vec_per_row + kScatterChunkVec - 1) / kScatterChunkVec;
    const int64_t items = T * chunks * dgroups;
    const int dests = K + S;
    const int per = (dests + dgroups - 1) / dgroups;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t item = warp; item < items; item += nwarps) {
        const int64_t tc = item / dgroups;
        const int g = (int)(item - tc * dgroups);
        const int64_t t = tc / chunks;
        const int64_t v0 = (tc - t * chunks) * kScatterChunkVec + lane;
        const int4 *src = x + t * vec_per_row;
        int4 buf[kScatterBatch];
#pragma unroll
        for (int j = 0; j < kScatterBatch; ++j) {
            const int64_t v = v0 + 32 * j;
            if (v < vec_per_row) buf[j] = __ldg(src + v);
        }
        const int32_t *pr = pair_row + t * K;
        const int k1 = min(dests, (g + 1) * per);
        for (int k = g * per; k < k1; ++k) {
            const int64_t r = k < K ? (int64_t)__ldg(pr + k) : shared_base + (int64_t)(k - K) * T + t;
            if (r < 0) continue;  // a slot whose expert id the permutation skipped owns no row
            int4 *dst = x_perm + r * vec_per_row;
#pragma unroll
            for (int j = 0; j < kScatterBatch; ++j) {
                const int64_t v = v0 + 32 * j;
                if (v < vec_per_row) __stcs(dst + v, buf[j]);
            }
        }
    }
}

cudaError_t launch_scatter_rows(const void *x, const int32_t *pair_row, int64_t T, int64_t K, int64_t S,
                                int64_t shared_base, int64_t d, int dtype, void *x_perm, cudaStream_t s) {
    const int64_t dests = K + S;
    if (T == 0 || dests == 0) return cudaSuccess;
    const int64_t vec = d * (dtype == MOGE_BF16 ? 2 : 4) / 16;
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t base_items = T * cdiv(vec, kScatterChunkVec);
    const int64_t want = (int64_t)sms * 16;  // warps to keep in flight
    const int dgroups = (int)std::min<int64_t>(dests, std::max<int64_t>(1, cdiv(want, base_items)));
    const int64_t warps_per_block = kScatterThreads / 32;
    const unsigned blocks =
        (unsigned)std::min<int64_t>(cdiv(base_items * dgroups, warps_per_block), (int64_t)1 << 30);
    cudaError_t err = launch_pdl(scatter_rows_kernel, dim3(blocks), dim3(kScatterThreads), 0, s, (const int4 *)x,
                                 pair_row, T, (int)K, (int)S, shared_base, vec, dgroups, (int4 *)x_perm);
    count_launches(1);
    return err;
}

// ---------------------------------------------------------------------------------------------
// Shared experts: every token visits each of the S shared experts, so their rows are fixed:
// expert N + s owns rows [P + s*T, P + (s+1)*T), row P + s*T + t holding token t.
// ---------------------------------------------------------------------------------------------
__global__ void shared_rows_kernel(int64_t T, int64_t N, int64_t S, int64_t P, int32_t *__restrict__ offsets,
                                   int32_t *__restrict__ row_token) {
    pdl_wait();
    pdl_trigger();
    const int64_t n = S * T;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        row_token[P + i] = (int32_t)(i % T);
    if (blockIdx.x == 0)
        for (int64_t s = threadIdx.x; s < S; s += blockDim.x) offsets[N + 1 + s] = (int32_t)(P + (s + 1) * T);
}

cudaError_t launch_shared_rows(int64_t T, int64_t N, int64_t S, int64_t P, int32_t *offsets, int32_t *row_token,
                               cudaStream_t s) {
    if (S == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(cdiv(S * T, 256), 1184));
    cudaError_t err = launch_pdl(shared_rows_kernel, dim3(blocks), dim3(256), 0, s, T, N, S, P, offsets, row_token);
    count_launches(1);
    return err;
}

// ---------------------------------------------------------------------------------------------
// Imbalance score: group loads, then (max - min) / T.  One block.
// ---------------------------------------------------------------------------------------------
__global__ void imbalance_kernel(const int32_t *__restrict__ counts, int64_t T, int N, int M,
                                 int32_t *__restrict__ group_load, float *__restrict__ score) {
    extern __shared__ int64_t loads[];  // [M]
    pdl_wait();
    pdl_trigger();
    const int G = N / M;
    for (int g = threadIdx.x; g < M; g += blockDim.x) {
        int64_t sum = 0;
        for (int e = g * G; e < (g + 1) * G; ++e) sum += counts[e];
        loads[g] = sum;
        if (group_load) group_load[g] = (int32_t)sum;
    }
    __syncthreads();
    if (threadIdx.x == 0 && score) {
        int64_t mx = loads[0], mn = loads[0];
        for (int g = 1; g < M; ++g) {
            mx = max(mx, loads[g]);
            mn = min(mn, loads[g]);
        }
        *score = (T > 0) ? (float)(mx - mn) / (float)T : 0.f;
    }
}

cudaError_t launch_imbalance(const int32_t *counts, int64_t T, int64_t N, int64_t M, int32_t *group_load,
                             float *score, cudaStream_t s) {
    cudaError_t err = launch_pdl(imbalance_kernel, dim3(1), dim3(256), (size_t)M * 8, s, counts, T, (int)N, (int)M,
                                 group_load, score);
    count_launches(1);
    return err;
}

}  // namespace moge
