// Weighted combine: y[t,:] = sum_{k=0..K-1} gate[t,k] * y_perm[pair_row[t,k],:], summed in
// slot order with fp32 accumulation and rounded once to the activation dtype.
// One block per token; each thread owns 16-byte column vectors of the row.
#include "common.cuh"

namespace moge {

template <typename T, int V>  // V elements per 16-byte vector
__global__ void combine_kernel(const T *__restrict__ y_perm, const int32_t *__restrict__ pair_row,
                               const float *__restrict__ gate, int K, int64_t d, T *__restrict__ y) {
    extern __shared__ float sgate[];  // [K] gates, then [K] rows (as int)
    int32_t *srow = (int32_t *)(sgate + K);
    const int64_t t = blockIdx.x;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        sgate[k] = gate[t * K + k];
        srow[k] = pair_row[t * K + k];
    }
    __syncthreads();
    const int64_t nvec = d / V;
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        float acc[V];
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = 0.f;
        for (int k = 0; k < K; ++k) {
            const int row = srow[k];
            if (row < 0) continue;
            const float g = sgate[k];
            const int4 raw = __ldg((const int4 *)(y_perm + (int64_t)row * d) + v);
            const T *e = (const T *)&raw;
#pragma unroll
            for (int j = 0; j < V; ++j) acc[j] = fmaf(g, to_f32(e[j]), acc[j]);
        }
        int4 out;
        T *o = (T *)&out;
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = from_f32<T>(acc[j]);
        ((int4 *)(y + t * d))[v] = out;
    }
}

cudaError_t launch_combine(const void *y_perm, const int32_t *pair_row, const float *gate, int64_t T,
                           int64_t K, int64_t d, int dtype, void *y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)K * 8;
    const int threads = 128;
    if (dtype == MOGE_BF16)
        combine_kernel<__nv_bfloat16, 8><<<(unsigned)T, threads, smem, s>>>(
            (const __nv_bfloat16 *)y_perm, pair_row, gate, (int)K, d, (__nv_bfloat16 *)y);
    else
        combine_kernel<float, 4><<<(unsigned)T, threads, smem, s>>>((const float *)y_perm, pair_row, gate,
                                                                    (int)K, d, (float *)y);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moge
