// Weighted combine: y[t,:] = sum_{k=0..K-1} gate[t,k] * y_perm[pair_row[t,k],:], summed in
// slot order with fp32 accumulation and rounded once to the activation dtype; with S shared
// experts their rows y_perm[shared_base + s*T + t,:] follow with weight 1, in order s = 0..S-1,
// and with a residual stream r the row r[t,:] is added last.  y may be r (each element is read
// and then written by the same thread).
// A pair_row entry outside [0, rows) (-1: the permutation skipped the slot's expert id) counts
// as an absent slot.
// Grid (token, column block): each thread owns one 16-byte column vector of one token and
// issues the loads of 8 slots before their FMAs, so the reads of y_perm stay in flight
// together instead of one round trip per slot.
#include "common.cuh"

namespace moge {

constexpr int kCombineThreads = 128;
constexpr int kSlotBatch = 8;

template <typename T, int V>  // V elements per 16-byte vector
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const T *__restrict__ y_perm, const int32_t *__restrict__ pair_row, const float *__restrict__ gate,
               int K, int64_t d, T *y, int S, int64_t shared_base, int64_t Tn, int64_t rows, const T *residual) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = blockIdx.x;
    const int64_t v = (int64_t)blockIdx.y * kCombineThreads + threadIdx.x;
    const int64_t nvec = d / V;
    if (v >= nvec) return;
    const int32_t *pr = pair_row + t * K;
    const float *gt = gate + t * K;
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += kSlotBatch) {
        int4 raw[kSlotBatch];
        float g[kSlotBatch];
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
            const int k = k0 + j;
            int row = k < K ? __ldg(pr + k) : -1;
            if (row >= rows) row = -1;
            g[j] = row >= 0 ? __ldg(gt + k) : 0.f;
            raw[j] = row >= 0 ? __ldg(reinterpret_cast<const int4 *>(y_perm + (int64_t)row * d) + v)
                              : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
            const T *e = reinterpret_cast<const T *>(&raw[j]);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(g[j], to_f32(e[i]), acc[i]);
        }
    }
    for (int s0 = 0; s0 < S; s0 += kSlotBatch) {
        int4 raw[kSlotBatch];
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
            const int64_t row = shared_base + (int64_t)(s0 + j) * Tn + t;
            raw[j] = s0 + j < S ? __ldg(reinterpret_cast<const int4 *>(y_perm + row * d) + v) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
            if (s0 + j >= S) break;
            const T *e = reinterpret_cast<const T *>(&raw[j]);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += to_f32(e[i]);
        }
    }
    if (residual) {
        const int4 rv = reinterpret_cast<const int4 *>(residual + t * d)[v];
        const T *e = reinterpret_cast<const T *>(&rv);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += to_f32(e[i]);
    }
    int4 out;
    T *o = reinterpret_cast<T *>(&out);
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = from_f32<T>(acc[i]);
    reinterpret_cast<int4 *>(y + t * d)[v] = out;
}

cudaError_t launch_combine(const void *y_perm, const int32_t *pair_row, const float *gate, int64_t T,
                           int64_t K, int64_t d, int dtype, void *y, cudaStream_t s, int64_t S, int64_t shared_base,
                           const void *residual) {
    if (T == 0) return cudaSuccess;
    const int V = dtype == MOGE_BF16 ? 8 : 4;
    dim3 grid((unsigned)T, (unsigned)cdiv(d / V, kCombineThreads));
    const int64_t rows = T * K + S * T;  // routed rows, then the shared experts' rows
    cudaError_t err = dtype == MOGE_BF16
        ? launch_pdl(combine_kernel<__nv_bfloat16, 8>, grid, dim3(kCombineThreads), 0, s,
                     (const __nv_bfloat16 *)y_perm, pair_row, gate, (int)K, d, (__nv_bfloat16 *)y, (int)S,
                     shared_base, T, rows, (const __nv_bfloat16 *)residual)
        : launch_pdl(combine_kernel<float, 4>, grid, dim3(kCombineThreads), 0, s, (const float *)y_perm, pair_row,
                     gate, (int)K, d, (float *)y, (int)S, shared_base, T, rows, (const float *)residual);
    count_launches(1);
    return err;
}

}  // namespace moge
