// Routing: global softmax over all N experts + top-K' inside each group
// (Pangu Pro MoE explainer, section 1 "innovative architecture"), and the
// conventional top-K over all experts it is compared with.
//
// A block stages 64 tokens' N scores in shared memory (row stride N+1) and
// routes them with route_rows_block: the selection compares fp32 scores with
// equal scores going to the lower expert index, so it is independent of how
// exp() rounds; the gates are exp(l - max) / sum_e exp(l_e - max).
#include "common.cuh"
#include "route_token.cuh"

namespace moge {

constexpr int kSelectThreads = 128;
constexpr int kSelectRows = 64;  // tokens per block (32 when N > 639, to fit the score tile)

__global__ void __launch_bounds__(kSelectThreads)
route_select_kernel(const float *__restrict__ logits, int T, int N, int groups, int G, int per, int rows_pb,
                    int32_t *__restrict__ idx, float *__restrict__ gate) {
    extern __shared__ float tile[];  // [rows_pb][N+1]
    __shared__ float row_max[kSelectRows], row_sum[kSelectRows];
    pdl_wait();
    pdl_trigger();
    const int64_t t0 = (int64_t)blockIdx.x * rows_pb;
    const int ntok = (int)min((int64_t)rows_pb, (int64_t)T - t0);
    const int stride = N + 1;
    const float *src = logits + t0 * N;
    for (int i = threadIdx.x; i < ntok * N; i += kSelectThreads) {
        const int r = i / N, c = i - r * N;
        tile[r * stride + c] = src[i];
    }
    __syncthreads();
    const int K = groups * per;
    route_rows_block(tile, stride, 0, ntok, N, groups, G, per, idx + t0 * K, gate + t0 * K, row_max, row_sum);
}

cudaError_t launch_route_select(const float *logits, int64_t T, int64_t N, int64_t M, int64_t kpg,
                                bool global, int32_t *idx, float *gate, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int rows_pb = N <= 639 ? kSelectRows : kSelectRows / 2;
    const size_t smem = (size_t)rows_pb * (N + 1) * sizeof(float);
    cudaError_t err = set_max_smem(route_select_kernel, (int)smem);
    if (err != cudaSuccess) return err;
    const int groups = global ? 1 : (int)M;
    const int G = global ? (int)N : (int)(N / M);
    const int per = global ? (int)(M * kpg) : (int)kpg;
    err = launch_pdl(route_select_kernel, dim3((unsigned)cdiv(T, rows_pb)), dim3(kSelectThreads), smem, s,
                     logits, (int)T, (int)N, groups, G, per, rows_pb, idx, gate);
    count_launches(1);
    return err;
}

// ---------------------------------------------------------------------------------------------
// Router projection on CUDA cores: logits[t,e] = sum_i x[t,i] W_r[e,i] + b[e] (fp32 accumulate).
// 32 tokens x 32 experts per block, 256 threads, 4 outputs per thread, k-chunks of 32.
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void router_logits_simt_kernel(const T *__restrict__ x, const T *__restrict__ w,
                                          const float *__restrict__ bias, int Tn, int d, int N,
                                          float *__restrict__ logits) {
    __shared__ float xs[32][33];
    __shared__ float ws[32][33];
    const int t0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // ty in [0,8)
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < d; k0 += 32) {
        for (int i = threadIdx.x; i < 32 * 32; i += 256) {
            const int r = i >> 5, c = i & 31;
            const int t = t0 + r, e = e0 + r, k = k0 + c;
            xs[r][c] = (t < Tn && k < d) ? to_f32(x[(int64_t)t * d + k]) : 0.f;
            ws[r][c] = (e < N && k < d) ? to_f32(w[(int64_t)e * d + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float wv = ws[tx][k];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(xs[ty + 8 * j][k], wv, acc[j]);
        }
        __syncthreads();
    }
    const int e = e0 + tx;
    if (e < N) {
        const float b = bias ? bias[e] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + ty + 8 * j;
            if (t < Tn) logits[(int64_t)t * N + e] = acc[j] + b;
        }
    }
}

cudaError_t launch_router_logits_simt(const void *x, const void *w_r, const float *bias, int64_t T,
                                      int64_t d, int64_t N, int dtype, float *logits, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    dim3 grid((unsigned)cdiv(T, 32), (unsigned)cdiv(N, 32));
    if (dtype == MOGE_BF16)
        router_logits_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w_r, bias, (int)T, (int)d, (int)N, logits);
    else
        router_logits_simt_kernel<float><<<grid, 256, 0, s>>>((const float *)x, (const float *)w_r, bias,
                                                               (int)T, (int)d, (int)N, logits);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace moge
