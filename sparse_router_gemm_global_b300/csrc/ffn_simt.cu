// Grouped expert SwiGLU FFN on CUDA cores (fp32 FMA; the all-fp32 path).
//   stage 1: h[r,:]      = silu(x_perm[r,:] W_gate[e]^T) * (x_perm[r,:] W_up[e]^T)
//   stage 2: y_perm[r,:] = h[r,:] W_down[e]^T
// Tiles of 32 rows x 32 outputs never straddle two experts: tile i of the
// grid is mapped to (expert, row block, column block) through the prefix sum
// of ceil(count_e / 32), which every block computes from `offsets` on the
// device; blocks past the last tile return at once.
#include "common.cuh"

namespace moge {

constexpr int kTile = 32;
constexpr int kMaxExpertsSimt = 1024;

// Map a linear tile id to (expert, row block).  tiles_before[e] in shared memory; segments
// clamped to the buffer's rows.
__device__ __forceinline__ bool tile_to_expert(const int32_t *__restrict__ offsets, int N, int rows,
                                               int64_t row_tile, int32_t *tiles_before, int *expert, int64_t *rb) {
    if (threadIdx.x == 0) {
        int64_t run = 0;
        for (int e = 0; e < N; ++e) {
            tiles_before[e] = (int32_t)run;
            int begin, count;
            expert_segment(offsets, e, rows, begin, count);
            run += cdiv(count, kTile);
        }
        tiles_before[N] = (int32_t)run;
    }
    __syncthreads();
    if (row_tile >= tiles_before[N]) return false;
    int lo = 0, hi = N - 1;  // last e with tiles_before[e] <= row_tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles_before[mid] <= row_tile) lo = mid; else hi = mid - 1;
    }
    *expert = lo;
    *rb = row_tile - tiles_before[lo];
    return true;
}

// out[r, c] for r in the expert's rows, c < OUT; A [P, Kd], W [N, OUT, Kd].
template <typename T, bool GLU>
__global__ void ffn_simt_kernel(const T *__restrict__ A, const int32_t *__restrict__ offsets, int N, int rows,
                                const T *__restrict__ W0, const T *__restrict__ W1, int64_t Kd, int64_t OUT,
                                T *__restrict__ out) {
    __shared__ int32_t tiles_before[kMaxExpertsSimt + 1];
    __shared__ float as[kTile][kTile + 1];
    __shared__ float w0s[kTile][kTile + 1];
    __shared__ float w1s[GLU ? kTile : 1][kTile + 1];
    int e;
    int64_t rb;
    if (!tile_to_expert(offsets, N, rows, blockIdx.x, tiles_before, &e, &rb)) return;
    int seg0, cnt;
    expert_segment(offsets, e, rows, seg0, cnt);
    const int64_t row0 = seg0 + rb * kTile;
    const int64_t row_end = seg0 + cnt;
    const int64_t c0 = (int64_t)blockIdx.y * kTile;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 warps, 4 rows each
    const T *W0e = W0 + (int64_t)e * OUT * Kd;
    const T *W1e = GLU ? W1 + (int64_t)e * OUT * Kd : nullptr;
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t k0 = 0; k0 < Kd; k0 += kTile) {
        for (int i = threadIdx.x; i < kTile * kTile; i += blockDim.x) {
            const int r = i >> 5, c = i & 31;
            const int64_t row = row0 + r, col = c0 + r, k = k0 + c;
            as[r][c] = (row < row_end && k < Kd) ? to_f32(A[row * Kd + k]) : 0.f;
            w0s[r][c] = (col < OUT && k < Kd) ? to_f32(W0e[col * Kd + k]) : 0.f;
            if (GLU) w1s[r][c] = (col < OUT && k < Kd) ? to_f32(W1e[col * Kd + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kTile; ++k) {
            const float w0 = w0s[tx][k];
            const float w1 = GLU ? w1s[tx][k] : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float av = as[ty + 8 * j][k];
                a0[j] = fmaf(av, w0, a0[j]);
                if (GLU) a1[j] = fmaf(av, w1, a1[j]);
            }
        }
        __syncthreads();
    }
    const int64_t col = c0 + tx;
    if (col >= OUT) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t row = row0 + ty + 8 * j;
        if (row < row_end) out[row * OUT + col] = from_f32<T>(GLU ? swiglu_precise(a0[j], a1[j]) : a0[j]);
    }
}

template <typename T>
static cudaError_t ffn_simt_typed(const T *x_perm, const int32_t *offsets, int64_t N, int64_t P, int64_t d,
                                  int64_t I, const T *wg, const T *wu, const T *wd, T *h, T *y_perm,
                                  cudaStream_t s) {
    const int64_t row_tiles = cdiv(P, kTile) + N;  // upper bound of sum_e ceil(count_e / kTile)
    dim3 g1((unsigned)row_tiles, (unsigned)cdiv(I, kTile));
    ffn_simt_kernel<T, true><<<g1, 256, 0, s>>>(x_perm, offsets, (int)N, (int)P, wg, wu, d, I, h);
    count_launches(1);
    mark_stage(MOGE_STAGE_DOWN, s);
    dim3 g2((unsigned)row_tiles, (unsigned)cdiv(d, kTile));
    ffn_simt_kernel<T, false><<<g2, 256, 0, s>>>(h, offsets, (int)N, (int)P, wd, nullptr, I, d, y_perm);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_ffn_simt(const void *x_perm, const int32_t *offsets, int64_t N, int64_t P, int64_t d,
                            int64_t I, int dtype, const void *w_gate, const void *w_up, const void *w_down,
                            void *h, void *y_perm, cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    if (N > kMaxExpertsSimt) return cudaErrorInvalidValue;
    if (dtype == MOGE_BF16)
        return ffn_simt_typed<__nv_bfloat16>((const __nv_bfloat16 *)x_perm, offsets, N, P, d, I,
                                             (const __nv_bfloat16 *)w_gate, (const __nv_bfloat16 *)w_up,
                                             (const __nv_bfloat16 *)w_down, (__nv_bfloat16 *)h,
                                             (__nv_bfloat16 *)y_perm, s);
    return ffn_simt_typed<float>((const float *)x_perm, offsets, N, P, d, I, (const float *)w_gate,
                                 (const float *)w_up, (const float *)w_down, (float *)h, (float *)y_perm, s);
}

}  // namespace moge
