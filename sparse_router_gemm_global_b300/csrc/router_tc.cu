// Fused router on tcgen05 tensor cores: scores = x W_r^T + b (bf16 in, fp32 accumulation in
// TMEM), then, in the same launch, the global softmax over all N experts and the top-K'
// selection inside every group (Pangu Pro MoE explainer, section 1: scores for all experts,
// one softmax over them, a local top-K' per group).
//
// One CTA per (128-token tile, slice of the reduction over d).  512 threads: thread 0 of warp 0
// issues TMA loads, thread 0 of warp 1 issues the MMAs (M = 128 tokens, N = N rounded up to 16
// experts), then all sixteen warps drain TMEM into shared memory (warp w reads TMEM lanes
// 32(w%4)..+31 = token rows, column chunks w/4, w/4+4, ...).  The epilogue (reduction of the
// slices, bias, softmax, selection) is latency-bound serial work per row, so it is spread over
// all sixteen warps: with four it took as long as streaming x through the MMAs.  The S slices of a tile form one thread-block cluster: after a cluster
// barrier, CTA j adds the S partial tiles for its share of the 128 tokens through distributed
// shared memory, in slice order (so the result does not depend on timing), and routes those
// tokens.  No CTA waits on a counter and nothing goes through global memory.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "route_token.cuh"
#include "tc_ptx.cuh"
#include "tc_wait.cuh"

namespace moge {
namespace rt {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kBM = kRouterTileRows;   // tokens per tile (MMA M)
constexpr int kBK = 64;                // bf16 elements per k-block (one 128-byte swizzle row)
constexpr int kMaxStages = 8;
constexpr int kMaxSlices = 8;          // slices of a tile = CTAs of its cluster (portable size)
constexpr int kSmemBudget = 200 * 1024;

struct Params {
    int T, d, N, npad, kblocks, kslices, kb_per_slice, stages, stage_bytes, tmem_cols;
    int groups, G, per;
    uint32_t idesc;
    const float *bias;
    float *logits;     // optional [T, N] output
    int32_t *idx;      // [T, K]
    float *gate;       // [T, K]
    uint32_t *status;
};

__global__ void __launch_bounds__(kThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                 const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], tfull_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float row_max[kBM], row_sum[kBM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = smem_u32(smem);
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int t0 = tile * kBM;
    const int ntok = min(kBM, p.T - t0);
    const int kb0 = slice * p.kb_per_slice;
    const int kb1 = min(p.kblocks, kb0 + p.kb_per_slice);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&tfull_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_w);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = tmem_slot;
    volatile int *abort_v = &abort_flag;

    if (warp == 0 && lane == 0) {
        // TMA producer
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % p.stages;
            const uint32_t ph = (it / p.stages) & 1;
            if (!wait_bar(smem_u32(&empty_bar[s]), ph ^ 1, abort_v, p.status)) break;
            const uint32_t fb = smem_u32(&full_bar[s]);
            const uint32_t sa = smem_base + s * p.stage_bytes;
            mbar_arrive_expect_tx(fb, p.stage_bytes);
            tma_load_2d(sa, &map_x, fb, kb * kBK, t0);                    // 128 token rows
            tma_load_2d(sa + kBM * 128, &map_w, fb, kb * kBK, 0);         // npad expert rows
        }
        for (uint32_t j = (it > (uint32_t)p.stages ? it - p.stages : 0); j < it; ++j)
            drain_wait(smem_u32(&full_bar[j % p.stages]), (j / p.stages) & 1, p.status);
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % p.stages;
            const uint32_t ph = (it / p.stages) & 1;
            if (!wait_bar(smem_u32(&full_bar[s]), ph, abort_v, p.status)) break;
            tc_fence_after();
            const uint32_t sa = smem_base + s * p.stage_bytes;
            const uint32_t sb = sa + kBM * 128;
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
                mma_bf16(tmem, smem_desc_sw128(sa + j * 32), smem_desc_sw128(sb + j * 32), p.idesc,
                         (kb > kb0 || j > 0) ? 1u : 0u);
            mma_commit(smem_u32(&empty_bar[s]));
        }
        mma_commit(smem_u32(&tfull_bar));  // also the drain: arrives once every MMA above is done
    }
    __syncwarp();

    // ---- drain TMEM into this CTA's partial tile: thread = token row r, stage[r][N+1]
    bool ok = wait_bar(smem_u32(&tfull_bar), 0, abort_v, p.status);
    ok = __all_sync(0xffffffffu, ok) && !*abort_v;
    tc_fence_after();
    const int quarter = warp & 3;  // TMEM lanes a warp may read: 32 * (warp % 4) ..
    const int r = quarter * 32 + lane;
    const int stride = p.N + 1;
    float *stage = reinterpret_cast<float *>(smem);  // [128][N+1], reuses the pipeline buffers
    const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
    for (int c0 = (warp >> 2) * 16; c0 < p.npad; c0 += 16 * (kThreads / 128)) {
        uint32_t v[16];
        if (ok) {
            tmem_ld_x16(taddr + c0, v);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = c0 + j;
            if (c < p.N) stage[r * stride + c] = __uint_as_float(v[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);

    // ---- the slices' partial tiles are summed in slice order; CTA `slice` takes the rows
    // [slice * rows_per, (slice + 1) * rows_per) of the tile
    const int S = p.kslices;
    const int rows_per = (kBM + S - 1) / S;
    const int r0 = slice * rows_per, r1 = min(kBM, r0 + rows_per);
    if (S > 1) {
        cluster_sync();  // every partial tile of the cluster is in shared memory
        const uint32_t my_stage = smem_u32(stage);
        for (int i = threadIdx.x; i < (r1 - r0) * p.N; i += kThreads) {
            const int rr = r0 + i / p.N, c = i - (i / p.N) * p.N;
            const uint32_t off = (uint32_t)(rr * stride + c) * 4u;
            float v[kMaxSlices];  // all slices' loads in flight together, then added in slice order
#pragma unroll
            for (int q = 0; q < kMaxSlices; ++q)
                v[q] = q < S ? ld_shared_cluster_f32(mapa_shared(my_stage + off, (uint32_t)q)) : 0.f;
            float acc = v[0];
#pragma unroll
            for (int q = 1; q < kMaxSlices; ++q)
                if (q < S) acc += v[q];
            if (p.bias) acc += p.bias[c];
            stage[rr * stride + c] = acc;  // rows [r0, r1) of this CTA are read by no other CTA
            if (p.logits && t0 + rr < p.T) p.logits[(size_t)(t0 + rr) * p.N + c] = acc;
        }
    } else {  // one slice: the bias pass alone
        for (int i = threadIdx.x; i < (r1 - r0) * p.N; i += kThreads) {
            const int rr = r0 + i / p.N, c = i - (i / p.N) * p.N;
            float v = stage[rr * stride + c];
            if (p.bias) v += p.bias[c];
            stage[rr * stride + c] = v;
            if (p.logits && t0 + rr < p.T) p.logits[(size_t)(t0 + rr) * p.N + c] = v;
        }
    }
    __syncthreads();

    // ---- softmax + selection of this CTA's rows
    const int rows = min(r1, ntok) - r0;
    if (rows > 0)
        route_rows_block(stage, stride, r0, r0 + rows, p.N, p.groups, p.G, p.per, p.idx + (size_t)t0 * (p.groups * p.per),
                         p.gate + (size_t)t0 * (p.groups * p.per), row_max, row_sum);
    if (S > 1) cluster_sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace rt

cudaError_t launch_router_tc(const void *x, const void *w_r, const float *bias, int64_t T, int64_t d, int64_t N,
                             int64_t M, int64_t kpg, bool global, float *logits_out, int32_t *idx, float *gate,
                             uint32_t *status, cudaStream_t s) {
    using namespace rt;
    if (T == 0) return cudaSuccess;
    if (N > 256) return cudaErrorInvalidValue;
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!fn) return cudaErrorNotSupported;
    Params p{};
    p.T = (int)T;
    p.d = (int)d;
    p.N = (int)N;
    p.npad = (int)round_up(N, 16);
    p.kblocks = (int)cdiv(d, kBK);
    p.kslices = router_kslices(T, d, N);
    p.kb_per_slice = (int)cdiv(p.kblocks, p.kslices);
    p.kslices = (int)cdiv(p.kblocks, p.kb_per_slice);  // no empty slice
    p.stage_bytes = kBM * 128 + p.npad * 128;
    p.stages = std::min(kMaxStages, kSmemBudget / p.stage_bytes);
    int cols = 32;
    while (cols < p.npad) cols <<= 1;
    p.tmem_cols = cols;
    p.groups = global ? 1 : (int)M;
    p.G = global ? (int)N : (int)(N / M);
    p.per = global ? (int)(M * kpg) : (int)kpg;
    p.idesc = ptx::idesc_bf16_f32(kBM, p.npad);
    p.bias = bias;
    p.logits = logits_out;
    p.idx = idx;
    p.gate = gate;
    p.status = status;
    const size_t stage_floats = (size_t)kBM * (N + 1) * 4;
    size_t smem = std::max((size_t)p.stages * p.stage_bytes, stage_floats) + 1024;

    CUtensorMap mx, mw;
    {
        cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)T};
        cuuint64_t strides[1] = {(cuuint64_t)d * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)d * 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)p.npad};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_r), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t err = set_max_smem(router_tc_kernel, (int)smem);
    if (err != cudaSuccess) return err;
    // the slices of a tile form one cluster (1 x kslices)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)cdiv(T, kBM), (unsigned)p.kslices);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = (unsigned)p.kslices;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, router_tc_kernel, mx, mw, p);
    count_launches(1);
    return err;
}

}  // namespace moge
