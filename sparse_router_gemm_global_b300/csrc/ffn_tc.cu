// Grouped expert SwiGLU FFN on 5th-generation tensor cores (tcgen05, sm_103a).
//
// Each GEMM (gate/up + SwiGLU -> h, then down -> y_perm) runs as persistent launches with one CTA
// per SM walking a tile list derived on the device from the expert offsets (no host round trip).
// Per CTA: warp 0 issues TMA loads into a shared-memory ring, warp 1 issues tcgen05.mma from one
// thread into TMEM accumulators, warp 2 owns the TMEM allocation, warps 4-7 (4-11 in the
// two-region CTA-pair tiles) drain TMEM (tcgen05.ld), apply the epilogue and store bf16.
//
// Tile shapes (M x N x K = rows of operand A x rows of operand B x 64 per k-block):
//   tokens-as-M on CTA pairs (cta_group::2), experts with more than kSmallExpertRows rows of a
//   batch whose experts hold many rows on average:
//     gate/up: A = 256 permuted token rows, two regions of B = 128 W_gate rows (even CTA) and the
//              matching 128 W_up rows (odd CTA); epilogue h = silu(acc[:, :128]) * acc[:, 128:]
//              per region, 256 features of h per tile.
//     down:    A = 256 h rows, B = 256 W_down rows; epilogue y_perm = acc.
//     Tiles are taken in list order from a counter.
//   weights-as-M ("swap") on single CTAs: A = 128 weight rows, B = the expert's token rows (BNT
//     per tile), so the weights stream at full MMA height; gate/up issue one MMA for W_gate and
//     one for W_up into two TMEM column ranges.  Every expert of a batch whose experts hold few
//     rows on average, or the experts of at most kSmallExpertRows rows beside the pair launch.
// Rows of a tile never belong to two experts: the tile list is built per expert, rows past
// the expert's count (or past the tensor) are loaded (other experts' rows or TMA zero fill)
// but never stored.
//
// Every mbarrier wait is bounded (kWaitTimeoutNs).  A wait that gives up sets the workspace
// status word (MOGE_ERR_TIMEOUT through moge_query_device_status), raises a CTA-wide abort
// flag that ends the other roles' loops, drains the copies and MMAs it issued and frees TMEM
// before the CTA exits.
#include <cudaTypedefs.h>
#include <mutex>

#include "ffn_tc.cuh"
#include "tc_ptx.cuh"
#include "tc_wait.cuh"

namespace moge {
namespace tc {

using namespace ptx;

constexpr int kBM = 128;            // MMA M
constexpr int kBK = 64;             // k-block: 64 bf16 = 128 bytes = one 128B-swizzle row
constexpr int kThreads = 256;       // 8 warps
constexpr int kEpiWarp0 = 4;        // epilogue warps 4..7 (TMEM lane quarter = warp % 4)
constexpr int kMaxExperts = 1024;
constexpr int kSmemBudget = 220 * 1024;

// Weights-as-M modes of the single-CTA kernel (values kept from the kernels' earlier names).
enum Mode { SWAP_GLU = 2, SWAP_PLAIN = 3 };

constexpr int kPairRows = 256;         // token rows of a CTA-pair tile
constexpr int kSmallExpertRows = 64;   // experts with at most this many rows take weights-as-M tiles
constexpr int kSmallExpertTile = 32;   // tokens per weights-as-M tile of those experts

// Which experts a single-CTA launch covers, and with how many token blocks of tok_block rows.
//   kBlocksAll:          every expert (the batch's tile plan chose weights-as-M tiles);
//   kBlocksSmallExperts: only experts with 1..kSmallExpertRows rows (the CTA-pair launch takes
//                        the others).
enum BlockRule { kBlocksAll = 0, kBlocksSmallExperts = 1 };

__device__ __forceinline__ int expert_blocks(int c, int tok_block, int rule) {
    if (rule == kBlocksSmallExperts && c > kSmallExpertRows) return 0;
    return (c + tok_block - 1) / tok_block;
}

// Tile geometry of the single-CTA weights-as-M kernel: A = 128 weight rows (two A tiles, W_gate
// and W_up, for gate/up), B = BNT token rows; 128 output features per tile.
template <int MODE, int BNT>
struct Cfg {
    static constexpr bool glu = MODE == SWAP_GLU;
    static constexpr int mma_n = BNT;                                   // MMA N (rows of operand B)
    static constexpr int tok_block = BNT;                               // tokens per tile
    static constexpr int feat_block = 128;                              // output features per tile
    static constexpr int a_tiles = glu ? 2 : 1;                         // W_gate + W_up as two A tiles
    static constexpr int a_bytes = kBM * 128;                           // one 128-row A tile
    static constexpr int b_bytes = mma_n * 128;
    static constexpr int stage_bytes = a_tiles * a_bytes + b_bytes;
    static constexpr int stages_raw = kSmemBudget / stage_bytes;
    static constexpr int stages = stages_raw > 12 ? 12 : stages_raw;
    static constexpr int acc_cols = glu ? 2 * BNT : BNT;                // fp32 columns per accumulator
    static constexpr int tmem_cols = (2 * acc_cols <= 32) ? 32 : (2 * acc_cols <= 64) ? 64
                                   : (2 * acc_cols <= 128) ? 128 : (2 * acc_cols <= 256) ? 256 : 512;
    static constexpr uint32_t idesc = idesc_bf16_f32(kBM, mma_n);
    static constexpr size_t smem_bytes = (size_t)stages * stage_bytes + 1024;  // + alignment slack
    static_assert(stage_bytes % 1024 == 0, "stage tiles must keep 1024-byte alignment");
    static_assert(stages >= 2, "pipeline needs two stages");
};

struct Params {
    const int32_t *offsets;  // [N+1] expert row offsets (device)
    int N;                   // experts
    int kdim;                // reduction length (d for gate/up, I for down)
    int out_dim;             // output features (I for gate/up, d for down)
    __nv_bfloat16 *out;      // [P, out_dim]
    uint32_t *status;        // workspace status word
    const int32_t *row_token;  // [P] token of each permuted row (gathering launches only)
    int rule;                  // BlockRule of the tile list
    int rows;                  // rows of the row buffers (act / out): segments are clamped to them
    uint32_t *sched;           // CTA-pair launches: {next tile, finished CTAs}, zero between launches
};

// prefix[e] = sum over e' < e of count(c_e'), c_e' = rows of expert e' (its segment clamped to
// the buffer's rows); every thread of the block (256..512 threads, warp_sums[16]), N <= 1024.
template <typename CountFn>
__device__ void build_prefix(const int32_t *__restrict__ offsets, int N, int rows, CountFn count, int32_t *prefix,
                             int32_t *warp_sums, int32_t *seg_begin = nullptr, int32_t *seg_count = nullptr) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    int v[4];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = t * 4 + i;
        int b = 0;
        if (e < N) {
            int begin, c;
            expert_segment(offsets, e, rows, begin, c);
            b = count(c);
            if (seg_begin) {  // segments cached in shared memory for the per-tile lookups
                seg_begin[e] = begin;
                seg_count[e] = c;
            }
        }
        local += b;
        v[i] = local;
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        const int nw = (int)(blockDim.x >> 5);
        int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = x - local + (w > 0 ? warp_sums[w - 1] : 0);
    if (t == 0) prefix[0] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = t * 4 + i;
        if (e < N) prefix[e + 1] = excl + v[i];
    }
    __syncthreads();
}

// tile -> (expert, token block inside the expert, feature block)
__device__ __forceinline__ void tile_coords(int tile, int nfb, const int32_t *prefix, int N, int &e, int &tb,
                                            int &fb) {
    const int tbg = tile / nfb;
    fb = tile - tbg * nfb;
    int lo = 0, hi = N - 1;  // last e with prefix[e] <= tbg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tbg) lo = mid; else hi = mid - 1;
    }
    e = lo;
    tb = tbg - prefix[lo];
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int MODE, int BNT, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
              const __grid_constant__ CUtensorMap map_b1, const Params p) {
    using C = Cfg<MODE, BNT>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int32_t prefix[kMaxExperts + 1];
    __shared__ int32_t warp_sums[16];
    __shared__ __align__(8) uint64_t full_bar[C::stages], empty_bar[C::stages];
    __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), 4);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b0);
        if (C::glu) tma_prefetch_desc(&map_b1);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&tmem_base_slot), C::tmem_cols);
        tmem_relinquish();
    }
    pdl_wait();  // the offsets (and the token rows) come from earlier kernels
    pdl_trigger();
    const int rule = p.rule;
    build_prefix(p.offsets, p.N, p.rows, [rule](int c) { return expert_blocks(c, C::tok_block, rule); }, prefix,
                 warp_sums);  // contains __syncthreads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;

    const int nfb = (p.out_dim + C::feat_block - 1) / C::feat_block;
    const int total_tiles = prefix[p.N] * nfb;
    const int kblocks = (p.kdim + kBK - 1) / kBK;
    volatile int *abort_v = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // Lane 0 owns the barriers and the weight loads.  With GATHER the token rows of the tile
        // come straight from x (map_a has a one-row box): lane i gathers tile rows 4i..4i+3 with
        // one tile::gather4 copy per k-block, through the row -> token map; otherwise lane 0 loads
        // the rows of the already permuted matrix as one tile.
        const bool gather_lane = GATHER && lane * 4 < BNT;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            int e, tb, fb;
            tile_coords(tile, nfb, prefix, p.N, e, tb, fb);
            int seg0, cnt;
            expert_segment(p.offsets, e, p.rows, seg0, cnt);
            const int tok0 = seg0 + tb * C::tok_block;
            const int f0 = fb * C::feat_block;
            int r4[4] = {0, 0, 0, 0};
            if (gather_lane) {
                const int last = seg0 + cnt - 1;  // rows past the expert repeat its last row
#pragma unroll
                for (int j = 0; j < 4; ++j) r4[j] = p.row_token[min(tok0 + lane * 4 + j, last)];
            }
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % C::stages;
                const uint32_t ph = (it / C::stages) & 1;
                const uint32_t fb_ = smem_u32(&full_bar[s]);
                int go = 1;
                if (lane == 0) {
                    go = wait_bar(smem_u32(&empty_bar[s]), ph ^ 1, abort_v, p.status);
                    if (go) mbar_arrive_expect_tx(fb_, C::stage_bytes);
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) { ok = false; break; }
                const uint32_t sa = smem_base + s * C::stage_bytes;
                const uint32_t sb = sa + C::a_tiles * C::a_bytes;
                const int k0 = kb * kBK;
                if (lane == 0) {
                    tma_load_3d(sa, &map_b0, fb_, k0, f0, e);                                // W_gate / W_down
                    if (C::glu) tma_load_3d(sa + C::a_bytes, &map_b1, fb_, k0, f0, e);      // W_up
                }
                if constexpr (GATHER) {
                    if (gather_lane) tma_gather4(sb + lane * 512, &map_a, fb_, k0, r4[0], r4[1], r4[2], r4[3]);
                } else {
                    if (lane == 0) tma_load_2d(sb, &map_a, fb_, k0, tok0);                   // token rows
                }
            }
        }
        // drain: the last fill of every stage must have landed before the CTA may exit
        if (lane == 0)
            for (uint32_t j = (it > (uint32_t)C::stages ? it - C::stages : 0); j < it; ++j)
                drain_wait(smem_u32(&full_bar[j % C::stages]), (j / C::stages) & 1, p.status);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t use = local >> 1;
                if (!wait_bar(smem_u32(&tempty_bar[acc]), (use & 1) ^ 1, abort_v, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::acc_cols;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % C::stages;
                    const uint32_t ph = (it / C::stages) & 1;
                    if (!wait_bar(smem_u32(&full_bar[s]), ph, abort_v, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_base + s * C::stage_bytes;
                    const uint32_t sb = sa + C::a_tiles * C::a_bytes;
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j) {
                        const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
                        const uint64_t bdesc = smem_desc_sw128(sb + j * 32);
                        mma_bf16(d_tmem, smem_desc_sw128(sa + j * 32), bdesc, C::idesc, accum);
                        if (C::glu)
                            mma_bf16(d_tmem + BNT, smem_desc_sw128(sa + C::a_bytes + j * 32), bdesc, C::idesc,
                                     accum);
                    }
                    mma_commit(smem_u32(&empty_bar[s]));  // frees the stage once these MMAs are done
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[acc]));      // accumulator ready for the epilogue
            }
            // drain: no MMA may be in flight when TMEM is freed
            mma_commit(smem_u32(&drain_bar));
            drain_wait(smem_u32(&drain_bar), 0, p.status);
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------ epilogue (warps 4..7)
        const int q = warp & 3;                    // TMEM lane quarter
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t use = local >> 1;
            bool ok = wait_bar(smem_u32(&tfull_bar[acc]), use & 1, abort_v, p.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            int e, tb, fb;
            tile_coords(tile, nfb, prefix, p.N, e, tb, fb);
            int seg0, cnt;
            expert_segment(p.offsets, e, p.rows, seg0, cnt);
            const int tok0 = seg0 + tb * C::tok_block;
            const int ntok = min(C::tok_block, cnt - tb * C::tok_block);  // valid token rows of this tile
            const int f0 = fb * C::feat_block;
            const uint32_t t_acc = tmem_base + acc * C::acc_cols + lane_addr;
            {
                // thread = output feature f; columns = token rows of the tile
                const int f = f0 + q * 32 + lane;
                const bool f_ok = f < p.out_dim;
                constexpr int CH = BNT < 32 ? BNT : 32;
#pragma unroll 1
                for (int c = 0; c < C::tok_block / CH; ++c) {
                    float o[CH];
                    if constexpr (CH == 32) {
                        uint32_t va[32];
                        tmem_ld_x32(t_acc + c * 32, va);
                        if constexpr (C::glu) {
                            uint32_t vu[32];
                            tmem_ld_x32(t_acc + BNT + c * 32, vu);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < CH; ++j)
                                o[j] = swiglu_fast(__uint_as_float(va[j]), __uint_as_float(vu[j]));
                        } else {
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < CH; ++j) o[j] = __uint_as_float(va[j]);
                        }
                    } else {
                        uint32_t va[16];
                        tmem_ld_x16(t_acc + c * 16, va);
                        if constexpr (C::glu) {
                            uint32_t vu[16];
                            tmem_ld_x16(t_acc + BNT + c * 16, vu);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < CH; ++j)
                                o[j] = swiglu_fast(__uint_as_float(va[j]), __uint_as_float(vu[j]));
                        } else {
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < CH; ++j) o[j] = __uint_as_float(va[j]);
                        }
                    }
                    if (f_ok) {
#pragma unroll
                        for (int j = 0; j < CH; ++j) {
                            const int t = c * CH + j;
                            if (t < ntok) p.out[(int64_t)(tok0 + t) * p.out_dim + f] = __float2bfloat16_rn(o[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem_base, C::tmem_cols);
}

// Stores a warp's 32 rows x 32 bf16 outputs (thread = row, o its 32 values) as 64-byte row
// segments: each thread packs its row into the warp's 2 KB staging buffer (16-byte units
// XOR-swizzled by row, so the eight threads of each shared-memory phase hit distinct banks), then
// each group of four lanes stores one row's 64 contiguous bytes -- a store instruction covers 8
// rows in whole 32-byte sectors instead of 32 rows in 16-byte pieces.  Rows >= nvalid and columns
// >= out_dim are not stored (out_dim is a multiple of 8).
__device__ __forceinline__ void store_rows_staged(const float (&o)[32], uint4 *stage, int lane,
                                                  __nv_bfloat16 *out, int64_t row0, int nvalid, int col0,
                                                  int out_dim) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint4 pk;
        pk.x = pack_bf16x2(o[v * 8 + 0], o[v * 8 + 1]);
        pk.y = pack_bf16x2(o[v * 8 + 2], o[v * 8 + 3]);
        pk.z = pack_bf16x2(o[v * 8 + 4], o[v * 8 + 5]);
        pk.w = pack_bf16x2(o[v * 8 + 6], o[v * 8 + 7]);
        stage[lane * 4 + (v ^ ((lane >> 1) & 3))] = pk;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2), j = lane & 3;
        const uint4 pk = stage[r * 4 + (j ^ ((r >> 1) & 3))];
        const int col = col0 + 8 * j;
        if (r < nvalid && col < out_dim) *reinterpret_cast<uint4 *>(out + (row0 + r) * out_dim + col) = pk;
    }
    __syncwarp();  // the buffer is rewritten by the next chunk
}

// ---------------------------------------------------------------------------------------------
// CTA-pair grouped GEMM (cluster of 2, tcgen05 cta_group::2): tokens-as-M tiles of the experts
// that hold more than kSmallExpertRows rows (the others take weights-as-M tiles in a second,
// single-CTA launch: see launch_ffn_tc).
//
// A tile covers 256 token rows x NREG regions of 256 accumulator columns.  A region is one N=256
// MMA per 16-deep k-step: each CTA of the pair supplies its 128 token rows (A, shared by the
// regions) and half of the region's 256 weight rows (gate/up: the even CTA W_gate, the odd CTA
// the matching W_up rows, so a region yields both halves of 128 features and the epilogue
// applies SwiGLU; down: 128 W_down rows each, 256 outputs).  Per k-block each SM receives 16 KB
// of token rows and NREG x 16 KB of weight rows.
//   NREG = 2 (gate/up): 256 features of h per tile, four 48 KB ring stages.  The two regions share
//     the token rows, so a k-block costs a quarter fewer operand bytes per FLOP than one region,
//     which sets the pace here (the copies of one-region tiles, timed alone, take nearly as long
//     as the whole GEMM).  The accumulator fills all 512 TMEM columns, so the MMAs of the next
//     tile wait for its drain: each region has its own full / empty barrier pair and its own four
//     epilogue warps (warps 4-7: region 0, warps 8-11: region 1), so both regions drain at once.
//     The 4096-deep reduction of gate/up keeps that wait to a few per cent of a tile.  A tile
//     whose second region starts past the last feature skips that region.
//   NREG = 1 (down): 256 outputs per tile, six 32 KB stages, two 256-column accumulators used in
//     turn, so the epilogue of a tile overlaps the MMAs of the next (the short reduction of the
//     down GEMM, d_ff deep, leaves too little MMA time per tile to hide a drain).
// The even CTA's thread issues the MMAs; its full barrier counts the bytes of both CTAs' copies
// (signalled across the pair), its commits arrive on both CTAs' empty and accumulator-full
// barriers, and both CTAs' epilogue warps arrive on its accumulator-empty barriers.  Each CTA's
// TMEM holds its own 128 rows x 512 fp32 columns.
// ---------------------------------------------------------------------------------------------
constexpr int kPairBlockBytes = kBM * 128;                 // 128 rows of one k-block (16 KB)
constexpr uint32_t kPairIdesc = idesc_bf16_f32(256, 256);
constexpr int kPairTmemCols = 512;

template <bool GLU, int NREG>
struct PairCfg {
    static constexpr int region_feat = GLU ? 128 : 256;                 // output features of a region
    static constexpr int feat = NREG * region_feat;                     // output features of a tile
    static constexpr int stage_bytes = (1 + NREG) * kPairBlockBytes;    // per CTA: token rows + weights
    static constexpr int stages = NREG == 1 ? 6 : 4;
    static constexpr int epi_warps = 4 * NREG;                          // warps 4 .. 3 + epi_warps
    static constexpr int threads = 32 * (4 + epi_warps);
    static constexpr size_t smem = (size_t)stages * stage_bytes + epi_warps * 2048 + 1024;  // ring, staging, align
    // two-region tiles: the even CTA's producer takes the tile ids just in time (else warp 3 does)
    static constexpr bool producer_claims = NREG == 2;
    // readers of a tile-ring slot: even CTA MMA thread, epilogue warps (and producer, unless it
    // takes the ids); odd CTA producer and epilogue warps
    static constexpr int slot_readers = 2 + 2 * epi_warps + (producer_claims ? 0 : 1);
};

// 256-row blocks of an expert with c rows in the CTA-pair launch.
__device__ __forceinline__ int pair_blocks(int c) { return c > kSmallExpertRows ? (int)cdiv(c, kPairRows) : 0; }

struct PairTile {
    int e;          // expert
    int row0;       // first row of the block (row of the activation / output buffers)
    int nrows;      // valid rows of the block
    int f0;         // first output feature of the tile
};

// tile -> PairTile from the prefix and the segments cached in shared memory.
__device__ __forceinline__ PairTile pair_tile(int tile, const int32_t *prefix, const int32_t *seg_begin,
                                              const int32_t *seg_count, int N, int nfb, int feat) {
    int lo = 0, hi = N - 1;  // last e with prefix[e] <= tile (that expert has tiles)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int local = tile - prefix[lo], pb = local / nfb;
    PairTile t;
    t.e = lo;
    t.row0 = seg_begin[lo] + pb * kPairRows;
    t.nrows = min(kPairRows, seg_count[lo] - pb * kPairRows);
    t.f0 = (local - pb * nfb) * feat;
    return t;
}

// Whether a two-region tile's second region holds output features.  Every expert contributes a
// multiple of nfb tiles, so the feature block is tile % nfb and no lookup is needed: only the
// last feature block can lack its second region.
__device__ __forceinline__ bool pair_tile_two_regions(int tile, int nfb, bool last_has_two) {
    return last_has_two || (tile % nfb) != nfb - 1;
}

// Dynamic tile order.  Tiles are taken in list order from a global counter by whichever pair is
// free: the tiles in flight stay a narrow window of the list (their A rows and weights stay in
// L2) and the pairs finish together.  Tile ids reach both CTAs' producers, the MMA thread and both
// CTAs' epilogue warps through a small ring in shared memory (kTileSlots ids), filled by the even
// CTA.  The MMA thread looks nothing up at a tile boundary (a shared-memory lookup there measured
// 5 % more cycles: the tensor pipe idles while it runs).  Who takes the ids:
//   one-region tiles (all of one length): a scheduler thread (warp 3 of the even CTA) takes each
//     id as soon as a ring slot frees, a few tiles ahead, so the odd CTA's producer never waits
//     for one at a tile boundary (taking them just in time made the down GEMM 5-9 % slower);
//   two-region tiles: the even CTA's producer takes the id of its next tile kClaimAhead k-blocks
//     before the end of the current tile's copies and publishes it a few k-blocks later.  Ids
//     taken tiles ahead would make each pair's lead the summed duration of its queued tiles,
//     which differ with the half-length last feature block; the six tiles that share a row
//     block's token rows then started tens of microseconds apart and re-read them from DRAM
//     (gate/up moved 1.5x its algorithmic bytes; 1.02x with ids taken just in time).
constexpr int kTileSlots = 4;
constexpr int kClaimAhead = 8;
constexpr int kPublishAfter = 4;

__device__ __forceinline__ int claim_tile(uint32_t *sched) { return (int)min(atomicAdd(sched, 1u), 0x7fffffffu); }

// Publish the k-th tile id in both CTAs' rings (even CTA); false when a wait gave up.
__device__ __forceinline__ bool publish_tile(uint32_t k, int tile, int32_t *ring, uint64_t *full, uint64_t *empty,
                                             volatile int *abort_v, uint32_t *status) {
    const int slot = (int)(k % kTileSlots);
    const uint32_t ph = (k / kTileSlots) & 1;
    if (!wait_bar_cluster(smem_u32(&empty[slot]), ph ^ 1, abort_v, status)) return false;
    ring[slot] = tile;
    st_shared_cluster_u32(mapa_shared(smem_u32(&ring[slot]), 1), (uint32_t)tile);
    mbar_arrive(smem_u32(&full[slot]));                             // this CTA's readers
    mbar_arrive_cluster(mapa_shared(smem_u32(&full[slot]), 1));     // the odd CTA's readers
    return true;
}

// The scheduler thread's loop (one-region tiles): publish ids until one is past the list.
__device__ __forceinline__ void schedule_tiles(int total_tiles, int32_t *ring, uint64_t *full, uint64_t *empty,
                                               uint32_t *sched, volatile int *abort_v, uint32_t *status) {
    for (uint32_t k = 0;; ++k) {
        const int tile = claim_tile(sched);
        if (!publish_tile(k, tile, ring, full, empty, abort_v, status) || tile >= total_tiles) return;
    }
}

// A reader (one thread): the k-th tile id, after which its slot is released on the even CTA's
// barrier; -1 when a wait gave up.  Readers in the odd CTA acquire at cluster scope (the id was
// written from the even CTA).
__device__ __forceinline__ int read_tile(uint32_t k, int32_t *ring, uint64_t *full, uint64_t *empty, bool leader,
                                         volatile int *abort_v, uint32_t *status) {
    const int slot = (int)(k % kTileSlots);
    const uint32_t ph = (k / kTileSlots) & 1;
    const uint32_t f = smem_u32(&full[slot]);
    if (!(leader ? wait_bar(f, ph, abort_v, status) : wait_bar_cluster(f, ph, abort_v, status))) return -1;
    const int tile = *reinterpret_cast<volatile int32_t *>(&ring[slot]);
    const uint32_t e = smem_u32(&empty[slot]);
    if (leader) mbar_arrive(e);
    else mbar_arrive_cluster(mapa_shared(e, 0));
    return tile;
}

template <bool GLU, int NREG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<GLU, NREG>::threads, 1)
ffn_tc_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const Params p) {
    using C = PairCfg<GLU, NREG>;
    constexpr int kStages = C::stages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int32_t prefix[kMaxExperts + 1];
    __shared__ int32_t warp_sums[16];
    __shared__ int32_t seg_begin[kMaxExperts], seg_count[kMaxExperts];
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
    // accumulator barriers: NREG = 1, the two buffers used in turn; NREG = 2, the two regions
    __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ __align__(8) uint64_t tile_full[kTileSlots], tile_empty[kTileSlots];
    __shared__ int32_t tile_ring[kTileSlots];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), 8);  // 4 epilogue warps of each CTA
        }
        for (int i = 0; i < kTileSlots; ++i) {
            mbar_init(smem_u32(&tile_full[i]), 1);                 // the even CTA's publisher
            mbar_init(smem_u32(&tile_empty[i]), C::slot_readers);  // (the even CTA's barrier only)
        }
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b0);
        if (GLU) tma_prefetch_desc(&map_b1);
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(&tmem_base_slot), kPairTmemCols);
        tmem_relinquish_pair();
    }
    pdl_wait();  // the offsets (and the token rows) come from earlier kernels
    pdl_trigger();
    const int nfb = (p.out_dim + C::feat - 1) / C::feat;
    const bool last_has_two = NREG == 1 || (nfb - 1) * C::feat + C::region_feat < p.out_dim;
    build_prefix(p.offsets, p.N, p.rows, [nfb](int c) { return pair_blocks(c) * nfb; }, prefix, warp_sums,
                 seg_begin, seg_count);  // contains __syncthreads
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised and their TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;

    const int total_tiles = prefix[p.N];
    const int kblocks = (p.kdim + kBK - 1) / kBK;
    volatile int *abort_v = &abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (one thread per CTA)
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            int tile = 0;
            const bool claims = C::producer_claims && leader;  // else the ids come from the ring
            if (claims) {
                tile = claim_tile(p.sched);
                ok = publish_tile(0, tile, tile_ring, tile_full, tile_empty, abort_v, p.status);
            }
            const int claim_kb = kblocks > kClaimAhead ? kblocks - kClaimAhead : 0;
            const int publish_kb = min(claim_kb + kPublishAfter, kblocks - 1);
            for (uint32_t k = 0; ok; ++k) {
                if (!claims) tile = read_tile(k, tile_ring, tile_full, tile_empty, leader, abort_v, p.status);
                if (tile < 0 || tile >= total_tiles) break;
                int next = 0;
                const PairTile t = pair_tile(tile, prefix, seg_begin, seg_count, p.N, nfb, C::feat);
                const int nreg = (NREG == 2 && pair_tile_two_regions(tile, nfb, last_has_two)) ? 2 : 1;
                const int trow = t.row0 + (int)rank * kBM;                 // this CTA's 128 token rows
                const int wrow = t.f0 + (GLU ? 0 : (int)rank * kBM);       // and its weight rows
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    if (claims && kb == claim_kb) next = claim_tile(p.sched);
                    if (claims && kb == publish_kb &&
                        !publish_tile(k + 1, next, tile_ring, tile_full, tile_empty, abort_v, p.status)) {
                        ok = false;
                        break;
                    }
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!wait_bar(smem_u32(&empty_bar[s]), ph ^ 1, abort_v, p.status)) { ok = false; break; }
                    const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[s]), 0);
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * (1 + nreg) * kPairBlockBytes);
                    const uint32_t sa = smem_base + s * C::stage_bytes;
                    const int k0 = kb * kBK;
                    tma_load_2d_pair(sa, &map_a, full_leader, k0, trow);                      // token rows
                    for (int r = 0; r < nreg; ++r) {
                        const uint32_t sb = sa + (1 + r) * kPairBlockBytes;
                        const int wr = wrow + r * C::region_feat;
                        if (GLU && !leader) tma_load_3d_pair(sb, &map_b1, full_leader, k0, wr, t.e);  // W_up
                        else tma_load_3d_pair(sb, &map_b0, full_leader, k0, wr, t.e);            // W_gate / W_down
                    }
                }
                if (claims) tile = next;
            }
            // drain (even CTA): its full barriers also count the odd CTA's copies
            if (leader)
                for (uint32_t j = (it > (uint32_t)kStages ? it - kStages : 0); j < it; ++j)
                    drain_wait(smem_u32(&full_bar[j % kStages]), (j / kStages) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one thread, even CTA)
        // Per tile: wait until every accumulator the tile uses has been drained, issue the
        // k-blocks (each stage freed by a commit once its MMAs complete), then commit the
        // accumulators.  (Waiting for a drained accumulator only at the tile's first k-block, after
        // that stage's copies, or committing the accumulators before the last stage, measured
        // 8-17 % more time.)
        if (lane == 0 && leader) {
            uint32_t it = 0, n[2] = {0, 0};  // tiles issued so far into region 0 / region 1
            bool ok = true;
            for (uint32_t k = 0; ok; ++k) {
                const int tile = read_tile(k, tile_ring, tile_full, tile_empty, true, abort_v, p.status);
                if (tile < 0 || tile >= total_tiles) break;
                const int nreg = (NREG == 2 && pair_tile_two_regions(tile, nfb, last_has_two)) ? 2 : 1;
                // accumulator barrier of region r and its use count: one region, two buffers in
                // turn; or two regions, one buffer each
                int b[NREG];
                uint32_t u[NREG];
#pragma unroll
                for (int r = 0; r < NREG; ++r) {
                    b[r] = NREG == 1 ? (int)(n[0] & 1) : r;
                    u[r] = NREG == 1 ? n[0] >> 1 : n[r];
                }
#pragma unroll
                for (int r = 0; r < NREG; ++r)
                    if (r < nreg && !wait_bar(smem_u32(&tempty_bar[b[r]]), (u[r] & 1) ^ 1, abort_v, p.status)) ok = false;
                if (!ok) break;
                tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!wait_bar(smem_u32(&full_bar[s]), ph, abort_v, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_base + s * C::stage_bytes;
#pragma unroll
                    for (int r = 0; r < NREG; ++r) {
                        if (r >= nreg) break;
#pragma unroll
                        for (int j = 0; j < kBK / 16; ++j)
                            mma_bf16_pair(tmem_base + b[r] * 256, smem_desc_sw128(sa + j * 32),
                                          smem_desc_sw128(sa + (1 + r) * kPairBlockBytes + j * 32), kPairIdesc,
                                          (kb > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit_pair_mc(smem_u32(&empty_bar[s]), 0x3);  // frees the stage in both CTAs
                }
                if (!ok) break;
#pragma unroll
                for (int r = 0; r < NREG; ++r)
                    if (r < nreg) mma_commit_pair_mc(smem_u32(&tfull_bar[b[r]]), 0x3);  // accumulators ready
                ++n[0];
                if (nreg == 2) ++n[1];
            }
            mma_commit_pair(smem_u32(&drain_bar));
            drain_wait(smem_u32(&drain_bar), 0, p.status);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------ tile scheduler (one-region tiles: one thread, even CTA)
        if (!C::producer_claims && lane == 0 && leader)
            schedule_tiles(total_tiles, tile_ring, tile_full, tile_empty, p.sched, abort_v, p.status);
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------ epilogue (warps 4 .. 3 + epi_warps of each CTA)
        const int region = (warp - kEpiWarp0) >> 2;
        const int q = warp & 3;  // TMEM lane quarter
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        uint4 *stage = reinterpret_cast<uint4 *>(smem + kStages * C::stage_bytes) + (warp - kEpiWarp0) * 128;
        uint32_t n = 0;  // tiles this warp has drained
        for (uint32_t k = 0;; ++k) {
            int tile = 0;
            if (lane == 0) tile = read_tile(k, tile_ring, tile_full, tile_empty, leader, abort_v, p.status);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0 || tile >= total_tiles) break;
            if (region == 1 && !pair_tile_two_regions(tile, nfb, last_has_two)) continue;
            const int b = NREG == 1 ? (int)(n & 1) : region;
            const uint32_t u = NREG == 1 ? n >> 1 : n;
            bool ok = wait_bar(smem_u32(&tfull_bar[b]), u & 1, abort_v, p.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const PairTile t = pair_tile(tile, prefix, seg_begin, seg_count, p.N, nfb, C::feat);
            const int warp_row0 = (int)rank * kBM + q * 32;     // the warp's first row inside the 256-row tile
            const uint32_t t_acc = tmem_base + b * 256 + lane_addr;
            const int f_region = t.f0 + region * C::region_feat;
            constexpr int chunks = GLU ? 4 : 8;
#pragma unroll 1
            for (int c = 0; c < chunks; ++c) {
                uint32_t va[32];
                float o[32];
                tmem_ld_x32(t_acc + c * 32, va);
                if constexpr (GLU) {
                    uint32_t vu[32];
                    tmem_ld_x32(t_acc + 128 + c * 32, vu);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = swiglu_fast(__uint_as_float(va[j]), __uint_as_float(vu[j]));
                } else {
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(va[j]);
                }
                store_rows_staged(o, stage, lane, p.out, (int64_t)t.row0 + warp_row0, t.nrows - warp_row0,
                                  f_region + c * 32, p.out_dim);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(smem_u32(&tempty_bar[b]));
                else mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[b]), 0));
            }
            ++n;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the odd CTA's shared memory and TMEM stay live until the even CTA's MMAs end
    tc_fence_after();
    if (warp == 2) tmem_dealloc_pair(tmem_base, kPairTmemCols);
    // the last CTA to finish returns the tile counters to zero for the next launch (every CTA
    // has left its loops, so no tile is taken after this)
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Host side: tensor maps and launches
// ---------------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

// 2D row-major [rows, cols] bf16, box {64, box_rows}, 128-byte swizzle.
bool make_map_2d(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D row-major [n, rows, cols] bf16 (one matrix per expert), box {64, box_rows, 1}.
bool make_map_3d(CUtensorMap *m, const void *base, int64_t n, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)n};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(cols * rows * 2)};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

template <int MODE, int BNT, bool GATHER>
cudaError_t launch_mode(const CUtensorMap &ma, const CUtensorMap &mb0, const CUtensorMap &mb1, const Params &p,
                        int64_t tile_bound, cudaStream_t s) {
    using C = Cfg<MODE, BNT>;
    auto kern = ffn_tc_kernel<MODE, BNT, GATHER>;
    cudaError_t err = set_max_smem(kern, (int)C::smem_bytes);
    if (err != cudaSuccess) return err;
    const int grid = (int)std::min<int64_t>(tile_bound, (int64_t)sm_count());
    if (grid <= 0) return cudaSuccess;
    err = launch_pdl(kern, dim3(grid), dim3(kThreads), C::smem_bytes, s, ma, mb0, mb1, p);
    count_launches(1);
    return err;
}

template <bool GLU, int NREG>
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb0, const CUtensorMap &mb1, const Params &p,
                        int64_t pair_tile_bound, cudaStream_t s) {
    using C = PairCfg<GLU, NREG>;
    auto kern = ffn_tc_pair_kernel<GLU, NREG>;
    cudaError_t err = set_max_smem(kern, (int)C::smem);
    if (err != cudaSuccess) return err;
    const int grid = (int)std::min<int64_t>(2 * pair_tile_bound, (int64_t)(sm_count() & ~1));  // whole pairs
    if (grid <= 0) return cudaSuccess;
    err = launch_pdl(kern, dim3(grid), dim3(C::threads), C::smem, s, ma, mb0, mb1, p);
    count_launches(1);
    return err;
}

// Token rows of the gate/up GEMM: gathered from x [T, d] through row_token (one-row box), or
// read from the already permuted x_perm [P, d] (box of `rows` rows).
bool make_act_map(CUtensorMap *m, const void *act, const int32_t *row_token, int64_t T, int64_t P, int64_t d,
                  int rows) {
    return row_token ? make_map_2d(m, act, T, d, 1) : make_map_2d(m, act, P, d, rows);
}

// Weights-as-M tiles of BNT tokens for every expert (rule kBlocksAll: the batch's plan) or for
// the small experts only (kBlocksSmallExperts, beside a CTA-pair launch): gate/up + SwiGLU -> h,
// and down -> y_perm.
template <int BNT>
cudaError_t launch_swap_gate_up(const void *act, const int32_t *row_token, const int32_t *offsets, int64_t N,
                                int64_t P, int64_t T, int64_t d, int64_t I, const CUtensorMap &mg,
                                const CUtensorMap &mu, void *h, uint32_t *status, int rule, cudaStream_t s) {
    CUtensorMap mx;
    if (!make_act_map(&mx, act, row_token, T, P, d, BNT)) return cudaErrorInvalidValue;
    const int64_t tok_blocks = rule == kBlocksAll ? cdiv(P, BNT) + N : N * cdiv(kSmallExpertRows, BNT);
    Params p{offsets, (int)N, (int)d, (int)I, (__nv_bfloat16 *)h, status, row_token, rule, (int)P, nullptr};
    return row_token ? launch_mode<SWAP_GLU, BNT, true>(mx, mg, mu, p, tok_blocks * cdiv(I, 128), s)
                     : launch_mode<SWAP_GLU, BNT, false>(mx, mg, mu, p, tok_blocks * cdiv(I, 128), s);
}

template <int BNT>
cudaError_t launch_swap_down(const int32_t *offsets, int64_t N, int64_t P, int64_t d, int64_t I,
                             const CUtensorMap &mdn, const void *h, void *y_perm, uint32_t *status, int rule,
                             cudaStream_t s) {
    CUtensorMap mh;
    if (!make_map_2d(&mh, h, P, I, BNT)) return cudaErrorInvalidValue;
    const int64_t tok_blocks = rule == kBlocksAll ? cdiv(P, BNT) + N : N * cdiv(kSmallExpertRows, BNT);
    Params p{offsets, (int)N, (int)I, (int)d, (__nv_bfloat16 *)y_perm, status, nullptr, rule, (int)P, nullptr};
    return launch_mode<SWAP_PLAIN, BNT, false>(mh, mdn, mdn, p, tok_blocks * cdiv(d, 128), s);
}

template <int BNT>
cudaError_t launch_swap(const void *act, const int32_t *row_token, const int32_t *offsets, int64_t N, int64_t P,
                        int64_t T, int64_t d, int64_t I, const void *wg, const void *wu, const void *wd, void *h,
                        void *y_perm, uint32_t *status, cudaStream_t s) {
    CUtensorMap mg, mu, mdn;
    if (!make_map_3d(&mg, wg, N, I, d, kBM) || !make_map_3d(&mu, wu, N, I, d, kBM) ||
        !make_map_3d(&mdn, wd, N, d, I, kBM))
        return cudaErrorInvalidValue;
    cudaError_t err = launch_swap_gate_up<BNT>(act, row_token, offsets, N, P, T, d, I, mg, mu, h, status, kBlocksAll, s);
    if (err != cudaSuccess) return err;
    mark_stage(MOGE_STAGE_DOWN, s);
    return launch_swap_down<BNT>(offsets, N, P, d, I, mdn, h, y_perm, status, kBlocksAll, s);
}

}  // namespace tc

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime (no -lcuda link).
void *tensor_map_encoder() {
    static void *fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = ptr;
    });
    return fn;
}

cudaError_t launch_ffn_tc(const void *act, const int32_t *row_token, const int32_t *offsets, int64_t N, int64_t P,
                          int64_t T, int64_t d, int64_t I, const void *w_gate, const void *w_up, const void *w_down,
                          void *h, void *y_perm, uint32_t *status, cudaStream_t s) {
    using namespace tc;
    if (P == 0) return cudaSuccess;
    if (N > kMaxExperts) return cudaErrorInvalidValue;
    switch (ffn_plan(T, P, N).tiles) {
        case kTilesSwap16:
            return launch_swap<16>(act, row_token, offsets, N, P, T, d, I, w_gate, w_up, w_down, h, y_perm, status,
                                   s);
        case kTilesSwap32:
            return launch_swap<32>(act, row_token, offsets, N, P, T, d, I, w_gate, w_up, w_down, h, y_perm, status,
                                   s);
        case kTilesSwap64:
            return launch_swap<64>(act, row_token, offsets, N, P, T, d, I, w_gate, w_up, w_down, h, y_perm, status,
                                   s);
        case kTilesSwap128:
            return launch_swap<128>(act, row_token, offsets, N, P, T, d, I, w_gate, w_up, w_down, h, y_perm, status,
                                    s);
        default:
            break;
    }
    // Many tokens: the tile is chosen per expert from its row count, on the device.  Experts with
    // more than kSmallExpertRows rows take CTA-pair tokens-as-M tiles (their last block padded
    // to 256 rows: it runs while the expert's weights are still in L2); experts with fewer take
    // 32-token weights-as-M tiles in a single-CTA launch after it (padding a 256-row block for a
    // few tokens would cost up to 256/c times the expert's MMA work, and the weights-as-M tiles
    // stream the weights at nearly the HBM rate).  Rows are read from x_perm.
    if (row_token || !status) return cudaErrorInvalidValue;
    CUtensorMap mx, mh, mg, mu, mdn;
    if (!make_map_2d(&mx, act, P, d, kBM) || !make_map_2d(&mh, h, P, I, kBM) ||
        !make_map_3d(&mg, w_gate, N, I, d, kBM) || !make_map_3d(&mu, w_up, N, I, d, kBM) ||
        !make_map_3d(&mdn, w_down, N, d, I, kBM))
        return cudaErrorInvalidValue;
    // bound of the tile count: sum over experts of ceil(count_e / 256) blocks
    const int64_t pair_blocks = cdiv(P, kPairRows) + N;
    uint32_t *sched_gu = status + kSchedGateUpOffset / 4, *sched_dn = status + kSchedDownOffset / 4;
    Params p1{offsets, (int)N, (int)d, (int)I, (__nv_bfloat16 *)h, status, nullptr, kBlocksAll, (int)P, sched_gu};
    cudaError_t err = launch_pair<true, 2>(mx, mg, mu, p1, pair_blocks * cdiv(I, PairCfg<true, 2>::feat), s);
    if (err == cudaSuccess)
        err = launch_swap_gate_up<kSmallExpertTile>(act, nullptr, offsets, N, P, T, d, I, mg, mu, h, status,
                                                    kBlocksSmallExperts, s);
    if (err != cudaSuccess) return err;
    mark_stage(MOGE_STAGE_DOWN, s);
    Params p2{offsets, (int)N, (int)I, (int)d, (__nv_bfloat16 *)y_perm, status, nullptr, kBlocksAll, (int)P,
              sched_dn};
    err = launch_pair<false, 1>(mh, mdn, mdn, p2, pair_blocks * cdiv(d, PairCfg<false, 1>::feat), s);
    if (err != cudaSuccess) return err;
    return launch_swap_down<kSmallExpertTile>(offsets, N, P, d, I, mdn, h, y_perm, status, kBlocksSmallExperts, s);
}

}  // namespace moge
