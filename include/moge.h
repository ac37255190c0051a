/*
 * moge.h -- C ABI of the B300 (sm_103a) Mixture-of-Grouped-Experts layer forward.
 *
 * The layer ("Pangu Pro MoE: Mixture of Grouped Experts for Efficient
 * Sparsity", retold in the Pangu Pro MoE explainer, section 1 "innovative
 * architecture"): N experts are split evenly into M groups of G = N/M; each
 * token's router scores go through one softmax over all N experts; inside
 * every group exactly K' = K/M experts are selected, so every group (one
 * device in expert parallelism) receives the same load and the imbalance
 * score is zero.  Tokens are then permuted to their experts, each selected
 * expert runs a SwiGLU FFN as a grouped GEMM, and the expert outputs are
 * summed weighted by their gates.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Memory: every pointer argument is DEVICE memory owned by the caller
 *    (except `cfg`, which is host memory read during the call).  The library
 *    allocates, frees and synchronises nothing on these paths; scratch space
 *    is the caller's `ws` buffer of `ws_bytes` bytes, sized by
 *    moge_workspace_bytes().
 *  - Streams: all device work is enqueued on `stream` (0 = legacy default).
 *    A call returns once its work is enqueued.
 *  - Layouts (row-major, contiguous): x [T,d]; w_router [N,d];
 *    w_gate, w_up [N,I,d]; w_down [N,d,I]; logits [T,N];
 *    topk_idx, topk_gate, pair_row [T,K] with K = M*K'; counts [N];
 *    offsets [N+1]; row_token [P] with P = T*K; x_perm [P,d]; y_perm [P,d];
 *    y [T,d]; group_load [M]; score: one float.
 *  - Element types: activations (x, x_perm, y_perm, y) and weights (w_*)
 *    have the configuration's dtype (fp32, or bf16 as raw 16-bit values);
 *    bias, logits, gates and score are fp32; indices and counts are int32.
 *  - Alignment: device pointers must be 16-byte aligned (MOGE_ERR_INVALID_ARGUMENT
 *    otherwise); the workspace must be 256-byte aligned.
 *  - Errors: argument checks run on the host before anything is launched;
 *    a rejected call leaves every output untouched.  Inputs must be finite
 *    (non-finite values are a precondition violation, not detected).
 *    Every bounded wait inside a kernel that gives up records
 *    MOGE_ERR_TIMEOUT in the workspace status word instead of hanging; read
 *    it with moge_query_device_status().
 *  - Determinism: every output is bit-reproducible for identical inputs and
 *    configuration (no floating-point atomics; fixed summation orders).
 *  - CUDA graphs: the layer calls synchronise nothing, allocate nothing and
 *    read nothing back to the host, so they can be captured into a graph and
 *    replayed.  The first call on a device sets kernel attributes and looks up
 *    a driver entry point; make one call of the same kind before capturing.
 *    moge_permute_noalloc's first call in a context also looks up the address
 *    of its static scratch array (see there).
 *  - Concurrency: all per-call state lives in the caller's workspace; calls
 *    on different streams need different workspaces.  The one exception is
 *    moge_permute_noalloc, whose scratch is a single array inside the library
 *    shared by all its calls: order those calls on one stream or synchronise
 *    between them.
 */
#ifndef MOGE_H
#define MOGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOGE_ABI_VERSION 1

typedef struct CUstream_st *moge_stream_t; /* same handle as cudaStream_t */

typedef enum {
    MOGE_OK = 0,
    MOGE_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad shape, N % M != 0, K' outside [1, N/M], misalignment */
    MOGE_ERR_UNSUPPORTED = 2,      /* dtype/shape combination the library does not handle */
    MOGE_ERR_WORKSPACE = 3,        /* ws is NULL or ws_bytes < moge_workspace_bytes(cfg) */
    MOGE_ERR_CUDA = 4,             /* a CUDA runtime call or kernel launch failed */
    MOGE_ERR_TIMEOUT = 5           /* a bounded device-side wait gave up (see moge_query_device_status) */
} moge_status_t;

typedef enum { MOGE_F32 = 0, MOGE_BF16 = 1 } moge_dtype_t;

typedef enum {
    MOGE_ROUTE_GROUPED = 0,    /* MoGE: top-K' inside each of the M groups */
    MOGE_ROUTE_GLOBAL_TOPK = 1 /* conventional MoE: top-K (K = M*K') over all N experts */
} moge_route_mode_t;

/* Layer shape.  T tokens, hidden size d, N experts in M groups, K' =
 * k_per_group experts chosen per group, expert FFN intermediate size I.
 * act_dtype and weight_dtype must be equal: F32 (all-fp32 path, CUDA-core FMA)
 * or BF16 (tensor-core path, fp32 accumulation). */
typedef struct {
    int64_t T, d, N, M, k_per_group, I;
    int32_t act_dtype;
    int32_t weight_dtype;
} moge_config_t;

/* Optional device outputs of moge_layer_forward; any field may be NULL. */
typedef struct {
    float *logits;      /* [T,N] router scores (fp32) */
    int32_t *topk_idx;  /* [T,K] */
    float *topk_gate;   /* [T,K] */
    int32_t *counts;    /* [N] */
    int32_t *offsets;   /* [N+1] */
    int32_t *group_load;/* [M] */
    float *score;       /* imbalance score, one float */
} moge_aux_t;

/* ABI version of the loaded library (MOGE_ABI_VERSION at build time). */
int moge_abi_version(void);

/* Static text for a status code. */
const char *moge_status_string(moge_status_t s);

/* Bytes of scratch needed by every call below for this configuration
 * (0 when cfg is invalid).  One workspace may serve all calls of a layer in
 * stream order (calls on different streams need different workspaces).  The
 * first 4096 bytes (the status page) hold the device status word, the
 * self-resetting per-tile counters of the router and the tile counters of the
 * grouped GEMM (each launch returns them to zero); they must be zero before
 * first use (see moge_reset_device_status). */
size_t moge_workspace_bytes(const moge_config_t *cfg);

/* Zero the 4096-byte status page at the start of ws (enqueued on stream). */
moge_status_t moge_reset_device_status(void *ws, moge_stream_t stream);

/* Synchronise `stream`, then read the status word at the start of ws:
 * MOGE_OK, or MOGE_ERR_TIMEOUT if a bounded device wait gave up since the
 * last reset, or MOGE_ERR_CUDA if the read itself failed. */
moge_status_t moge_query_device_status(const void *ws, moge_stream_t stream);

/* Routing: router scores -> global softmax -> selection.
 * Defined by the Pangu Pro MoE explainer, section 1: scores for all N
 * experts, one softmax over all of them, then top-K' inside each group
 * (MOGE_ROUTE_GROUPED) or, for the conventional MoE it is compared with,
 * top-K over all experts (MOGE_ROUTE_GLOBAL_TOPK).
 *   x        [T,d] or NULL.  If NULL, `logits` is the INPUT [T,N] fp32.
 *   w_router [N,d] (ignored when x is NULL); bias [N] fp32 or NULL, added to
 *            the scores before the softmax.
 *   logits   [T,N] fp32: input when x is NULL, else an optional output (NULL
 *            to skip).
 *   topk_idx [T,K] out: expert ids.  GROUPED: slot g*K'+r holds the r-th best
 *            expert of group g (groups are the contiguous ranges [gG,(g+1)G)).
 *            GLOBAL_TOPK: slot r holds the r-th best expert overall.
 *            "Best" compares fp32 scores; equal scores go to the lower index.
 *   topk_gate[T,K] out: the global softmax probability of each selected
 *            expert (not renormalised over the selection).
 * Needs ws (moge_workspace_bytes). */
moge_status_t moge_route(const moge_config_t *cfg, moge_route_mode_t mode, const void *x,
                         const void *w_router, const float *bias, float *logits, int32_t *topk_idx,
                         float *topk_gate, void *ws, size_t ws_bytes, moge_stream_t stream);

/* Permutation of the T*K (token, slot) pairs into expert-contiguous rows
 * (histogram + prefix sum + deterministic scatter).  Works for either
 * routing mode: it only needs every token's K experts to be distinct ids in
 * [0,N) (an id outside that range is skipped and sets no output row).
 *   counts[e]     = number of pairs routed to expert e
 *   offsets[e]    = counts[0] + ... + counts[e-1];  offsets[N] = P
 *   pair_row[t,k] = offsets[e] + #{t' < t routed to e}, e = topk_idx[t,k]
 *   row_token[r]  = token of row r
 *   x_perm[r,:]   = x[row_token[r],:]   (skipped when x or x_perm is NULL)
 * row_token and pair_row may be NULL when not wanted, except that x_perm needs
 * row_token.  With pair_row given the copy runs token by token (each row of x
 * is read once and stored to the rows of its pairs); without it, row by row
 * through row_token.  Rows r >= offsets[N] of x_perm are not written. */
moge_status_t moge_permute(const moge_config_t *cfg, const int32_t *topk_idx, const void *x,
                           int32_t *counts, int32_t *offsets, int32_t *pair_row, int32_t *row_token,
                           void *x_perm, void *ws, size_t ws_bytes, moge_stream_t stream);

/* moge_permute without a workspace.  The method has no counterpart: this entry
 * point exists for callers that cannot allocate device memory (a serving
 * runtime whose pool already owns all of HBM and hands a plugin only its input
 * and output buffers, or a latency-critical loop that must not call cudaMalloc,
 * which can synchronise the device).  Arguments, outputs, checks and errors
 * are those of moge_permute minus ws/ws_bytes.
 *   Scratch: a static device array of 256 KiB inside the library (held by every
 *   GPU that loads it until the process exits), enough for
 *   ceil(T/256) * N <= 65536 (e.g. T <= 16384 with N <= 256); larger problems
 *   return MOGE_ERR_UNSUPPORTED before anything is launched.
 *   The first call in each CUDA context (normally a device's primary context)
 *   looks up the array's device address in that context (cudaGetSymbolAddress)
 *   and remembers it for the context; make that first call before any stream
 *   capture.  After cudaDeviceReset the remembered address belongs to a context
 *   that no longer exists: do not call this entry point in that process again.
 *   All calls share the array and it keeps the last call's contents (nothing in
 *   it needs to start at zero): calls that overlap on the GPU race, so order
 *   them on one stream or synchronise between them.
 *   This call allocates nothing (no cudaMalloc, cudaFree or allocating library
 *   routine).  An out-of-range expert id is skipped (its pair_row is -1) but,
 *   having no workspace, is not reported through a status word. */
moge_status_t moge_permute_noalloc(const moge_config_t *cfg, const int32_t *topk_idx, const void *x,
                                   int32_t *counts, int32_t *offsets, int32_t *pair_row, int32_t *row_token,
                                   void *x_perm, moge_stream_t stream);

/* Grouped expert FFN over the permuted rows (SwiGLU; bf16 on tcgen05 tensor
 * cores with TMEM accumulators, fp32 on CUDA cores).  For every expert e and
 * row r in [offsets[e], offsets[e+1]):
 *   h[r,:]      = silu(x_perm[r,:] W_gate[e]^T) * (x_perm[r,:] W_up[e]^T)
 *   y_perm[r,:] = h[r,:] W_down[e]^T
 * with fp32 accumulation; for bf16, h is rounded to bf16 before the down
 * projection and y_perm is bf16.  `offsets` is read on the device only; it
 * should hold 0 <= offsets[0] <= ... <= offsets[N] <= P (P = T*K), as
 * moge_permute writes it.  Segments outside [0, P) are clamped to it, so no
 * offsets make the call touch a row outside x_perm, h or y_perm; rows that no
 * segment covers are left unwritten.
 * Needs ws (h lives there). */
moge_status_t moge_expert_ffn(const moge_config_t *cfg, const void *x_perm, const int32_t *offsets,
                              const void *w_gate, const void *w_up, const void *w_down, void *y_perm,
                              void *ws, size_t ws_bytes, moge_stream_t stream);

/* Weighted combine in fixed slot order with fp32 accumulation:
 *   y[t,:] = sum_{k=0..K-1} topk_gate[t,k] * y_perm[pair_row[t,k],:]
 * rounded once to the activation dtype.  A pair_row entry outside [0, T*K)
 * (moge_permute writes -1 for a skipped expert id) is an absent slot. */
moge_status_t moge_combine(const moge_config_t *cfg, const void *y_perm, const int32_t *pair_row,
                           const float *topk_gate, void *y, moge_stream_t stream);

/* Imbalance score (Pangu Pro MoE explainer, section 1: load of the busiest
 * device minus load of the idlest over a batch; one group = one device),
 * normalised by the token count:
 *   group_load[g] = sum of counts[e] over e in [gG,(g+1)G)
 *   score         = (max_g group_load[g] - min_g group_load[g]) / T   (fp32 division)
 * group_load may be NULL. */
moge_status_t moge_imbalance_score(const moge_config_t *cfg, const int32_t *counts,
                                   int32_t *group_load, float *score, moge_stream_t stream);

/* The whole layer: moge_route(GROUPED) -> moge_permute -> moge_expert_ffn ->
 * moge_combine, plus moge_imbalance_score when aux->score or aux->group_load
 * is set.  x [T,d] in, y [T,d] out; aux (or any of its fields) may be NULL. */
moge_status_t moge_layer_forward(const moge_config_t *cfg, const void *x, const void *w_router,
                                 const float *bias, const void *w_gate, const void *w_up,
                                 const void *w_down, void *y, const moge_aux_t *aux, void *ws,
                                 size_t ws_bytes, moge_stream_t stream);

/* The layer with S = n_shared shared experts in addition to the N routed ones
 * (the Pangu Pro MoE explainer, section 2 "hardware co-design", gives the model
 * 64 routed and 4 shared experts; the pages say no more about them).  Reading
 * taken: every token visits every shared expert, each a SwiGLU FFN of the same
 * shape as a routed expert, and their outputs are added with weight 1:
 *   y[t] = sum_k gate[t,k] FFN_{idx[t,k]}(x[t]) + sum_{s<S} FFN_{N+s}(x[t]).
 * w_gate, w_up [N+S,I,d] and w_down [N+S,d,I] hold the routed experts first and
 * the shared ones after them.  Routing, aux outputs (aux->offsets: the N+1
 * routed offsets) and errors are those of moge_layer_forward; 0 <= n_shared <= 64
 * and N + n_shared <= 1024.  Needs moge_workspace_bytes_shared(cfg, n_shared)
 * bytes of workspace (0 when cfg or n_shared is invalid). */
size_t moge_workspace_bytes_shared(const moge_config_t *cfg, int64_t n_shared);
moge_status_t moge_layer_forward_shared(const moge_config_t *cfg, int64_t n_shared, const void *x,
                                        const void *w_router, const float *bias, const void *w_gate,
                                        const void *w_up, const void *w_down, void *y, const moge_aux_t *aux,
                                        void *ws, size_t ws_bytes, moge_stream_t stream);

/* The layer (with S = n_shared >= 0 shared experts, as moge_layer_forward_shared)
 * added to a residual stream: the pages describe no residual; the reading taken
 * is the transformer block's, where the layer's output is added once per token,
 * unweighted, to the hidden state it was computed from:
 *   y[t] = residual[t] + sum_k gate[t,k] FFN_{idx[t,k]}(x[t]) + sum_{s<S} FFN_{N+s}(x[t]),
 * summed in fp32 (routed slots in slot order, then shared experts, then the
 * residual) and rounded once.  residual [T,d] has the activation dtype, is
 * 16-byte aligned and must not be NULL when T > 0; y may be the residual buffer
 * itself (in-place update of the residual stream) or any other [T,d] buffer.
 * Everything else (arguments, aux outputs, workspace size
 * moge_workspace_bytes_shared(cfg, n_shared), errors) is moge_layer_forward_shared's. */
moge_status_t moge_layer_forward_residual(const moge_config_t *cfg, int64_t n_shared, const void *x,
                                          const void *residual, const void *w_router, const float *bias,
                                          const void *w_gate, const void *w_up, const void *w_down, void *y,
                                          const moge_aux_t *aux, void *ws, size_t ws_bytes, moge_stream_t stream);

/* Monte-Carlo study of the imbalance score (Pangu Pro MoE explainer, section 1:
 * a Monte-Carlo simulation finds the imbalance score of conventional top-K
 * routing almost always above zero; MoGE's group top-K' keeps it at zero).
 * For every batch b in [0, batches) of cfg->T tokens and cfg->N experts the
 * call draws scores on the device,
 *   s[b,t,e] = z((b*T + t)*N + e) + bias[e]     (bias may be NULL = 0),
 * where z(i) is an Irwin-Hall approximation of N(0,1): the twelve 16-bit fields
 * u of the splitmix64 words mix(key + 3i), mix(key + 3i + 1), mix(key + 3i + 2),
 * key = mix(seed XOR 8), give z = sum (u + 1/2) / 2^16 - 6 (exact in fp32).
 * Each token is routed both ways on its fp32 scores (group top-K' as in
 * moge_route(MOGE_ROUTE_GROUPED), and top-K over all N with K = M*K'; ties go to
 * the lower index), and the groups of the selected experts are counted:
 *   loads_grouped[b*M + g], loads_global[b*M + g]   (int32, outputs, required)
 *   is_grouped[b], is_global[b] = (max_g load - min_g load) / T  (fp32, or NULL)
 * Only T, N, M and k_per_group of cfg are used; N <= 256.  Allocates nothing;
 * the load arrays are zeroed by the call.  Exact and reproducible (integer
 * counts). */
moge_status_t moge_imbalance_study(const moge_config_t *cfg, int64_t batches, uint64_t seed, const float *bias,
                                   int32_t *loads_grouped, int32_t *loads_global, float *is_grouped,
                                   float *is_global, moge_stream_t stream);

/* ---- Instrumentation (no counterpart on the pages: measurement support) ---- */

/* Stages of moge_layer_forward, in launch order. */
typedef enum {
    MOGE_STAGE_ROUTE = 0,     /* router projection + softmax + selection */
    MOGE_STAGE_PERMUTE = 1,   /* histogram + prefix sum + scatter */
    MOGE_STAGE_GATHER = 2,    /* x rows -> x_perm */
    MOGE_STAGE_GATE_UP = 3,   /* grouped GEMM with W_gate/W_up + SwiGLU -> h */
    MOGE_STAGE_DOWN = 4,      /* grouped GEMM with W_down -> y_perm */
    MOGE_STAGE_COMBINE = 5,   /* weighted combine -> y */
    MOGE_STAGE_IMBALANCE = 6, /* group loads + imbalance score (may be empty) */
    MOGE_NUM_STAGES = 7
} moge_stage_t;

/* Ask moge_layer_forward (on the calling host thread) to record events[i]
 * (cudaEvent_t handles owned by the caller) on its stream right before stage i
 * and events[MOGE_NUM_STAGES] after the last stage, so that
 * cudaEventElapsedTime(events[i], events[i+1]) is the device time of stage i.
 * n must be MOGE_NUM_STAGES + 1; a NULL entry skips that boundary (each
 * recorded event costs a few microseconds of device time, so time one stage
 * by setting only its two boundaries); events == NULL turns recording off.
 * The array is read at each call, so it must stay valid while recording is on. */
moge_status_t moge_set_stage_events(void *const *events, int n);

/* Failure-detection self-test (no counterpart on the pages): one small kernel
 * runs the bounded mbarrier wait used by the tensor-core kernels on barriers
 * that nothing completes.  One wait gives up after timeout_ns (1 ns .. 1 s),
 * raises the kernel's abort flag and records MOGE_ERR_TIMEOUT in the status
 * word of ws (read it with moge_query_device_status, clear it with
 * moge_reset_device_status); a second wait, with a longer limit, must leave
 * through the abort flag.  result (device, 16-byte aligned, 3 words) receives
 * {wait 1 succeeded, wait 2 succeeded, abort flag}: {0, 0, 1} when the
 * machinery works.  Nothing faults or hangs; the GPU stays usable. */
moge_status_t moge_selftest_bounded_wait(void *ws, uint64_t timeout_ns, uint32_t *result, moge_stream_t stream);

/* Number of kernels this library has launched since it was loaded (all host
 * threads).  Lets a caller count the device work behind a region of calls. */
uint64_t moge_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOGE_H */
