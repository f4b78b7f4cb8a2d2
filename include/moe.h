/*
 * moe.h -- C ABI of the single-GPU expert-parallel MoE layer forward (B300, sm_103a).
 *
 * The layer follows the four steps of an expert-parallel MoE layer as the Ultralytics
 * glossary page "Expert Parallelism" states them (section "How tokens move between
 * GPUs"): (1) a router scores every token against every expert and keeps the k best;
 * (2) each token's hidden state is sent to the partition that owns each chosen expert;
 * (3) every partition runs its local experts on the rows it received; (4) the outputs
 * return to their token, are weighted by the router scores and summed. The Hugging Face
 * "Expert parallelism" docs describe the same token-dispatch path (section "Token
 * dispatch") and the alternative masking + all-reduce rule ("ep_router" +
 * "moe_tp_experts", section "DistributedConfig").
 *
 * On one GPU the ep_size "ranks" are logical partitions of device memory: expert e
 * belongs to partition e / (E / ep_size) (Hugging Face page, "How the sizes combine");
 * the first all-to-all becomes the write into a send buffer grouped by expert (so each
 * partition's rows are contiguous), the second becomes the weighted un-permute.
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer owned by the caller unless stated
 *    otherwise; the library allocates no memory in any entry point and keeps no
 *    pointer after returning.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Work is enqueued asynchronously on it; no entry point synchronises the host,
 *    except moe_read_device_status.
 *  - Matrices are dense row-major. Element type of x, w_router, expert weights, send,
 *    out_slots and out is cfg->dtype (MOE_DTYPE_BF16 or MOE_DTYPE_FP32); router bias,
 *    routing weights and accumulation are fp32; indices are int32.
 *  - All arguments are validated before anything is enqueued (the Hugging Face page
 *    likewise rejects a bad plan "before anything is sharded"). On error nothing is
 *    launched and the call returns a status other than MOE_OK; moe_last_error() then
 *    gives a one-line reason (thread-local, valid until the next call on the thread).
 *  - num_tokens == 0 is valid and enqueues nothing.
 *  - Pointers to matrices must be 16-byte aligned; hidden and intermediate must be
 *    multiples of 8.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status_t {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad size, pointer, alignment, dtype or mode */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle (e.g. E>256) */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_size */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (see device status) */
} moe_status_t;

enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP32 = 1 };
enum { MOE_MODE_DISPATCH = 0, MOE_MODE_MASK_SUM = 1 };
/* Order in which a capacity limit ranks an expert's pairs (moe_config.capacity_priority). */
enum { MOE_PRIORITY_TOKEN = 0, MOE_PRIORITY_SLOT = 1 };

/* Device status word bits (moe_read_device_status). */
enum {
    MOE_DEV_OK = 0,
    MOE_DEV_TIMEOUT = 1,        /* a pipeline wait exceeded its limit; results invalid */
    MOE_DEV_BAD_EXPERT_ID = 2   /* a topk_idx entry outside [0, E); that pair was dropped */
};

/*
 * Sizes of one layer call. The argument list follows the pages' statement of the
 * problem: hidden states (num_tokens x hidden), a router over num_experts experts,
 * top_k experts per token (Ultralytics page, step 1: "usually one, two or eight"),
 * ep_size partitions that must divide num_experts (Hugging Face page, launch rules),
 * an optional capacity factor (Ultralytics page, "Load balancing and capacity") and
 * the dispatch-versus-mask-and-sum mode.
 *
 *  num_tokens       N >= 0
 *  hidden           H, multiple of 8
 *  intermediate     I, SwiGLU expert intermediate size, multiple of 8
 *  num_experts      E, 1..256
 *  top_k            k, 1..min(E, 32)
 *  ep_size          P, divides E
 *  capacity_factor  <= 0: no limit. Otherwise every expert keeps at most
 *                   C = ceil(capacity_factor * N * k / E) (token, expert) pairs, the
 *                   first C in token order; the rest contribute zero (no
 *                   renormalisation). NaN is rejected.
 *  mode             MOE_MODE_DISPATCH or MOE_MODE_MASK_SUM
 *  dtype            MOE_DTYPE_BF16 (tcgen05 tensor-core experts) or MOE_DTYPE_FP32
 *                   (fp32 FFMA experts)
 *  has_bias         1 if the router has a bias vector (fp32 [E])
 *
 * Routing variants (Ultralytics page, "Load balancing and capacity": DeepSeek-V3's
 * bias-based balancing and its limit on the nodes a token is sent to):
 *  group_limit      0: none. Otherwise each token's top_k experts are taken from at
 *                   most group_limit of the ep_size partitions: a partition scores the
 *                   best selection score of its experts, the group_limit best partitions
 *                   are kept (ties: lower partition id) and the top_k experts inside
 *                   them are chosen. Needs group_limit * (E / ep_size) >= top_k,
 *                   group_limit <= 8 and ep_size <= 64.
 *  selection_bias   NULL, or fp32 [E] device array added to the logits for choosing
 *                   experts only; the routing weights remain the softmax of the chosen
 *                   experts' own logits. moe_update_selection_bias adjusts it.
 *
 * Capacity priority (Ultralytics page, "Load balancing and capacity"; the order in which
 * an over-full expert keeps pairs is left open there):
 *  capacity_priority  MOE_PRIORITY_TOKEN (0): an expert's pairs are ranked by token
 *                   index. MOE_PRIORITY_SLOT (1), GShard-style: ranked slot-major --
 *                   every token's first choice before any token's second choice, then by
 *                   token -- so pair (t, j) has priority j*N + t. The rank decides which
 *                   pairs the capacity keeps and orders the rows of the expert's segment
 *                   in the send layout.
 *
 * Training:
 *  training         0: inference. 1: moe_layer_forward also keeps, in the workspace, what
 *                   moe_layer_backward needs (the routing, the send layout and the gate /
 *                   up pre-activations; the workspace grows accordingly), and copies the
 *                   routing arrays it keeps to any moe_diagnostics buffers given.
 *                   Both dtypes (bf16: tensor-core backward; fp32: FFMA backward).
 */
typedef struct moe_config {
    int64_t num_tokens;
    int64_t hidden;
    int64_t intermediate;
    int32_t num_experts;
    int32_t top_k;
    int32_t ep_size;
    float capacity_factor;
    int32_t mode;
    int32_t dtype;
    int32_t has_bias;
    int32_t group_limit;
    const float *selection_bias;
    int32_t capacity_priority;
    int32_t training;
} moe_config;

/* Stage boundaries recorded by moe_layer_forward when moe_diagnostics.stage_events is
 * set: event i is recorded on the stream just before stage i is enqueued, event
 * MOE_NUM_STAGES after the last one. */
enum {
    MOE_STAGE_ROUTE = 0,     /* router + top-k + softmax + segment histogram: 1 kernel */
    MOE_STAGE_SCAN = 1,      /* counts, offsets and the stable slot of every pair: 1 kernel */
    MOE_STAGE_ASSIGN = 2,    /* empty: the slots are assigned in MOE_STAGE_SCAN's kernel */
    MOE_STAGE_PERMUTE = 3,   /* hidden-state rows into the send buffer: 1 kernel */
    MOE_STAGE_GATE_UP = 4,   /* grouped GEMM gate/up + SwiGLU: 1 kernel */
    MOE_STAGE_DOWN = 5,      /* grouped GEMM down + weighted un-permute: 1 kernel */
    MOE_STAGE_COMBINE = 6,   /* slot sum or masked partials + partition sum: 1 kernel */
    MOE_NUM_STAGES = 7
};

/* Optional outputs of moe_layer_forward: every non-NULL pointer receives the same
 * array the corresponding step entry point would write. */
typedef struct moe_diagnostics {
    int32_t *topk_idx;        /* [N, k] */
    float *topk_w;            /* [N, k] */
    int32_t *routed_counts;   /* [E]    */
    int32_t *counts;          /* [E]    */
    int32_t *expert_offsets;  /* [E+1]  */
    int32_t *part_offsets;    /* [P+1]  */
    int32_t *perm;            /* [N*k]  (first expert_offsets[E] entries meaningful) */
    int32_t *slot_pos;        /* [N*k]  */
    /* NULL, or MOE_NUM_STAGES + 1 cudaEvent_t handles (created by the caller) to record
     * at the stage boundaries, for per-kernel timing on the caller's stream. */
    void *const *stage_events;
    /* NULL, or fp32 [N, E], 16-byte aligned: the router logits with the router bias
     * (without the selection bias), for moe_balance_stats. */
    float *router_logits;
} moe_diagnostics;

/* Human-readable name of a status code (static string). */
const char *moe_status_string(moe_status_t status);

/* Reason for the last non-OK status returned on the calling thread (static until the
 * next call on that thread; "" if none). */
const char *moe_last_error(void);

/* Bytes of device workspace that moe_layer_forward needs for `cfg`; the same size is
 * enough for every other entry point of the same cfg. Writes *bytes; returns
 * MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED for a config the library rejects.
 * The workspace must be 256-byte aligned. Its first 32 bytes hold the device status
 * word (moe_read_device_status): zero them once before the first call. */
moe_status_t moe_workspace_size(const moe_config *cfg, size_t *bytes);

/* Bytes of the packed gate/up weight buffer moe_pack_weights writes for `cfg`. */
moe_status_t moe_packed_gate_up_size(const moe_config *cfg, size_t *bytes);

/*
 * One-time weight preparation (not part of the timed forward). Interleaves each
 * expert's gate and up projections in blocks of 64 output rows, zero-padding I up to
 * a multiple of 128, so that the accumulator of one SM holds matching gate and up rows
 * for the fused SwiGLU.
 *   w_gate, w_up        [E, I, H] dtype (nn.Linear layout: out x in)
 *   w_gate_up_packed    [E, 2*Ipad, H] dtype, Ipad = ceil(I/128)*128; for block b,
 *                       rows 128b..128b+63 are gate rows 64b.., the next 64 are up rows
 */
moe_status_t moe_pack_weights(const moe_config *cfg, const void *w_gate, const void *w_up,
                              void *w_gate_up_packed, void *stream);

/*
 * Step 1 -- routing (Ultralytics page, "How tokens move between GPUs", step 1 and its
 * routing example: a linear router, top-k of the raw logits).
 *   x         [N, H] dtype
 *   w_router  [E, H] dtype (nn.Linear layout)
 *   b_router  [E] fp32, or NULL when cfg->has_bias == 0
 *   topk_idx  [N, k] int32 out: chosen experts, descending logit, ties to lower id
 *   topk_w    [N, k] fp32 out: softmax over the k chosen logits
 * Logits are accumulated in fp32 and never written to memory.
 */
moe_status_t moe_route(const moe_config *cfg, const void *x, const void *w_router,
                       const float *b_router, int32_t *topk_idx, float *topk_w,
                       void *stream);

/*
 * After-step update of the selection bias (Ultralytics page, "Load balancing and
 * capacity": the bias of an overloaded expert is lowered and that of an idle expert
 * raised after each step). Overloaded / idle: routed_counts[e] above / below the equal
 * share num_tokens * top_k / num_experts (compared exactly, as integers); the step is
 * gamma: selection_bias[e] -= gamma or += gamma in fp32, unchanged at the share.
 *   routed_counts   [E] int32, the step's assignments per expert before capacity
 *                   (moe_dispatch's routed_counts)
 *   selection_bias  [E] fp32, updated in place
 * Both are device pointers owned by the caller. Enqueued on `stream`.
 */
moe_status_t moe_update_selection_bias(const moe_config *cfg, const int32_t *routed_counts,
                                       float *selection_bias, float gamma, void *stream);

/*
 * Step 2 -- dispatch (Hugging Face page, "Token dispatch": every (token, expert) pair
 * goes to the rank that owns the expert; Ultralytics page, step 2 and "Load balancing
 * and capacity"). Builds the send layout grouped by expert (hence by partition) and
 * copies each kept pair's hidden-state row into it. Pair p = t*k + j.
 *   topk_idx        [N, k] int32 in (ids outside [0,E) are dropped, see device status)
 *   x               [N, H] dtype in
 *   routed_counts   [E] out: pairs routed to each expert (before capacity)
 *   counts          [E] out: pairs kept
 *   expert_offsets  [E+1] out: exclusive prefix sum of counts
 *   part_offsets    [P+1] out: expert_offsets[p*E/P] (rows of partition p)
 *   perm            [N*k] out: perm[r] = pair held by send row r, r < expert_offsets[E]
 *   slot_pos        [N*k] out: send row of pair p, -1 if dropped
 *   send            [N*k, H] dtype out: send[r] = x[perm[r] / k]
 *   workspace       >= moe_workspace_size bytes (histograms)
 * Results are bit-exact and deterministic: within an expert, rows are in token order.
 */
moe_status_t moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                          int32_t *routed_counts, int32_t *counts, int32_t *expert_offsets,
                          int32_t *part_offsets, int32_t *perm, int32_t *slot_pos,
                          void *send, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * moe_dispatch without a workspace argument. The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory on their own -- code that
 * runs under an allocator that owns all device memory and hands out only the layer's
 * inputs and outputs, and therefore cannot provide moe_dispatch's workspace. (It makes
 * CUDA calls, so like every entry point here it must not be called from a host function
 * enqueued on a stream.)
 *
 * Same arguments, results and errors as moe_dispatch, minus workspace and its size. The
 * per-segment histograms live instead in a fixed array of device memory inside the
 * library (1 MiB, plus 256 bytes for a status word), which every GPU that
 * loads the library keeps until the process exits. Limit: segments * num_experts must
 * not exceed 262144, where segments = ceil(num_tokens / 64) in token-order capacity
 * priority and top_k * ceil(num_tokens / (64 * top_k)) in slot-major priority (for
 * example 65536 tokens with 256 experts in token order); larger calls return
 * MOE_ERR_UNSUPPORTED and enqueue nothing.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *  - The first call on a device looks up the array's device address on that device
 *    (cudaGetSymbolAddress, with that device current); make that first call before
 *    any stream capture. The address is kept for the life of the process, so the
 *    device must not be reset (cudaDeviceReset) nor its primary context destroyed
 *    while the library is in use.
 *  - All calls share the one array: calls whose work overlaps on the GPU (on different
 *    streams, or from different threads) race and corrupt each other's results. Order
 *    them on one stream or synchronise between them.
 *  - Pairs with an expert id outside [0, E) are dropped, as in moe_dispatch; this entry
 *    point does not report them.
 */
moe_status_t moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                                  int32_t *routed_counts, int32_t *counts,
                                  int32_t *expert_offsets, int32_t *part_offsets, int32_t *perm,
                                  int32_t *slot_pos, void *send, void *stream);

/*
 * Step 3 -- local experts (Ultralytics page, step 3; Hugging Face page, "grouped_gemm"
 * rule: expert weights split along the expert dimension). For every expert e in
 * [expert_begin, expert_end) -- all experts, or one partition's range -- runs the
 * SwiGLU FFN y = W_down (silu(W_gate x) * (W_up x)) on send rows
 * [expert_offsets[e], expert_offsets[e+1]) as a grouped GEMM, and writes the weighted
 * un-permuted result out_slots[perm[r]] = topk_w[perm[r]] * y_r (the return all-to-all
 * fused into the epilogue). Rows of other experts and dropped pairs are not written.
 *   send              [N*k, H] dtype
 *   expert_offsets    [E+1] int32
 *   w_gate_up_packed  from moe_pack_weights
 *   w_down            [E, H, I] dtype
 *   perm, topk_w      as written by moe_dispatch / moe_route
 *   out_slots         [N*k, H] dtype out (row = pair id)
 */
moe_status_t moe_expert_ffn(const moe_config *cfg, const void *send,
                            const int32_t *expert_offsets, int32_t expert_begin,
                            int32_t expert_end, const void *w_gate_up_packed,
                            const void *w_down, const int32_t *perm, const float *topk_w,
                            void *out_slots, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Step 4 -- combine (Ultralytics page, step 4: results weighted by the router scores
 * and summed at the token's origin).
 *   MOE_MODE_DISPATCH: out[t] = sum over kept slots j, in slot order, of
 *                      out_slots[t*k + j] (already weighted).
 *   MOE_MODE_MASK_SUM: every partition p first forms its masked partial output
 *                      partial_p[t] = sum of token t's kept slots whose expert lives in
 *                      p (fp32, in slot order), then out = partial_0 + ... +
 *                      partial_{P-1} in partition order (the all-reduce of the
 *                      "ep_router" + "moe_tp_experts" rule).
 *   out_slots  [N*k, H] dtype; topk_idx, slot_pos [N*k] int32; out [N, H] dtype.
 * A token whose pairs were all dropped gets a zero row.
 */
moe_status_t moe_combine(const moe_config *cfg, const void *out_slots,
                         const int32_t *topk_idx, const int32_t *slot_pos, void *out,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * The whole layer: route -> dispatch -> local experts -> combine, enqueued on `stream`
 * with no host synchronisation. Intermediates live in `workspace`; `diag` (may be
 * NULL) selects which of them are also written to caller buffers. Both modes run all
 * partitions' experts in one launch per GEMM (an expert's outputs do not depend on
 * which launch computes them); they differ in the combine.
 *   x [N,H], w_router [E,H], b_router [E] or NULL, w_gate_up_packed, w_down [E,H,I],
 *   out [N,H] dtype.
 */
moe_status_t moe_layer_forward(const moe_config *cfg, const void *x, const void *w_router,
                               const float *b_router, const void *w_gate_up_packed,
                               const void *w_down, void *out, const moe_diagnostics *diag,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, reads the device status word kept in `workspace` (an OR of
 * MOE_DEV_* bits accumulated since the last reset) into *flags, and clears it when
 * `reset` != 0. Returns MOE_ERR_TIMEOUT if MOE_DEV_TIMEOUT is set.
 */
moe_status_t moe_read_device_status(const moe_config *cfg, void *workspace,
                                    size_t workspace_bytes, int32_t *flags, int32_t reset,
                                    void *stream);

/*
 * Backward of the whole layer (the chain rule through moe_layer_forward; an expert's
 * weight gradient sums over every row it received -- Hugging Face page, "How the sizes
 * combine"). Call it after moe_layer_forward with the same cfg (training = 1), inputs
 * and workspace, on the same stream; the forward's state in the workspace must not be
 * overwritten in between.
 *   dout       [N, H] dtype     gradient of the layer output
 *   dx         [N, H] dtype out (expert paths plus the router's)
 *   dw_router  [E, H] fp32 out
 *   db_router  [E] fp32 out, or NULL
 *   dw_gate, dw_up [E, I, H] dtype out; dw_down [E, H, I] dtype out (nn.Linear layouts)
 * The expert selection and the capacity drops are piecewise constant and carry no
 * gradient; a dropped pair contributes no expert gradient but its routing weight still
 * gets a logit gradient through the softmax. All products accumulate in fp32; the
 * experts' weight gradients are one fp32 sum per expert over its rows, rounded once.
 * Deterministic: no atomics on values.
 */
moe_status_t moe_layer_backward(const moe_config *cfg, const void *x, const void *w_router,
                                const void *w_gate_up_packed, const void *w_down,
                                const void *dout, void *dx, float *dw_router, float *db_router,
                                void *dw_gate, void *dw_up, void *dw_down, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Router load statistics (Ultralytics page, "Load balancing and capacity": an auxiliary
 * loss term encourages the router to spread tokens evenly; the page gives no formula,
 * so this computes the two per-expert quantities such a term is built from, not a
 * loss):
 *   load_frac[e] = routed_counts[e] / (N * k)    share of the step's routed pairs
 *   prob_mean[e] = mean over the N tokens of softmax(router_logits[t])[e]
 *   router_logits  [N, E] fp32 (moe_diagnostics.router_logits of moe_layer_forward)
 *   routed_counts  [E] int32 (before capacity)
 *   load_frac, prob_mean  [E] fp32 out
 * Deterministic (fixed summation order). N = 0 gives zeros. Uses the workspace.
 */
moe_status_t moe_balance_stats(const moe_config *cfg, const float *router_logits,
                               const int32_t *routed_counts, float *load_frac, float *prob_mean,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * TP row split (Hugging Face page, "With tensor parallelism"): the tp_size ranks of a TP
 * group hold the same batch; each dispatches a disjoint slice of its tokens, and an
 * all-reduce over the group of the zero-padded slice outputs restores the full output.
 *
 * moe_tp_slice: the token rows [*begin, *end) of rank tp_rank: contiguous slices, the
 * first num_tokens mod tp_size ranks one token longer; slices may be empty (for
 * example a single decode token with tp_size 2). Host only; enqueues nothing.
 *
 * moe_tp_reduce: out = padded[0] + padded[1] + ... + padded[tp_size-1] (fp32
 * accumulation in rank order, rounded once to dtype), the single-device stand-in for
 * the all-reduce. padded is [tp_size, N, H] dtype, slice s's output at its rows and
 * zeros elsewhere (each slice is one moe_layer_forward over its rows, whose output
 * pointer is padded + (s*N + begin_s)*H); out is [N, H] dtype. Both 16-byte aligned.
 */
moe_status_t moe_tp_slice(int64_t num_tokens, int32_t tp_size, int32_t tp_rank, int64_t *begin,
                          int64_t *end);
moe_status_t moe_tp_reduce(const moe_config *cfg, int32_t tp_size, const void *padded, void *out,
                           void *stream);

/*
 * Check of the device-side failure path (not part of the layer): enqueues one warp that
 * waits, with the bounded mbarrier wait every tensor-core kernel of the library uses, on
 * a barrier that nothing arrives at. After the wait limit (about 2 s) it records
 * MOE_DEV_TIMEOUT in the workspace's status word and returns; no fault or trap is
 * involved and the context stays usable. moe_read_device_status then reports
 * MOE_ERR_TIMEOUT (and clears the word when asked to).
 */
moe_status_t moe_check_wait_timeout(const moe_config *cfg, void *workspace,
                                   size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
