/*
 * moe_dispatch.h -- C ABI of the GB300 (sm_103a) MoE token dispatch/combine
 * library, libmoe_gb300.so.
 *
 * The problem, as the pages state it: every token of a data-parallel group
 * goes to its top-K experts; a dispatch step moves each token's hidden row
 * into contiguous per-expert buffers that feed the grouped expert GEMM, and a
 * combine step returns the experts' outputs to the token and forms their
 * router-weighted sum ("Efficient and portable mixture-of-experts
 * communication", Introduction, Portable Kernels, Dispatch, Combine).  Here
 * the R "ranks" are logical partitions of one GPU's HBM: rank r owns tokens
 * [r*T, (r+1)*T) of every token-indexed array.  No call talks to another GPU.
 *
 * Notation: R ranks, T tokens per rank, N = R*T, H hidden size, E experts,
 * K experts per token, cap rows per expert in the padded buffers, global
 * token id g = r*T + t, routed entry (g, k).  All arrays are row-major.
 *
 * Conventions shared by every entry point
 *  - Pointers: every array is caller-owned DEVICE memory on the current
 *    device, unless stated otherwise.  The library allocates no memory and
 *    keeps no global state; everything that persists lives in the caller's
 *    workspace.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Every call only enqueues work on `stream` and returns
 *    without waiting for the device, except moe_read_status.  Calls are
 *    therefore usable inside CUDA-graph capture.
 *  - One workspace must not be used by two calls that may run at the same
 *    time (different streams without ordering).
 *  - Errors: argument errors are detected on the host and returned at once,
 *    with nothing enqueued.  Errors that depend on the data (an expert id out
 *    of range, more rows for an expert than `cap`, a wait that timed out) are
 *    found by the plan kernel and stored in the workspace status word; the
 *    dispatch and combine kernels read it first and write nothing when it is
 *    set.  moe_read_status returns it.
 */
#ifndef MOE_DISPATCH_H
#define MOE_DISPATCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, size overflow */
  MOE_ERR_UNSUPPORTED = 2,  /* shape outside the supported limits (below) */
  MOE_ERR_ALIGNMENT = 3,    /* a pointer is not aligned as required */
  MOE_ERR_BAD_EXPERT = 4,   /* device: some topk_idx outside [0, E) */
  MOE_ERR_CAPACITY = 5,     /* device: some expert receives more than cap rows */
  MOE_ERR_TIMEOUT = 6,      /* device: a wait between thread blocks ran out */
  MOE_ERR_CUDA = 7,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_WORKSPACE = 8     /* workspace missing or smaller than required */
} moe_status;

typedef enum {
  MOE_PAYLOAD_BF16 = 0,     /* expert_x rows are bf16 copies of x */
  MOE_PAYLOAD_FP8_E4M3 = 1, /* expert_x rows are OCP E4M3 bytes + fp32 scales [E, cap, nb],
                               nb = ceil(H / 128) */
  MOE_PAYLOAD_FP8_E4M3_TSCALE = 2  /* the same bytes; the scales transposed per expert,
                                      [E, nb, cap], as a grouped GEMM loads them: the
                                      scales of one 128-column block of one expert's rows
                                      are contiguous.  Every scale is then a separate
                                      4-byte store: slower than FP8_E4M3 */
} moe_payload;

/* Problem shape.  Limits: all sizes >= 1 except T, which may be 0 (an empty
 * batch: moe_plan writes zero counts and offsets, dispatch and combine do
 * nothing); K <= 32; E <= 2048; N*K < 2^31; E*cap < 2^31; H % 8 == 0
 * (H % 16 == 0 for the fp8 payloads, whose last 128-element scale block is
 * short when H % 128 != 0: "Lower latency and higher throughput with
 * multi-node DeepSeek deployment", Quantization, scale shape
 * M x ceil_div(K, 128)). */
typedef struct {
  int32_t num_ranks;        /* R */
  int32_t tokens_per_rank;  /* T */
  int32_t hidden;           /* H */
  int32_t num_experts;      /* E */
  int32_t top_k;            /* K */
  int32_t capacity;         /* cap: rows per expert in expert_x / expert_y */
  int32_t payload;          /* a moe_payload value */
} moe_shape;

/* Bytes of workspace the calls need for this shape (host only, no CUDA
 * call).  Returns 0 when the shape is invalid or unsupported. */
size_t moe_workspace_size(const moe_shape *shape);

/* Zero a workspace before its first use (enqueued on `stream`).  After
 * that the workspace keeps its counters consistent by itself, across shapes
 * and across calls that reported an error (the last thread block of every
 * moe_plan resets them).  A zero-filled allocation is already initialised.
 * Errors: INVALID_ARG (null), ALIGNMENT (not 16-byte aligned), CUDA. */
moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* Plan: per-expert counts, per-rank offsets and stable slots.
 *
 * Follows "Efficient and portable mixture-of-experts communication",
 * Dispatch (the sender counts the tokens each expert receives; the receiver
 * records source rank, expert and token index so combine can send each row
 * back) and "Enabling trillion-parameter models on AWS EFA", Send and Receive
 * Buffers / Dispatch and Combine (counts are known before any row is
 * written; a cumulative sum of per-expert counts gives every sender its
 * offset in the receiver's contiguous buffer).  The pages' receivers place
 * rows in arrival order; here the order is stable by (rank, token, k).
 *
 * In:   topk_idx            [N, K] int32, expert of routed entry (g, k)
 * Out:  expert_num_tokens   [E] int32:   count[e] = #{(g,k): idx = e}
 *       expert_rank_offsets [E, R+1] int32: entry r = #{(g,k): idx = e, g < r*T};
 *                           entry R = count[e]
 *       slot_of             [N, K] int32: row of (g,k) inside its expert's
 *                           buffer = #{(g',k') before (g,k) with the same expert}
 *       src_of              [E, cap] int32: src_of[e][slot_of[g,k]] = g*K + k;
 *                           only rows [0, min(count, cap)) are written
 * Work: `workspace` of at least moe_workspace_size(shape) bytes, 16-byte
 *       aligned, initialised once by moe_workspace_init.
 * Device errors (status word): BAD_EXPERT (outputs unspecified), CAPACITY
 *       (counts, offsets and slot_of are exact; src_of rows stop at cap),
 *       TIMEOUT.  The status word is replaced by each moe_plan call.
 * Host errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT (int32 arrays need 4-byte
 *       alignment), WORKSPACE, CUDA. */
moe_status moe_plan(const moe_shape *shape, const int32_t *topk_idx,
                    int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                    int32_t *slot_of, int32_t *src_of,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Plan for ragged ranks and masked routing.
 *
 * Follows "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", CUDA Graph (data-parallel groups run different batch sizes,
 * without padding every group to the largest) and "Efficient and portable
 * mixture-of-experts communication", Portable Kernels (a fixed maximum
 * number of tokens per group, here T).
 *
 * As moe_plan, except that entry (g, k) of token g = r*T + t is routed only
 * if t < clamp(num_tokens[r], 0, T) and topk_idx[g,k] != -1.  Unrouted
 * entries are not counted, get slot_of = -1, and are skipped by moe_dispatch
 * and moe_combine; ids of tokens beyond num_tokens[r] are never read.  A
 * token with no routed entry combines to y = +0.
 * In:   num_tokens [R] int32 device array (4-byte aligned), or NULL for all T.
 * Errors: as moe_plan (a routed id outside [0, E) is BAD_EXPERT). */
moe_status moe_plan_masked(const moe_shape *shape, const int32_t *topk_idx,
                           const int32_t *num_tokens, int32_t *expert_num_tokens,
                           int32_t *expert_rank_offsets, int32_t *slot_of, int32_t *src_of,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Dispatch: write each token's row to every (expert, slot) it is routed to.
 *
 * Follows "Efficient and portable mixture-of-experts communication", Dispatch
 * (tokens with their block scales are packed and moved into contiguous
 * per-expert tensors for the grouped GEMM) and, for the fp8 payload, "Lower
 * latency and higher throughput with multi-node DeepSeek deployment",
 * Quantization (activations quantised on the fly, one scale per 128-element
 * vector from its absolute maximum).
 *
 * In:   x            [N, H] bf16, 16-byte aligned
 *       topk_idx     [N, K] int32, slot_of [N, K] int32 (from moe_plan)
 * Out:  expert_x     [E, cap, H]: bf16 (payload BF16) or E4M3 bytes (payload
 *                    FP8_E4M3), 16-byte aligned.  Row (e, s) is written only
 *                    for s < count[e]; other rows are not touched.
 *       expert_x_scale [E, cap, nb] fp32 for FP8_E4M3, [E, nb, cap] for
 *                    FP8_E4M3_TSCALE (4-byte aligned), NULL for BF16;
 *                    nb = ceil(H / 128), the last block holding the H % 128
 *                    leftover elements when H is not a multiple of 128.  Per
 *                    block: scale = amax / 448,
 *                    q = e4m3_rn_satfinite(x / scale); an all-zero block has
 *                    scale 0 and q = 0.
 * Work: the workspace moe_plan used; the call writes nothing if its status
 *       word is set.  Requires moe_plan on the same topk_idx, ordered before
 *       this call.  An entry whose expert or slot is out of range is skipped
 *       and sets the status word (BAD_EXPERT / CAPACITY); an entry with
 *       slot_of = -1 (not routed, see moe_plan_masked) is skipped silently.
 * Ordering: the kernel is launched as a programmatic dependent of the
 *       previous kernel in the stream (normally moe_plan's), so its blocks
 *       may start before that kernel has completed; each waits for it to
 *       complete before its first read of any input, x included.  Any
 *       kernel may therefore produce x just before this call, even one that
 *       lets its dependents start early (griddepcontrol.launch_dependents).
 *       moe_dispatch_ex with MOE_DISPATCH_EARLY_X reads x sooner.
 * Host errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA. */
moe_status moe_dispatch(const moe_shape *shape, const void *x,
                        const int32_t *topk_idx, const int32_t *slot_of,
                        void *expert_x, float *expert_x_scale,
                        void *workspace, void *stream);

/* Flags of moe_dispatch_ex. */
enum {
  /* The caller asserts that x was final before the kernel that precedes this
   * call in the stream began: that kernel is moe_plan (an ordinary launch,
   * which starts only after every earlier kernel has completed, and which
   * never writes x) or another kernel that leaves x alone.  The dispatch
   * then loads (fp8: and quantises) the first rows of x while that kernel
   * is still finishing, and waits for it only before reading slot_of, the
   * routes and the status.  Without the assertion holding, rows may be
   * dispatched from stale x. */
  MOE_DISPATCH_EARLY_X = 1u
};

/* moe_dispatch with flags (0 = moe_dispatch).  Same inputs, outputs and
 * errors; an unknown flag bit is INVALID_ARG.  moe_plan_dispatch, when it
 * runs as two launches, dispatches this way after its own plan. */
moe_status moe_dispatch_ex(const moe_shape *shape, const void *x,
                           const int32_t *topk_idx, const int32_t *slot_of,
                           void *expert_x, float *expert_x_scale,
                           void *workspace, void *stream, uint32_t flags);

/* Plan and dispatch in one call: the outputs of moe_plan followed by
 * moe_dispatch, bit for bit, from a single kernel launch where the shape
 * allows it.
 *
 * Follows the passages of moe_plan and moe_dispatch.  At decode sizes the
 * plan is a short chain of dependent steps whose latency, plus the kernel
 * boundary, is a large part of plan + dispatch; here every thread block
 * finds the slots of its own tokens by reading the routing table itself, so
 * no block waits for another.  Taken when N*K <= 16384 and the block tables
 * fit in shared memory; other shapes (and T = 0) run moe_plan and
 * moe_dispatch, two launches, with the same results.
 * In:   x, topk_idx as moe_dispatch and moe_plan.
 * Out:  expert_num_tokens, expert_rank_offsets, slot_of, src_of as moe_plan;
 *       expert_x, expert_x_scale as moe_dispatch.
 * Work: as moe_plan (the status word is replaced by this call).
 * Device errors: the status word and the plan outputs are exactly those of
 *       moe_plan.  Unlike moe_dispatch, which writes nothing after a plan
 *       error, rows of entries whose expert is in range and whose slot is
 *       below cap may be written even when the status reports BAD_EXPERT or
 *       CAPACITY: no block waits for the others' outcome.
 * Ordering: the one-launch kernel is a programmatic dependent of the
 *       previous kernel in the stream: its blocks may be scheduled while
 *       that kernel drains, but they read nothing from global memory (x,
 *       topk_idx, the workspace) before it has completed.  The two-launch
 *       path is moe_plan, which waits for every earlier kernel, then
 *       moe_dispatch_ex(MOE_DISPATCH_EARLY_X), whose early read of x is
 *       therefore safe.
 * Host errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA. */
moe_status moe_plan_dispatch(const moe_shape *shape, const void *x, const int32_t *topk_idx,
                             int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                             int32_t *slot_of, int32_t *src_of, void *expert_x,
                             float *expert_x_scale, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Combine: y[g] = bf16( sum over k of w[g,k] * expert_y[idx[g,k]][slot_of[g,k]] ).
 *
 * Follows "Efficient and portable mixture-of-experts communication",
 * Introduction and Combine (the receiver reads the 16-bit expert outputs of
 * each token and forms their router-weighted sum) and "Enabling
 * trillion-parameter models on AWS EFA", Dispatch and Combine.  Arithmetic:
 * one fp32 accumulator from +0, one fused multiply-add per k in ascending k,
 * one round-to-nearest-even to bf16.
 *
 * In:   expert_y     [E, cap, H] bf16, 16-byte aligned; only rows
 *                    (idx[g,k], slot_of[g,k]) are read
 *       topk_idx, slot_of [N, K] int32; topk_weights [N, K] fp32
 * Out:  y            [N, H] bf16, 16-byte aligned
 * Work: the workspace moe_plan used; nothing is written if its status word
 *       is set; entries out of range are skipped and set it; entries with
 *       slot_of = -1 (not routed) are skipped silently.
 * Host errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA. */
moe_status moe_combine(const moe_shape *shape, const void *expert_y,
                       const int32_t *topk_idx, const int32_t *slot_of,
                       const float *topk_weights, void *y,
                       void *workspace, void *stream);

/* Combine fused with the shared expert:
 * y[g] = bf16( shared_y[g] + sum over k of w[g,k] * expert_y[idx[g,k]][slot_of[g,k]] ).
 *
 * Follows "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", Expert Parallelism and Compute/Communication Overlap (every
 * token also passes through a shared expert whose output is added to the
 * routed sum).  Arithmetic: the fp32 accumulator starts at the bf16 shared
 * value, then one fused multiply-add per k in ascending k, one final
 * round-to-nearest-even -- one pass instead of a combine plus an add.
 * In:   shared_y [N, H] bf16, 16-byte aligned (may be the same array as y);
 *       everything else as moe_combine.
 * Errors: as moe_combine. */
moe_status moe_combine_shared(const moe_shape *shape, const void *expert_y,
                              const int32_t *topk_idx, const int32_t *slot_of,
                              const float *topk_weights, const void *shared_y, void *y,
                              void *workspace, void *stream);

/* Router: top-K experts and their weights from router logits, ready for
 * moe_plan.
 *
 * Follows "Efficient and portable mixture-of-experts communication",
 * Introduction (the router produces a probability distribution over the
 * experts; the K highest-scoring experts are chosen and their outputs are
 * averaged with weights from that distribution) and "Lower latency and
 * higher throughput with multi-node DeepSeek deployment", MoE Router (a
 * sort that tracks indices; sparse kernels consume the top-K indices and
 * scores directly).  Per token: the K largest logits in descending order,
 * ties to the lower expert index; weights = softmax over those K logits,
 * exp(l_k - l_max) / sum, rounded once to fp32.  The weights are computed in
 * float-float arithmetic (pairs of fp32 values), within about 2^-36 of the
 * exact value before that rounding: each is the correctly rounded weight or
 * a neighbouring fp32 value (1 ulp).  The indices are exact.
 * In:   logits [N, E] fp32 (4-byte aligned).
 * Out:  topk_idx [N, K] int32, topk_weights [N, K] fp32.
 * Limits: K <= E <= 1024 (else UNSUPPORTED).  NaN logits: unspecified.
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, CUDA.  No workspace. */
moe_status moe_router_topk(const moe_shape *shape, const float *logits, int32_t *topk_idx,
                           float *topk_weights, void *stream);

/* Activation between the expert GEMMs, driven by the routing counts:
 * for expert e and row s < clamp(expert_num_tokens[e], 0, cap),
 *   a = SiLU(gate) * up   (gate, up = first and second half of expert_h[e][s]),
 * then 1x128 E4M3 quantisation of a by the same rule as moe_dispatch.
 *
 * Follows "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", Quantization (the SiLU kernel quantises its output on the fly
 * with one scale per 128 elements from the absolute maximum, and reads the
 * per-expert token counts, not the buffer sizes, so that it stays valid in a
 * CUDA graph).  SiLU(g) = g / (1 + e^-g) in binary32 with e^x by a fixed
 * sequence of IEEE operations (Cody-Waite reduction, degree-7 Taylor
 * polynomial with fused multiply-adds), so the bytes are reproducible.
 * In:   expert_h [E, cap, 2*intermediate] bf16, 16-byte aligned;
 *       expert_num_tokens [E] int32 (from moe_plan);
 * Out:  act_q [E, cap, intermediate] E4M3 (16-byte aligned) and act_scale
 *       [E, cap, nb] fp32, or [E, nb, cap] when shape->payload is
 *       FP8_E4M3_TSCALE, nb = ceil(intermediate / 128) (the last block is
 *       short when intermediate % 128 != 0); rows below the count only.
 * Work: the workspace of the plan that produced the counts; nothing is
 *       written if its status word is set.  Uses E and cap of `shape`.
 * Errors: INVALID_ARG, UNSUPPORTED (intermediate % 16 != 0), ALIGNMENT,
 *       WORKSPACE, CUDA. */
moe_status moe_silu_mul_quant(const moe_shape *shape, int32_t intermediate, const void *expert_h,
                              const int32_t *expert_num_tokens, void *act_q, float *act_scale,
                              void *workspace, void *stream);

/* Synchronise `stream` and read the workspace status word into *out (MOE_OK
 * or a device error).  The only call that waits for the device; meant for
 * tests and error handling, not for the hot path.
 * Errors: INVALID_ARG, CUDA. */
moe_status moe_read_status(const void *workspace, void *stream, moe_status *out);

/* Static description of a status code (never NULL). */
const char *moe_status_string(moe_status status);

/* moe_plan without a workspace, for callers that cannot allocate device
 * memory: code that is handed only its inputs and outputs, such as a plugin
 * whose host framework owns every device allocation, or a latency-critical
 * caller that must not call cudaMalloc because it can synchronise the
 * device.  The pages have no counterpart; it computes exactly what moe_plan
 * computes.
 *
 * Scratch: a 1 MiB static device array inside the library, held by every
 * GPU that loads the library until the process exits.  Shapes whose
 * moe_workspace_size exceeds 1 MiB are rejected with MOE_ERR_WORKSPACE.  All
 * calls on a device share the array: calls that may run at the same time on
 * the GPU (different streams without ordering) race, and must not be issued.
 * Each call clears the array's counters and flags before its kernel runs.
 * The first call on each device looks up the array's device address with
 * that device current (a one-time set-up); make that first call before any
 * stream capture.
 * In/Out: as moe_plan; status_out is a device int32 that receives the plan's
 *       status (MOE_OK or a device error, as moe_read_status would report).
 *       Nothing is allocated and nothing waits for the device.
 * Host errors: INVALID_ARG, UNSUPPORTED, WORKSPACE (shape too large for the
 *       static scratch), ALIGNMENT, CUDA. */
moe_status moe_plan_noalloc(const moe_shape *shape, const int32_t *topk_idx,
                            int32_t *expert_num_tokens, int32_t *expert_rank_offsets,
                            int32_t *slot_of, int32_t *src_of, int32_t *status_out,
                            void *stream);

/* Test hook (enqueued on `stream`): `flags` bit 0 makes the first tile of
 * the next moe_plan calls withhold its counts from the others, so their
 * bounded waits run out and the call reports MOE_ERR_TIMEOUT;
 * `timeout_ns` replaces the 1 s default limit of those waits (0 = default).
 * Errors: INVALID_ARG, CUDA. */
moe_status moe_workspace_set_debug(void *workspace, uint32_t flags,
                                   uint64_t timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DISPATCH_H */
