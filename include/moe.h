/*
 * moe.h -- C ABI of the GB300 (sm_103a) local Mixture-of-Experts FFN forward.
 *
 * The computation, following the ruDNN user guide (sections 3-7) and the
 * aclnnMoeDistributeCombineAddRmsNormV2 "Function" formula:
 *
 *   logits [T,E] --route--> expert indices [T,k] (U32), weights [T,k]
 *     --dispatch--> rows grouped by expert (no token dropped) + saved map
 *     --experts--> per row of expert e: (SiLU(x Wg[e]^T) * (x Wu[e]^T)) Wd[e]^T
 *     --combine--> y[t] = sum_j w[t,j] * expert_out[row of (t,j)]
 *     (--optional--> x = y + residual, out = x / sqrt(mean(x^2) + eps) * gamma)
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller (for
 *     example a torch tensor's data_ptr()); tensors are dense, row-major,
 *     with the shapes given below. The library never allocates, frees or
 *     retains memory: scratch space is a caller-provided workspace whose size
 *     the matching *_workspace_size() returns (0 means none is needed).
 *   - Tensor and workspace pointers must be 16-byte aligned (the workspace
 *     256-byte aligned); otherwise MOE_ERR_ALIGN / MOE_ERR_WORKSPACE.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     compute call only enqueues kernels on it and returns without waiting;
 *     outputs are valid once the stream reaches that point.
 *   - Arguments are validated on the host before anything is enqueued. A
 *     call that returns an error has enqueued nothing and left every output
 *     untouched. T == 0 is valid and enqueues nothing.
 *   - Errors found on the device (an expert index >= E handed to
 *     moe_dispatch; a bounded wait inside a kernel that ran out) do not stop
 *     the stream: the affected output rows become NaN and a per-device status
 *     word records the error; read it with moe_device_status().
 *
 * Element types: expert weights, x, intermediate and output activations share
 * one dtype (ruDNN user guide section 5: "same floating-point dtype"). FP32
 * runs on CUDA cores in true FP32; BF16 and F16 run on the tcgen05 tensor
 * cores with FP32 accumulation. Logits may be F32, BF16 or F16 on their own
 * (ruDNN user guide section 4).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum moe_dtype {
    MOE_F32 = 0,
    MOE_BF16 = 1,
    MOE_F16 = 2
} moe_dtype;

/* Status codes (every entry point returns one as an int). */
typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULL = 1,           /* a required pointer is NULL */
    MOE_ERR_SHAPE = 2,          /* a size is out of range or inconsistent */
    MOE_ERR_DTYPE = 3,          /* unsupported dtype or dtype combination */
    MOE_ERR_VALUE = 4,          /* a scalar argument is invalid (eps) */
    MOE_ERR_ALIGN = 5,          /* a tensor pointer is not 16-byte aligned */
    MOE_ERR_WORKSPACE = 6,      /* workspace too small or misaligned */
    MOE_ERR_CUDA = 7,           /* the CUDA runtime reported an error */
    MOE_ERR_DEVICE_TIMEOUT = 8, /* device status: a bounded wait gave up */
    MOE_ERR_BAD_INDEX = 9,      /* device status: an expert index >= E */
    MOE_ERR_BOUNDS = 10         /* device status (bounds-checking build only): an
                                   index read from a buffer lay outside the buffer it
                                   addresses; the access was skipped */
} moe_status;

/* Human-readable text of a status code; never NULL. */
const char *moe_status_string(int status);

/* Library ABI version (major * 100 + minor): 101. */
int moe_abi_version(void);

/* Text describing the last error returned on the calling thread (which
 * argument or which CUDA call failed); "" if none. Never NULL. */
const char *moe_last_error_detail(void);

/*
 * moe_route -- softmax top-k routing.
 * ruDNN user guide, section 4 "Routing contract".
 *
 *   logits          [T, E], dtype logits_dtype (F32/BF16/F16), read only.
 *   T >= 0, 1 <= E <= 1024, 1 <= top_k <= E.
 *   expert_indices  [T, top_k] uint32, written.
 *   weights         [T, top_k] in logits_dtype, written.
 *
 * Per token: FP32 softmax over all E logits; the top_k experts by FP32
 * logit, highest first, the lower expert id first among equal logits (the
 * softmax is strictly increasing, so this is its top-k); if renormalize != 0
 * the selected probabilities are divided by their FP32 sum; the result is
 * rounded once to logits_dtype. A row holding NaN or +inf, or holding only
 * -inf, gets indices 0..top_k-1 and NaN weights (it is not replaced by a
 * uniform distribution). A -inf logit in an otherwise valid row has weight 0.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_ALIGN,
 * MOE_ERR_CUDA.
 */
int moe_route(const void *logits, int logits_dtype, int64_t T, int64_t E,
              int top_k, int renormalize, uint32_t *expert_indices,
              void *weights, void *stream);

/*
 * moe_route_sigmoid_grouped -- group-limited sigmoid routing.
 * ruDNN user guide, section 10 "Group-limited sigmoid MoE routing".
 *
 *   logits          [T, E], dtype logits_dtype (F32/BF16/F16), read only.
 *   bias            [E] FP32 correction, read only; NULL means all zero.
 *   T >= 0, 1 <= E <= 1024, 1 <= groups <= 128 with E % groups == 0,
 *   1 <= selected_groups <= groups, 1 <= top_k <= 64 and
 *   top_k <= selected_groups * (E / groups); group_top_two needs
 *   E / groups >= 2; scale finite and > 0.
 *   expert_indices  [T, top_k] uint32, written.
 *   weights         [T, top_k] in logits_dtype, written.
 *
 * Per token: FP32 scores s_e = 1 / (1 + exp(-l_e)); selection scores
 * c_e = s_e + bias_e (FP32; the bias affects the selection only); groups
 * are the E/groups consecutive experts starting at g*(E/groups), each scored
 * by its largest c, or by the FP32 sum of its two largest c when
 * group_top_two != 0; the selected_groups best groups are kept (higher score
 * first, lower group id among equal scores); top_k experts of the kept
 * groups are picked by c, highest first, lower id among equal c; their
 * weights are the scores s, divided by their FP32 sum (in pick order) when
 * renormalize != 0, then multiplied by scale and rounded once to
 * logits_dtype. A row whose corrected scores hold a NaN (a NaN logit or bias)
 * gets indices 0..top_k-1 and NaN weights. +inf and -inf logits are valid
 * (scores 1 and 0).
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_VALUE (scale),
 * MOE_ERR_ALIGN (logits, indices, weights and a non-NULL bias must be
 * 16-byte aligned), MOE_ERR_CUDA.
 */
int moe_route_sigmoid_grouped(const void *logits, int logits_dtype, int64_t T, int64_t E,
                              const float *bias, int top_k, int groups, int selected_groups,
                              int group_top_two, int renormalize, float scale,
                              uint32_t *expert_indices, void *weights, void *stream);

/*
 * moe_dispatch -- compact dispatch with a saved map; nothing is dropped.
 * ruDNN user guide, section 5 "Expert weights and dispatch".
 *
 *   expert_indices  [T, top_k] uint32 (as written by moe_route), read only.
 *   x               [T, H] in x_dtype, read only. H >= 1.
 *   counts          [E] int32, written: assignments per expert.
 *   offsets         [E + 1] int32, written: exclusive prefix sum of counts;
 *                   the rows of expert e are [offsets[e], offsets[e+1]).
 *   row_of          [T * top_k] int32, written: row_of[t*top_k + j] is the
 *                   dispatched row of assignment (t, j).
 *   src_of          [T * top_k] int32, written: the inverse map,
 *                   src_of[row] = t*top_k + j.
 *   x_disp          [T * top_k, H] in x_dtype, written: x_disp[row] = x[t].
 *   workspace       moe_dispatch_workspace_size(T, top_k, E) bytes.
 *
 * Rows inside one expert's segment follow the assignment order t*top_k + j
 * (the pages leave this order unspecified; the library makes it
 * deterministic). An index >= E gets no row: row_of = -1, the status word
 * records MOE_ERR_BAD_INDEX, src_of/x_disp rows past offsets[E] are -1 /
 * untouched. Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE,
 * MOE_ERR_ALIGN, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
size_t moe_dispatch_workspace_size(int64_t T, int top_k, int64_t E);
int moe_dispatch(const uint32_t *expert_indices, int64_t T, int top_k,
                 int64_t E, const void *x, int x_dtype, int64_t H,
                 int32_t *counts, int32_t *offsets, int32_t *row_of,
                 int32_t *src_of, void *x_disp, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * moe_dispatch_special -- moe_dispatch for routing that also names special
 * experts (aclnnMoeDistributeCombineAddRmsNormV2, parameter list: zero, copy
 * and const experts take the ids after the E routed experts). Ids in
 * [E, E + special_experts) get no dispatched row (row_of = -1) and are not
 * reported as bad indices; moe_combine_v2 computes their contribution. Ids
 * >= E + special_experts are bad indices as in moe_dispatch. Arguments,
 * workspace and errors are those of moe_dispatch; special_experts >= 0.
 */
int moe_dispatch_special(const uint32_t *expert_indices, int64_t T, int top_k, int64_t E,
                         int64_t special_experts, const void *x, int x_dtype, int64_t H,
                         int32_t *counts, int32_t *offsets, int32_t *row_of, int32_t *src_of,
                         void *x_disp, void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_dispatch_noalloc -- moe_dispatch for callers that cannot allocate.
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot supply device scratch memory: code whose device memory belongs
 * to a pool that permits no allocation after start-up (for example a serving
 * engine that reserves HBM up front, or a plugin whose host framework gives
 * it no scratch in its enqueue step), and code that cannot pay for the
 * device-wide synchronisation cudaMalloc / cudaFree bring on a latency-
 * critical path.
 *
 * Arguments, outputs, ordering and errors are those of moe_dispatch, minus
 * the workspace: the scratch lives in a 256 KiB array that the library owns
 * on each device (kept until the process exits). It serves every problem
 * whose moe_dispatch_workspace_size(T, top_k, E) is at most 256 KiB (on a
 * 152-SM GB300 that covers, for example, every T*top_k <= 65536 with
 * E <= 256 and every T*top_k <= 16384 with E <= 1024); larger problems
 * return MOE_ERR_WORKSPACE before anything is enqueued.
 * The library allocates nothing for this call. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) and caches it;
 * make that first call before any stream capture. Every call on a device
 * shares the one array: calls whose kernels overlap on the GPU (different
 * streams without ordering between them) race on it. Nothing in the array
 * has to start at zero: each call writes every counter it reads.
 */
int moe_dispatch_noalloc(const uint32_t *expert_indices, int64_t T, int top_k,
                         int64_t E, const void *x, int x_dtype, int64_t H,
                         int32_t *counts, int32_t *offsets, int32_t *row_of,
                         int32_t *src_of, void *x_disp, void *stream);

/*
 * moe_experts_forward -- bias-free SwiGLU experts on dispatched rows.
 * ruDNN user guide, sections 3 and 5 (SwiGluExperts::forward_dispatched);
 * aclnnFFN "Formula" with no bias and a SwiGLU activation.
 *
 *   x_disp    [rows, H] in dtype, read only.
 *   offsets   [E + 1] int32 (device), read only: rows of expert e are
 *             [offsets[e], offsets[e+1]); offsets[E] <= rows.
 *   gate, up  [E, I, H] in dtype;  down [E, H, I] in dtype.
 *   out_disp  [rows, H] in out_dtype (dtype or MOE_F32), written for rows
 *             < offsets[E]; rows past offsets[E] are left untouched.
 *   workspace moe_experts_workspace_size(...) bytes (holds h [rows, I]).
 *
 * For each row r of expert e: g = Wg[e] x_r, u = Wu[e] x_r,
 * h = SiLU(g) * u with SiLU(z) = z / (1 + exp(-z)), out_r = Wd[e] h.
 * BF16/F16: tcgen05 tensor cores, FP32 accumulation, h rounded to dtype
 * between the two GEMMs; out_dtype MOE_F32 keeps the expert outputs
 * unrounded for a following combine. F32: CUDA cores, FP32 throughout.
 * Constraints: H*elem and I*elem multiples of 16 bytes (BF16/F16: H % 8 and
 * I % 8 == 0; F32: H % 4 and I % 4 == 0); 1 <= E <= 1024.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_ALIGN,
 * MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
size_t moe_experts_workspace_size(int64_t rows, int64_t E, int64_t H,
                                  int64_t I, int dtype);
int moe_experts_forward(const void *x_disp, const int32_t *offsets,
                        int64_t rows, const void *gate, const void *up,
                        const void *down, int64_t E, int64_t H, int64_t I,
                        int dtype, void *out_disp, int out_dtype,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_combine -- restore token order and sum the weighted expert outputs.
 * ruDNN user guide, sections 3 and 6 (DispatchedTokens::combine).
 *
 *   out_disp  [T * top_k, H] in out_dtype (dtype or MOE_F32), read only.
 *   weights   [T, top_k] in weights_dtype (F32, BF16 or F16), read only.
 *   row_of    [T * top_k] int32, read only (from moe_dispatch).
 *   y         [T, H] in dtype, written.
 *
 * y[t] = sum over j < top_k, in slot order, of weights[t,j] *
 * out_disp[row_of[t*top_k + j]], accumulated in FP32, rounded once to dtype.
 * A slot with row_of < 0 or >= T * top_k (no row inside out_disp) makes the
 * token's row NaN. Needs H % 8 == 0.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_ALIGN,
 * MOE_ERR_CUDA.
 */
int moe_combine(const void *out_disp, int out_dtype, const void *weights,
                int weights_dtype, const int32_t *row_of, int64_t T, int top_k,
                int64_t H, void *y, int dtype, void *stream);

/*
 * moe_combine_add_rmsnorm -- combine, residual Add and RMSNorm in one pass.
 * aclnnMoeDistributeCombineAddRmsNormV2, "Function" formula, without its
 * ReduceScatterV / AlltoAllV exchange (this library is single-GPU):
 *   x = combine + residual,  y = x / sqrt(mean(x^2) + eps) * gamma.
 * ruDNN user guide section 7: eps finite and > 0, FP32 statistics.
 *
 *   out_disp, out_dtype, weights, row_of, T, top_k, H as for moe_combine.
 *   residual  [T, H] in dtype, read only.
 *   gamma     [H] in gamma_dtype (F32, BF16 or F16), read only.
 *   y         [T, H] in dtype, written (normalised output, yOut).
 *   x_out     [T, H] in dtype, written (the pre-norm sum, xOut).
 *   rstd      [T] float, written: 1 / sqrt(mean(x_out^2) + eps) (rstdOut).
 *
 * The statistics are taken on x_out after it is rounded to dtype, so y
 * equals RMSNorm applied to x_out. Needs H % 8 == 0 and H <= 16384 (a row
 * is normalised in one pass from registers). Errors: MOE_ERR_NULL,
 * MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_VALUE, MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_combine_add_rmsnorm(const void *out_disp, int out_dtype,
                            const void *weights, int weights_dtype,
                            const int32_t *row_of, const void *residual,
                            int dtype, const void *gamma, int gamma_dtype,
                            float eps, int64_t T, int top_k, int64_t H,
                            void *y, void *x_out, float *rstd, void *stream);

/*
 * Optional inputs of moe_combine_v2 (aclnnMoeDistributeCombineAddRmsNormV2,
 * formula and parameter list). All pointers are device pointers owned by the
 * caller; a NULL pointer or zero count turns the feature off.
 *   expert_indices   [T, top_k] uint32 ids the tokens were routed to; needed
 *                    when any special experts are configured.
 *   num_experts      E: ids below E are routed experts (rows via row_of).
 *   zero_experts     ids [E, E+zero) contribute 0 (zero experts).
 *   copy_experts     the next copy_experts ids contribute ori_x[t].
 *   const_experts    the next const_experts ids, c = id - E - zero - copy,
 *                    contribute const_alpha1[c] * ori_x[t]
 *                    + const_alpha2[c] * const_v[c].
 *   ori_x            [T, H] in the activation dtype: the tokens before the
 *                    FFN (needed for copy or const experts; 16-byte aligned).
 *   const_alpha1/2   [const_experts] in the activation dtype.
 *   const_v          [const_experts, H] in the activation dtype (aligned).
 *   shared_expert_x  [T, H] in the activation dtype, or NULL: the shared
 *                    expert's output, added once per kept slot scaled by
 *                    that slot's weight, as the formula prints it.
 *   active_mask      NULL, [T] (active_mask_dims 1) or [T, top_k] (2) bytes,
 *                    nonzero = kept. A dropped token (1-D) or slot (2-D)
 *                    contributes nothing. The operator requires a 1-D mask to
 *                    keep its tokens first; here each token follows its flag.
 */
typedef struct moe_combine_extras {
    const uint32_t *expert_indices;
    int64_t num_experts;
    int64_t zero_experts;
    int64_t copy_experts;
    int64_t const_experts;
    const void *ori_x;
    const void *const_alpha1;
    const void *const_alpha2;
    const void *const_v;
    const void *shared_expert_x;
    const uint8_t *active_mask;
    int active_mask_dims;
} moe_combine_extras;

/*
 * moe_combine_v2 -- the local math of aclnnMoeDistributeCombineAddRmsNormV2:
 * combineOut[t] = sum over kept slots j of (w[t,j] * o_j + w[t,j] * sharedX[t])
 * with o_j the routed expert's row out_disp[row_of[t*top_k+j]] or the
 * special expert's output (see moe_combine_extras); then, when residual is
 * not NULL, x = combineOut + residual (x_out, rounded to dtype), rstd and
 * y = x / sqrt(mean(x^2) + eps) * gamma exactly as moe_combine_add_rmsnorm;
 * when residual is NULL, y = combineOut rounded to dtype and gamma, eps,
 * x_out, rstd are unused. extras may be NULL (then this is moe_combine or
 * moe_combine_add_rmsnorm). A routed slot without a row, or an id past the
 * last special expert, makes the token's row NaN. Arguments and errors as
 * moe_combine / moe_combine_add_rmsnorm, plus MOE_ERR_NULL / MOE_ERR_ALIGN /
 * MOE_ERR_SHAPE for inconsistent extras.
 */
int moe_combine_v2(const void *out_disp, int out_dtype, const void *weights, int weights_dtype,
                   const int32_t *row_of, const moe_combine_extras *extras,
                   const void *residual, const void *gamma, int gamma_dtype, float eps,
                   int64_t T, int top_k, int64_t H, void *y, int dtype, void *x_out,
                   float *rstd, void *stream);

/*
 * moe_rmsnorm -- RMSNorm over the last axis.
 * ruDNN user guide, section 7 "LayerNorm, RMSNorm and Softmax".
 *
 *   x      [rows, H] in dtype (F32/BF16/F16), read only; H % 8 == 0,
 *          1 <= H <= 16384.
 *   gamma  [H] in gamma_dtype (F32, or dtype).
 *   eps    finite and > 0.
 *   y      [rows, H] in dtype, written: x / sqrt(mean(x^2) + eps) * gamma.
 *   rstd   [rows] FP32, written when not NULL: 1 / sqrt(mean(x^2) + eps).
 * Statistics and the affine step in FP32, output rounded once to dtype.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_VALUE (eps),
 * MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_rmsnorm(const void *x, int dtype, const void *gamma, int gamma_dtype, float eps,
                int64_t rows, int64_t H, void *y, float *rstd, void *stream);

/*
 * moe_forward -- the whole local forward in one call: route, dispatch,
 * experts, combine. ruDNN user guide, section 6 (SwiGluExperts::forward):
 * takes precomputed logits (no gate projection, no weight loading).
 *
 *   x       [T, H] in dtype;   logits [T, E] in logits_dtype.
 *   gate, up [E, I, H];  down [E, H, I], in dtype.
 *   y       [T, H] in dtype, written.
 *   workspace moe_forward_workspace_size(...) bytes; it holds the routing
 *           plan, the dispatch map and the dispatched activations.
 * Same rules and errors as the staged calls, and the same arithmetic as
 * moe_route -> moe_dispatch -> moe_experts_forward (out_dtype MOE_F32) ->
 * moe_combine: expert outputs reach the combine unrounded. For BF16/F16 with
 * T*H*4 <= 64 MiB (an accumulator that stays in L2) the combine runs inside
 * the second expert GEMM, which adds each weighted row into an FP32 [T, H]
 * accumulator with reductions whose order varies from run to run: each FP32
 * sum is within k * 2^-24 * sum_j |w_j * o_j| of the exact sum, so repeated
 * calls may differ by that much plus one unit in the last place of the
 * output dtype (usually at most the one unit; more only where the k terms
 * cancel). Otherwise, for FP32 runs, and for the staged calls the result is
 * bit-reproducible. Needs H % 8 == 0.
 */
size_t moe_forward_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E,
                                  int top_k, int dtype, int logits_dtype);
int moe_forward(const void *x, int dtype, const void *logits,
                int logits_dtype, const void *gate, const void *up,
                const void *down, int64_t T, int64_t H, int64_t I, int64_t E,
                int top_k, int renormalize, void *y, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * moe_forward_sigmoid_grouped -- the one-call forward of moe_forward with
 * group-limited sigmoid routing in place of softmax top-k routing
 * (ruDNN user guide, section 10, SwiGluExperts::forward_sigmoid_grouped):
 * moe_route_sigmoid_grouped -> dispatch -> SwiGLU experts -> weighted
 * combine. Arguments are those of moe_forward plus the routing arguments of
 * moe_route_sigmoid_grouped (same limits and errors); the workspace is
 * moe_forward_workspace_size(T, H, I, E, top_k, dtype, logits_dtype) bytes.
 * The routing weights enter the combine as they are (with scale applied).
 */
int moe_forward_sigmoid_grouped(const void *x, int dtype, const void *logits, int logits_dtype,
                                const float *bias, const void *gate, const void *up,
                                const void *down, int64_t T, int64_t H, int64_t I, int64_t E,
                                int top_k, int groups, int selected_groups, int group_top_two,
                                int renormalize, float scale, void *y, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * moe_forward_ex -- moe_forward / moe_forward_sigmoid_grouped with options.
 * Same computation, arguments and errors as moe_forward (ruDNN user guide,
 * section 6, SwiGluExperts::forward), plus:
 *
 *   options  NULL, or a moe_forward_options read during the call:
 *     flags            MOE_FORWARD_* bits; other bits give MOE_ERR_VALUE.
 *       MOE_FORWARD_DETERMINISTIC  the combine always runs as its own kernel
 *                      in slot order over FP32 expert outputs (as in the
 *                      staged calls), so repeated calls on the same inputs
 *                      give bit-identical y; without it BF16/F16 forwards
 *                      whose T*H*4 <= 64 MiB fold the combine into the second
 *                      expert GEMM (see moe_forward). It needs the larger
 *                      workspace moe_forward_workspace_size_ex(..., flags).
 *     sigmoid_grouped  NULL: softmax top-k routing (moe_route); else the
 *                      group-limited sigmoid routing of
 *                      moe_route_sigmoid_grouped with these arguments (ruDNN
 *                      user guide, section 10), as moe_forward_sigmoid_grouped.
 *     experts_begin_event, experts_end_event  NULL, or cudaEvent_t handles
 *                      recorded on `stream` right before the first and right
 *                      after the last expert GEMM launch, so a caller can time
 *                      the expert GEMMs inside the one-call forward. A
 *                      recorded event stops the kernel after it from starting
 *                      early, so calls with events run slightly slower.
 *   workspace  moe_forward_workspace_size_ex(T, H, I, E, top_k, dtype,
 *              logits_dtype, flags) bytes.
 */
#define MOE_FORWARD_DETERMINISTIC 1u

typedef struct moe_sigmoid_grouped_routing {
    const float *bias;          /* [E] FP32 correction or NULL */
    int groups;
    int selected_groups;
    int group_top_two;
    float scale;
} moe_sigmoid_grouped_routing;

typedef struct moe_forward_options {
    unsigned flags;
    const moe_sigmoid_grouped_routing *sigmoid_grouped;
    void *experts_begin_event;
    void *experts_end_event;
} moe_forward_options;

size_t moe_forward_workspace_size_ex(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                                     int dtype, int logits_dtype, unsigned flags);
int moe_forward_ex(const void *x, int dtype, const void *logits, int logits_dtype,
                   const void *gate, const void *up, const void *down, int64_t T, int64_t H,
                   int64_t I, int64_t E, int top_k, int renormalize, void *y, void *workspace,
                   size_t workspace_bytes, const moe_forward_options *options, void *stream);

/*
 * moe_forward_workspace_layout -- where the one-call forward keeps its
 * routing plan and dispatch map inside the workspace (ruDNN user guide,
 * section 5: dispatch produces a saved map that combine and backward reuse).
 * For the arguments of moe_forward_workspace_size_ex, writes byte offsets
 * from the workspace start; after a moe_forward / moe_forward_ex call with
 * these sizes and flags has run, the workspace holds there:
 *   expert_indices [T, top_k] uint32, weights [T, top_k] in logits_dtype (as
 *   moe_route or moe_route_sigmoid_grouped write them), counts [E] int32,
 *   offsets [E + 1] int32, row_of and src_of [T * top_k] int32, x_disp
 *   [T * top_k, H] in dtype (as moe_dispatch writes them);
 * total is the workspace size. The layout depends only on the arguments.
 * Errors: MOE_ERR_NULL (layout), MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_VALUE
 * (unknown flag).
 */
typedef struct moe_forward_layout {
    size_t expert_indices;
    size_t weights;
    size_t counts;
    size_t offsets;
    size_t row_of;
    size_t src_of;
    size_t x_disp;
    size_t total;
} moe_forward_layout;

int moe_forward_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                                 int dtype, int logits_dtype, unsigned flags,
                                 moe_forward_layout *layout);

/* ======================================================================
 * First-order training.
 * ruDNN user guide, section 12 "MoE first-order training": the weights of a
 * fixed selection and their logits gradient; expert training in the order
 *   combine backward -> expert backward -> dispatch backward -> router
 *   backward,
 * with FP32 routing-weight and expert-weight gradients. Nothing is
 * differentiated through the top-k / group selection or a correction bias.
 * ====================================================================== */

/* Scoring of the training weights. */
typedef enum moe_router_scoring {
    MOE_SCORING_SOFTMAX = 0,
    MOE_SCORING_SIGMOID = 1
} moe_router_scoring;

/* Element type of a selection's expert ids (the section accepts U32, I32,
 * I64). */
typedef enum moe_index_dtype {
    MOE_INDEX_U32 = 0,
    MOE_INDEX_I32 = 1,
    MOE_INDEX_I64 = 2
} moe_index_dtype;

/*
 * moe_router_weights -- weights of a fixed selection (selected_router_weights).
 *
 *   logits   [T, E] in logits_dtype (F32/BF16/F16), read only.
 *   indices  [T, top_k] expert ids in index_dtype, read only.
 *   T >= 0, 1 <= E <= 1024, 1 <= top_k <= min(E, 64); scale finite and > 0.
 *   weights  [T, top_k] FP32, written.
 *
 * Slot j of token t scores s_j = softmax(logits[t])[id] (MOE_SCORING_SOFTMAX,
 * over all E logits) or sigmoid(logits[t, id]) (MOE_SCORING_SIGMOID), with
 * id = indices[t, j]; a repeated id is gathered again. With renormalize != 0
 * each s_j is divided by the sum over the k slots; every weight is then
 * multiplied by scale. FP32 arithmetic. An id outside [0, E) (negative, or
 * >= E) makes the token's row NaN, reads nothing out of bounds and sets
 * MOE_ERR_BAD_INDEX in the device status word; a softmax row holding NaN or
 * +inf, or only -inf, is NaN too (as in moe_route).
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE (logits or index dtype,
 * scoring), MOE_ERR_VALUE (scale), MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_router_weights(const void *logits, int logits_dtype, int64_t T, int64_t E,
                       const void *indices, int index_dtype, int top_k, int scoring,
                       int renormalize, float scale, float *weights, void *stream);

/*
 * moe_router_backward -- logits gradient of moe_router_weights
 * (selected_router_backward), for the same arguments and an upstream
 * gradient grad_weights [T, top_k] FP32.
 *
 *   grad_logits  [T, E] in logits_dtype, written.
 *
 * With ds_j = scale * g_j (no renormalisation) or
 * ds_j = scale * (g_j - sum_i g_i s_i / Z) / Z, Z = sum_i s_i, and G_e the
 * sum of ds_j over the slots holding expert e:
 *   softmax: d logit_e = p_e * (G_e - sum_f p_f G_f)  (every expert);
 *   sigmoid: d logit_e = G_e * s_e * (1 - s_e) for selected experts, 0 else.
 * FP32 arithmetic, rounded once to logits_dtype. Rows that
 * moe_router_weights makes NaN are NaN here. Errors as moe_router_weights.
 */
int moe_router_backward(const void *logits, int logits_dtype, int64_t T, int64_t E,
                        const void *indices, int index_dtype, int top_k,
                        const float *grad_weights, int scoring, int renormalize, float scale,
                        void *grad_logits, void *stream);

/*
 * moe_combine_backward -- backward of moe_combine
 * (DispatchedTokens::combine_backward).
 *
 *   out_disp   [T * top_k, H] expert outputs of the forward, out_dtype (dtype
 *              or F32), read only.
 *   weights    [T, top_k] routing weights in weights_dtype, read only.
 *   row_of     [T * top_k] int32 (from moe_dispatch), read only.
 *   grad_y     [T, H] in dtype, read only: the gradient of the combine output.
 *   grad_out_disp [T * top_k, H] in dtype, written for every row some slot
 *              names: grad_out_disp[row_of[t*k + j]] = weights[t, j] * grad_y[t].
 *   grad_weights  [T, top_k] FP32, written:
 *              sum over h of grad_y[t, h] * out_disp[row_of[t*k + j], h].
 *
 * FP32 arithmetic. A slot with row_of < 0 writes no row and gets a NaN
 * weight gradient. Needs H % 8 == 0. Errors: MOE_ERR_NULL, MOE_ERR_SHAPE,
 * MOE_ERR_DTYPE, MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_combine_backward(const void *out_disp, int out_dtype, const void *weights,
                         int weights_dtype, const int32_t *row_of, const void *grad_y,
                         int64_t T, int top_k, int64_t H, int dtype, void *grad_out_disp,
                         float *grad_weights, void *stream);

/*
 * moe_dispatch_backward -- backward of the dispatch gather
 * (DispatchedTokens::dispatch_backward).
 *
 *   grad_x_disp [T * top_k, H] in dtype, read only (from moe_experts_backward).
 *   row_of      [T * top_k] int32 (from moe_dispatch), read only.
 *   grad_x      [T, H] in dtype, written: sum over slots j, in slot order, of
 *               grad_x_disp[row_of[t*k + j]]; FP32 sum rounded once. The
 *               routing weight is not applied again. Slots with row_of < 0
 *               add nothing.
 * Needs H % 8 == 0. Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE,
 * MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_dispatch_backward(const void *grad_x_disp, int dtype, const int32_t *row_of,
                          int64_t T, int top_k, int64_t H, void *grad_x, void *stream);

/*
 * moe_experts_forward_training -- moe_experts_forward that also keeps what
 * the backward needs (SwiGluExperts::forward_dispatched_training).
 *
 *   Arguments as moe_experts_forward, except that the cache replaces the
 *   workspace:
 *   cache  moe_experts_training_cache_size(rows, I, dtype) bytes, 256-byte
 *          aligned, written: h [rows, I] in dtype, then g = x Wg^T and
 *          u = x Wu^T of every row as two [rows, I] FP32 arrays (kept in FP32
 *          so the backward's SiLU derivative starts from unrounded values).
 *          Keep it, unchanged, for moe_experts_backward.
 * out_disp matches moe_experts_forward with the same arguments.
 */
size_t moe_experts_training_cache_size(int64_t rows, int64_t I, int dtype);
int moe_experts_forward_training(const void *x_disp, const int32_t *offsets, int64_t rows,
                                 const void *gate, const void *up, const void *down, int64_t E,
                                 int64_t H, int64_t I, int dtype, void *out_disp, int out_dtype,
                                 void *cache, size_t cache_bytes, void *stream);

/*
 * moe_experts_backward -- backward of the SwiGLU experts (cache.backward).
 *
 *   x_disp, offsets, rows, gate, up, down, E, H, I, dtype: as given to
 *          moe_experts_forward_training; cache: what it wrote.
 *   grad_out     [rows, H] in dtype, read only: gradient of the expert
 *                outputs (grad_out_disp of moe_combine_backward).
 *   grad_x_disp  [rows, H] in dtype, written (rows < offsets[E]).
 *   grad_gate, grad_up [E, I, H] FP32, grad_down [E, H, I] FP32, written in
 *                full (experts without rows get zeros).
 *   workspace    moe_experts_backward_workspace_size(...) bytes, 256-byte
 *                aligned: dg | du [rows, 2I] in dtype and, for BF16 / F16,
 *                per-expert TMA descriptors of the weight-gradient GEMMs
 *                (so it is needed even when rows == 0).
 *
 * Per row of expert e (s = sigmoid(g)): dh = do Wd[e],
 * dg = dh * u * s * (1 + g (1 - s)), du = dh * g * s, dx = dg Wg[e] + du Wu[e];
 * dWd[e] = sum do^T h, dWg[e] = sum dg^T x, dWu[e] = sum du^T x over the
 * expert's rows. BF16/F16 run on tcgen05 tensor cores with FP32
 * accumulation (dg and du rounded to dtype between the GEMMs; h as cached);
 * F32 runs in FP32 on CUDA cores. Constraints and errors as
 * moe_experts_forward.
 */
size_t moe_experts_backward_workspace_size(int64_t rows, int64_t E, int64_t H, int64_t I,
                                           int dtype);
int moe_experts_backward(const void *x_disp, const int32_t *offsets, int64_t rows,
                         const void *gate, const void *up, const void *down, int64_t E,
                         int64_t H, int64_t I, int dtype, const void *cache,
                         const void *grad_out, void *grad_x_disp, float *grad_gate,
                         float *grad_up, float *grad_down, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * moe_device_status -- read the current device's status word.
 * Synchronises `stream`, then returns MOE_OK, MOE_ERR_BAD_INDEX,
 * MOE_ERR_BOUNDS or MOE_ERR_DEVICE_TIMEOUT (when several are set, the
 * timeout wins, then the bounds check). If clear != 0 the word is reset to
 * zero afterwards. MOE_ERR_CUDA if the read fails.
 *
 * The bounds-checking build of the library (the same ABI, built with
 * MOE_DEBUG_BOUNDS=1; the Python binding loads it when the environment
 * variable MOE_DEBUG_BOUNDS is 1) also checks, on the device, the indices
 * the kernels read from buffers before using them: the expert offsets given
 * to the expert GEMMs (they must start at 0 and never fall), the rows the
 * dispatch ranks (inside the expert's segment) and the map entries the
 * gather follows (below T * top_k). A failed check skips the access and
 * records MOE_ERR_BOUNDS. It is meant for tests and debugging, in place of
 * a memory checker.
 * (Router training in the ruDNN user guide, section 12, fixes the same rule
 * for illegal indices: NaN rows, no out-of-bounds read, no host sync.)
 */
int moe_device_status(void *stream, int clear);

/*
 * moe_set_wait_limit_ns -- how long a bounded device wait may last before it
 * gives up (the error convention of the ruDNN user guide, section 3: a
 * MoeError instead of a hang). Every spin-wait inside the tcgen05 expert
 * GEMMs (pipeline barriers, and the per-expert readiness counters of the
 * one-call forward) stops after this many nanoseconds, records
 * MOE_ERR_DEVICE_TIMEOUT in the status word, drains its own copies and MMAs
 * and lets the kernel exit. Process-wide; read when a kernel is launched
 * (a captured graph keeps the value of its capture). 0 restores the
 * default of 2 s; more than 60 s gives MOE_ERR_VALUE. Meant for tests of the
 * failure path, which shorten it so an expiry costs milliseconds.
 * moe_wait_limit_ns returns the limit in force.
 */
int moe_set_wait_limit_ns(uint64_t limit_ns);
uint64_t moe_wait_limit_ns(void);

/*
 * moe_selftest_wait_expiry -- runs the failure path of the bounded waits on
 * the GPU, without a fault. It launches the second expert GEMM of the
 * one-call forward on its own (BF16, combine folded into y_acc, top_k 1,
 * E experts of rows_per_expert rows each, all data zero) with per-expert
 * readiness counters that no first GEMM ever raises: each of its producers
 * waits the bounded time, gives up, records MOE_ERR_DEVICE_TIMEOUT, and the
 * kernel drains and exits without touching y_acc. The pages have no
 * counterpart; it exists so a test can check that a wait that can never be
 * satisfied ends in a status rather than a hang.
 *
 *   y_acc      [E * rows_per_expert, H] FP32 (16-byte aligned): not written.
 *   workspace  moe_selftest_wait_expiry_workspace_size(...) bytes, 256-byte
 *              aligned (offsets, map, routing weights, counters, h, down).
 *   1 <= E <= 1024, 1 <= rows_per_expert <= 4096, H and I multiples of 8 in
 *   [8, 8192]. Afterwards moe_device_status() reports the timeout.
 * Errors: MOE_ERR_SHAPE, MOE_ERR_NULL, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA.
 */
size_t moe_selftest_wait_expiry_workspace_size(int64_t E, int64_t rows_per_expert, int64_t H,
                                               int64_t I);
int moe_selftest_wait_expiry(int64_t E, int64_t rows_per_expert, int64_t H, int64_t I,
                             float *y_acc, void *workspace, size_t workspace_bytes,
                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
