/*
 * moe.h — C ABI of the GB300 (sm_103a) Mixture-of-Experts layer forward path.
 *
 * The path, in order: gating softmax-top-k over router logits; the
 * indices <-> multihot routing map with its position map; grouping of the
 * routed slots by expert (counts, offsets, sorted token ids and weights,
 * reverse slot ids); per-expert FC1 (w13) -> silu_and_mul -> FC2 (w2); the
 * weighted sum of each token's k expert outputs.
 *
 * Sources of the semantics (web pages):
 *   [mlc]  mlc-llm, python/mlc_llm/op/moe_misc.py, "Mixture of Experts operators":
 *          gating_topk, gating_softmax_topk, moe_cumsum, get_indices,
 *          get_indptr, scatter_output, moe_sum.
 *   [mgt]  Megatron-LM, megatron/core/fusions/fused_indices_converter.py:
 *          _indices_to_multihot_kernel, _multihot_to_indices_kernel,
 *          IndicesToMultihot.
 *   [p6]   project_6, ex_engine/csrc/moe_expert_gemm.cpp:
 *          moe_decode_experts, moe_prefill_experts.
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *     row-major, at least 16-byte aligned (256-byte for the workspace). Outputs
 *     are preallocated by the caller; the library never allocates device memory.
 *     Scratch comes from a caller-provided workspace sized by the matching
 *     *_workspace_size() function.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream and performs no host
 *     synchronisation.
 *   - Return value: MOE_OK, or an MOE_ERR_* code when the host-side argument
 *     check fails (nothing is launched) or a launch fails. moe_last_error()
 *     gives a message for the calling thread's last failure.
 *   - Problems found on the device (an expert index outside [0, E), a bounded
 *     wait that gave up) are OR-ed as MOE_STATUS_* bits into the optional
 *     caller word `status` (device int32, zeroed by the caller). Kernels never
 *     trap.
 *   - Index tensors are int32; T*k must be below 2^31.
 *   - dtype is MOE_F32 or MOE_BF16 for hidden, w13, w2, out (and the FFN's
 *     intermediate activation). Router logits, routing weights and probs are
 *     float32.
 *   - Logits must be finite. Rows of `indices` must name distinct experts.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* return codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1   /* null pointer, bad size, misalignment, k > E ... */
#define MOE_ERR_UNSUPPORTED 2   /* a dtype/shape combination the library does not run */
#define MOE_ERR_CUDA 3          /* a CUDA runtime or launch error */
#define MOE_ERR_WORKSPACE 4     /* workspace pointer null/misaligned or too small */

/* dtypes */
#define MOE_F32 0
#define MOE_BF16 1

/* device status bits */
#define MOE_STATUS_BAD_INDEX 1  /* a routed expert index was outside [0, E); the slot was dropped */
#define MOE_STATUS_TIMEOUT 2    /* a bounded on-device wait gave up; outputs are invalid */

/* Limits: 1 <= k <= 32, k <= E <= 1024. */
#define MOE_MAX_TOPK 32
#define MOE_MAX_EXPERTS 1024

/*
 * Gating softmax-top-k.  [mlc] gating_topk / gating_softmax_topk.
 *   logits   [T, E] float32 (finite).
 *   weights  [T, k] float32 out: norm_topk_prob != 0: softmax over the k
 *            selected logits; == 0: the full-row softmax probability of each
 *            selected expert.
 *   indices  [T, k] int32 out: the k experts with the largest logits in
 *            descending order; of equal logits the lower expert index comes
 *            first (the page keeps a value only when a candidate is strictly
 *            greater).
 * Selection is made on the logits in both modes: softmax is strictly
 * increasing, so this equals ranking the probabilities. T may be 0.
 */
MOE_API int moe_gating_softmax_topk(const float* logits, int T, int E, int k, int norm_topk_prob,
                                    float* weights, int32_t* indices, void* stream);

/*
 * Gating softmax-top-k on bf16 logits ([T, E], raw bfloat16 bits, finite).
 * [mlc] gating_softmax_topk takes the logits dtype as a parameter; this is the
 * bf16 instance. Each logit is widened to float32 exactly, and the result is
 * bit-identical to moe_gating_softmax_topk on the widened row: same indices,
 * same float32 weights. The page casts the weights back to the logits dtype;
 * here they stay float32, the precision the align and FFN steps take. Ties are
 * frequent with 8-bit mantissas and follow the same rule (lower index first).
 * Errors and alignment as moe_gating_softmax_topk.
 */
MOE_API int moe_gating_softmax_topk_bf16(const void* logits, int T, int E, int k, int norm_topk_prob,
                                         float* weights, int32_t* indices, void* stream);

/*
 * Group-limited top-k (DeepSeek-style routing).  [mlc] group_limited_greedy_topk.
 *   scores   [T, E] float32 (finite), E = n_group * group_size.
 *   bias     [E] float32, the score correction added for the choice (method
 *            MOE_GROUP_TOPK_NOAUX_TC; may be NULL for MOE_GROUP_TOPK_GREEDY).
 *   weights  [T, k] float32 out, indices [T, k] int32 out.
 * Steps: choice = scores (+ bias); group score = largest choice value of the
 * group (GREEDY) or the float32 sum of its two largest (NOAUX_TC); the
 * topk_group best groups are kept (ties to the lower group); experts of the
 * other groups are excluded; the k largest remaining choice values are taken
 * (ties to the lower expert). weights = the choice values (GREEDY) or the
 * un-biased scores of the chosen experts (NOAUX_TC).
 * Limits: 1 <= n_group <= 32, E % n_group == 0, 1 <= topk_group <= n_group,
 * 1 <= k <= min(32, topk_group * E / n_group); NOAUX_TC needs E / n_group >= 2.
 */
#define MOE_GROUP_TOPK_GREEDY 0
#define MOE_GROUP_TOPK_NOAUX_TC 1
MOE_API int moe_group_limited_topk(const float* scores, const float* bias, int T, int E, int k,
                                   int n_group, int topk_group, int method, float* weights,
                                   int32_t* indices, void* stream);

/*
 * Indices -> multihot routing map.  [mgt] _indices_to_multihot_kernel.
 *   indices            [T, k] int32; an entry outside [0, E) (e.g. -1) is not routed.
 *   probs              [T, k] float32.
 *   multihot           [T, E] uint8 out: 1 where routed, else 0.
 *   probs_in_multihot  [T, E] float32 out: probs[t, j] at expert indices[t, j], else 0.
 *   position_map       [T, E] int32 out: j at expert indices[t, j], else -1.
 * Every output element is written exactly once. If a row names an expert twice
 * the lowest j is recorded.
 */
MOE_API int moe_indices_to_multihot(const int32_t* indices, const float* probs, int T, int k, int E,
                                    uint8_t* multihot, float* probs_in_multihot,
                                    int32_t* position_map, void* stream);

/*
 * Multihot -> indices (the inverse map).  [mgt] _multihot_to_indices_kernel.
 *   probs_in_multihot  [T, E] float32, position_map [T, E] int32 (j or -1).
 *   probs              [T, k] float32 out: probs[t, pos[t, e]] = probs_in_multihot[t, e];
 *                      slots no expert maps to are 0.
 *   indices_or_null    [T, k] int32 out (optional): the expert of each slot, -1 if none.
 * Positions outside [0, k) are ignored; two experts of one row must not share a slot.
 */
MOE_API int moe_multihot_to_indices(const float* probs_in_multihot, const int32_t* position_map,
                                    int T, int E, int k, float* probs, int32_t* indices_or_null,
                                    void* stream);

/*
 * Align by expert.  [mlc] moe_cumsum + get_indptr (exclusive) + get_indices;
 * [p6] moe_prefill_experts (counts, sorted_token_ids, sorted_weights).
 *   indices  [T, k] int32, weights [T, k] float32 (the routing of each slot).
 *   counts            [E]   int32 out: routed slots per expert.
 *   offsets           [E+1] int32 out: exclusive prefix of counts, offsets[E] = routed slots.
 *   sorted_token_ids  [T*k] int32 out: token of each sorted position.
 *   sorted_weights    [T*k] float32 out: routing weight of each sorted position.
 *   reverse_indices   [T*k] int32 out: flat slot t*k + j of each sorted position.
 * Sorted position of slot (t, j) with expert e: offsets[e] + (number of tokens
 * t' < t routed to e) — expert-major, ascending token, exactly the page's
 * mask-cumsum order. A slot whose expert lies outside [0, E) is dropped and
 * sets MOE_STATUS_BAD_INDEX; positions >= offsets[E] are then left unwritten.
 *   ws / ws_bytes: workspace of at least moe_align_workspace_size(T, k, E) bytes.
 */
MOE_API size_t moe_align_workspace_size(int T, int k, int E);
MOE_API int moe_align_by_expert(const int32_t* indices, const float* weights, int T, int k, int E,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_token_ids,
                                float* sorted_weights, int32_t* reverse_indices, void* ws,
                                size_t ws_bytes, int32_t* status, void* stream);

/*
 * Align by expert without a workspace. The source pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory when
 * they call in (host code handed tensors by a framework whose allocator it
 * cannot reach, or a runtime whose device memory is fixed at start-up), so
 * they cannot supply `ws`. Same arguments and results as moe_align_by_expert,
 * minus the workspace; it allocates nothing.
 *   - Its scratch is a fixed device array inside the library of
 *     MOE_ALIGN_NOALLOC_SCRATCH_INTS int32 (256 KiB), present on every GPU that
 *     loads the library until the process exits. Sizes needing more,
 *     ceil(T*k / 4096) * E > MOE_ALIGN_NOALLOC_SCRATCH_INTS, are rejected with
 *     MOE_ERR_UNSUPPORTED and a message from moe_last_error(); nothing is
 *     launched. (E = 128 allows T*k up to 2,097,152; E = 1024 up to 262,144.)
 *   - The first call that needs the array (T*k > 4096) in a CUDA context looks
 *     up its device address in that context (once per device for callers of
 *     the runtime's primary context; again for each context of their own, or
 *     after cudaDeviceReset); make that first call before any stream capture.
 *   - All calls share the array: calls whose work overlaps on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 */
#define MOE_ALIGN_NOALLOC_SCRATCH_INTS 65536
MOE_API int moe_align_by_expert_noalloc(const int32_t* indices, const float* weights, int T, int k,
                                        int E, int32_t* counts, int32_t* offsets,
                                        int32_t* sorted_token_ids, float* sorted_weights,
                                        int32_t* reverse_indices, int32_t* status, void* stream);

/*
 * Grouped expert FFN and weighted combine.  [p6] moe_prefill_experts /
 * moe_decode_experts; [mlc] scatter_output, moe_sum.
 *   hidden  [T, H]      dtype.
 *   w13     [E, 2I, H]  dtype; rows 0..I-1 of w13[e] are the gate projection,
 *                       rows I..2I-1 the up projection; used as x @ w13[e]^T.
 *   w2      [E, H, I]   dtype; used as act @ w2[e]^T.
 *   counts, offsets, sorted_token_ids, sorted_weights, reverse_indices: as
 *                       produced by moe_align_by_expert.
 *   out     [T, H]      dtype out:
 *     out[t] = sum_{j<k} w[t,j] * FC2_e(silu(FC1g_e(x_t)) * FC1u_e(x_t)),  e = expert of slot (t, j),
 *     with float32 accumulation; for bf16 the activation is rounded to bf16
 *     before FC2 and the output once at the end. Slots that were dropped by
 *     the align step contribute nothing.
 *   ws / ws_bytes: at least moe_grouped_ffn_workspace_size(...) bytes.
 * bf16 with H % 64 == 0 and I % 64 == 0 runs on the tcgen05 tensor cores;
 * other shapes and float32 run on a CUDA-core path.
 */
MOE_API size_t moe_grouped_ffn_workspace_size(int dtype, int T, int H, int I, int E, int k);
MOE_API int moe_grouped_ffn(const void* hidden, const void* w13, const void* w2, int dtype, int T,
                            int H, int I, int E, int k, const int32_t* counts,
                            const int32_t* offsets, const int32_t* sorted_token_ids,
                            const float* sorted_weights, const int32_t* reverse_indices,
                            void* out, void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * Backward of the grouped expert FFN and the weighted combine (the training
 * side of moe_grouped_ffn). The pages print the forward ([p6]
 * moe_prefill_experts; [mlc] scatter_output, moe_sum) and name the training
 * use ([mgt] IndicesToMultihot has a backward); this is the derivative of that
 * forward. Per routed slot p (token t, expert e, weight w_p; g, u the gate and
 * up pre-activations, s = sigmoid(g), a = g s u rounded to bf16 as in the
 * forward, y = a W2[e]^T):
 *   d_weights[t, j] = <d_out[t], y_p>                  (slot p = (t, j))
 *   d_w2[e]         = sum_p (w_p d_out[t]) a_p^T        [H, I]
 *   da_p = w_p d_out[t] W2[e];  dg = da u s (1 + g (1 - s));  du = da g s
 *   d_w13[e]        = sum_p [dg du]_p^T x_t             [2I, H]
 *   d_hidden[t]     = sum_j [dg du]_p W13[e]            [H]
 * The bf16 rounding of a is differentiated as the identity. FC1 is
 * recomputed (nothing from the forward call is needed besides its inputs and
 * its routing). Inputs as moe_grouped_ffn plus d_out [T, H] bf16; outputs
 * d_hidden [T, H], d_w13 [E, 2I, H], d_w2 [E, H, I] (bf16, float32
 * accumulation, one rounding) and d_weights_or_null [T, k] float32 (0 for
 * dropped slots). Experts without rows get zero weight gradients.
 * bf16 with H % 64 == 0 and I % 64 == 0 only (MOE_ERR_UNSUPPORTED otherwise).
 * ws / ws_bytes: at least moe_grouped_ffn_backward_workspace_size(...) bytes
 * (0 for an unsupported dtype).
 */
MOE_API size_t moe_grouped_ffn_backward_workspace_size(int dtype, int T, int H, int I, int E, int k);
MOE_API int moe_grouped_ffn_backward(const void* hidden, const void* w13, const void* w2, int dtype, int T,
                                     int H, int I, int E, int k, const int32_t* counts,
                                     const int32_t* offsets, const int32_t* sorted_token_ids,
                                     const float* sorted_weights, const int32_t* reverse_indices,
                                     const void* d_out, void* d_hidden, void* d_w13, void* d_w2,
                                     float* d_weights_or_null, void* ws, size_t ws_bytes, int32_t* status,
                                     void* stream);

/*
 * Whole layer: gating -> align -> grouped FFN -> combine, in one call, on one
 * stream, without host synchronisation.
 *   hidden [T, H] dtype, router_logits [T, E] float32, w13, w2 as above.
 *   out [T, H] dtype out.
 *   topk_weights_or_null [T, k] float32 / topk_indices_or_null [T, k] int32:
 *     optional copies of the gating result.
 *   ws / ws_bytes: at least moe_layer_workspace_size(...) bytes; calls that may
 *     run at the same time need separate workspaces.
 * For T <= 2 (bf16, E <= 64) the grouped FFN is one kernel whose CTAs wait for
 * one another's FC1 work (per-expert counters; one CTA on every SM but one, all
 * resident together); if such a wait runs out (moe_set_wait_limit_ns) the call
 * sets MOE_STATUS_TIMEOUT in *status and its output is not valid.
 */
MOE_API size_t moe_layer_workspace_size(int dtype, int T, int H, int I, int E, int k);
MOE_API int moe_layer_forward(const void* hidden, const float* router_logits, const void* w13,
                              const void* w2, int dtype, int T, int H, int I, int E, int k,
                              int norm_topk_prob, void* out, float* topk_weights_or_null,
                              int32_t* topk_indices_or_null, void* ws, size_t ws_bytes,
                              int32_t* status, void* stream);

/*
 * Expert-parallel exchange: G ranks, rank r owning the E_local = E / G
 * consecutive experts [r*E_local, (r+1)*E_local). [mgt]
 * _indices_to_multihot_kernel restricts a rank's routing map to its local
 * experts; the owner runs [p6] moe_prefill_experts on the rows routed to them;
 * the sender forms [mlc] scatter_output + moe_sum. These calls are the index
 * and row work on either side of the two all-to-all exchanges (which the
 * caller runs, e.g. with NCCL):
 *   sender:   gating, moe_align_by_expert (global E), moe_gather_rows; the rows
 *             for owner r are x_sorted[offsets[r*E_local] .. offsets[(r+1)*E_local])
 *             and go out in rank order, with the [G, E_local] slices of counts;
 *   owner:    moe_ep_receive_index on the received counts table, then
 *             moe_grouped_ffn on the received rows with k = 1, sorted_token_ids =
 *             reverse_indices = perm and weights 1: its output rows stay in the
 *             received order;
 *   sender:   the rows come back in x_sorted order; moe_ep_combine.
 */

/*
 * x_sorted[p] = hidden[sorted_token_ids[p]] for p < offsets[E] (rows beyond are
 * left as they are). hidden [T, H] dtype; sorted_token_ids [T*k] and offsets
 * [E+1] from moe_align_by_expert; x_sorted [T*k, H] dtype. Rows must be a
 * multiple of 16 bytes (H % 8 == 0 for bf16, H % 4 for float32), else
 * MOE_ERR_UNSUPPORTED.
 */
MOE_API int moe_gather_rows(const void* hidden, const int32_t* sorted_token_ids, const int32_t* offsets,
                            int dtype, int T, int H, int E, int k, void* x_sorted, void* stream);

/*
 * Owner side. recv_counts [G, E_local] int32: row g = the counts of this
 * rank's experts that source g sent (its rows arrive source-major, each
 * source's rows expert-major); R = their sum (rows received).
 *   local_counts  [E_local]      rows per local expert;
 *   local_offsets [E_local + 1]  exclusive prefix;
 *   perm          [R]            perm[p] = received row at expert-major position
 *                                p (sources in rank order within an expert).
 * G * E_local <= 65536. ws / ws_bytes: moe_ep_receive_workspace_size(G, E_local).
 */
MOE_API size_t moe_ep_receive_workspace_size(int G, int E_local);
MOE_API int moe_ep_receive_index(const int32_t* recv_counts, int G, int E_local, int R, int32_t* local_counts,
                                 int32_t* local_offsets, int32_t* perm, void* ws, size_t ws_bytes, void* stream);

/*
 * Sender side, after the return exchange: y_sorted [T*k, H] dtype holds the
 * expert output of sorted row p (its first offsets[E] rows are used);
 *   out[t] = sum_{j<k} topk_weights[t, j] * y_sorted[pos(t*k + j)]
 * where pos inverts reverse_indices (slots the align step dropped add
 * nothing); float32 accumulation in j order, one rounding to dtype. Rows must
 * be a multiple of 16 bytes. ws / ws_bytes: moe_ep_combine_workspace_size(T, k).
 */
MOE_API size_t moe_ep_combine_workspace_size(int T, int k);
MOE_API int moe_ep_combine(const void* y_sorted, const float* topk_weights, const int32_t* reverse_indices,
                           const int32_t* offsets, int dtype, int T, int k, int H, int E, void* out, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * Bounded waits. Every wait of the tensor-core FFN kernels (forward
 * prefill and decode) on another role of the same kernel (a pipeline slot,
 * an accumulator buffer) gives up after `ns` nanoseconds of GPU global time:
 * the kernel then stops issuing work, lets the copies and MMAs it already
 * issued finish, frees its tensor memory, ORs MOE_STATUS_TIMEOUT into the
 * call's `status` word and returns, leaving the CUDA context usable (the
 * call's output is then undefined). The default is 2 s; ns = 0 restores it.
 * The value is read when a kernel is launched (a captured CUDA graph keeps
 * the value of its capture). Returns the previous limit. The pages have no
 * counterpart: this is the watchdog of the library's own pipelines.
 */
MOE_API uint64_t moe_set_wait_limit_ns(uint64_t ns);

/*
 * Kernel timing.  moe_profiler_enable(1) makes every launch of this library
 * record a CUDA event pair on its stream; moe_profiler_report() synchronises
 * on those events, writes a JSON object {"kernel": {"launches": n,
 * "total_ms": t}, ...} into buf (NUL-terminated, truncated to len) and clears
 * the record. Returns the number of bytes needed (excluding the NUL).
 * Not for use inside CUDA graph capture.
 */
MOE_API int moe_profiler_enable(int on);
MOE_API int moe_profiler_report(char* buf, size_t len);

/* Message for the calling thread's last failed call ("" if none). */
MOE_API const char* moe_last_error(void);
/* Build identification string. */
MOE_API const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
