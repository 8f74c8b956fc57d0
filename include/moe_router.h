/*
 * moe_router.h -- C ABI of the GB300 (sm_103a) MoE routing library
 * (libmoerouter.so).
 *
 * The routing hot path of a mixture-of-experts layer, as described by
 *   [TE]   NVIDIA TransformerEngine PR 3012, "[Common] Optimize fused router
 *          forward/backward kernels" (fused_topk_with_score_function,
 *          fused_score_for_moe_aux_loss, forward and backward; "Hardening";
 *          "Performance");
 *   [FLY]  ROCm FlyDSL PR 582, "Fuse TopKGatingSoftmax and MoE Sorting
 *          kernels" (top-k gating + MoE sorting, fused at decode sizes);
 *   [GEMM] ROCm FlyDSL PR 947, "Port moe_gemm_2stage ..." (the consumer of the
 *          sorted layout: id = token*topk + slot; sentinel rows contribute 0);
 *   [AIT]  ROCm aiter PR 3828, "flydsl mxfp4 a4w4 MoE gemm1/gemm2" (bare
 *          device pointers as kernel arguments; Kimi-K2.5 NE=385 TOPK=9).
 *
 * Conventions for every entry point
 *   - Array arguments are DEVICE pointers to caller-owned, contiguous,
 *     row-major memory. The library never allocates, frees or synchronises.
 *     Rows whose bases are 16-byte aligned (and E a multiple of 4) take the
 *     vectorised path; any other alignment of the element type is accepted and
 *     takes a scalar path.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; outputs are valid once the stream
 *     reaches that point.
 *   - Return value: MR_OK, or an mr_status error code. Argument errors are
 *     detected on the host BEFORE anything is enqueued (no partial writes);
 *     MR_ECUDA reports a failed launch (cudaGetLastError after the launch).
 *   - Nothing here traps or asserts on the device.
 *   - Calls on different streams may run concurrently as long as they write
 *     disjoint memory.
 */
#ifndef MOE_ROUTER_H
#define MOE_ROUTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* mr_stream_t;

typedef enum {
    MR_OK = 0,
    MR_EINVAL = 1,       /* bad argument: null required pointer, size or option out of range */
    MR_EUNSUPPORTED = 2, /* valid on the pages but outside this library's limits (below) */
    MR_ECUDA = 3,        /* a CUDA launch or query failed */
    MR_ERANGE = 4,       /* (device status only) an expert id outside [0, E_tot) was dropped */
    MR_ETIMEOUT = 5      /* (device status only) a bounded in-kernel wait gave up; the
                            outputs of the call that reported it are not valid */
} mr_status;

/*
 * Device status words. A kernel reports a condition by raising a device int32
 * status word to the condition's code with an atomic maximum, so a word holds
 * the most severe code reported since it was last zeroed (MR_ETIMEOUT >
 * MR_ERANGE > MR_OK). Calls that take a nullable `int32_t* status` report into
 * that word (the caller zeroes it before the call); a call given NULL, and
 * moe_aux_scores_fwd, report timeouts into the library's per-device word
 * instead (moe_router_device_status reads and clears it), so none is lost.
 */

typedef enum { MR_SOFTMAX = 0, MR_SIGMOID = 1 } mr_score_fn;
typedef enum { MR_F32 = 0, MR_BF16 = 1 } mr_dtype;

/* Library limits (MR_EUNSUPPORTED beyond them). */
#define MR_MAX_EXPERTS 8192      /* E, routed experts per token row (rows wider than 1024
                                    are held in shared memory; [TE] flowchart: radix top-k
                                    while num_experts <= 8160) */
#define MR_MAX_TOPK 256          /* topk - n_shared, routed slots */
#define MR_MAX_GROUPS 32         /* n_group */
#define MR_MAX_GROUP_TOPK 8      /* (topk - n_shared) / topk_group, keys summed per group */
#define MR_MAX_SORT_EXPERTS 4096 /* E_tot for moe_sort */
#define MR_MAX_FUSED_TOKENS 16   /* T at or below which the fused call is one launch ... */
#define MR_MAX_FUSED_EXPERTS 1024 /* ... when E is at most this */
#define MR_MAX_FUSED_TOKENS_SMALL_E 64  /* and T at or below which it is one launch ... */
#define MR_MAX_FUSED_EXPERTS_SMALL 256  /* ... when E is at most this */

/*
 * Router options, one token per row ([TE] fused_topk_with_score_function).
 *   T            tokens (rows), >= 0 (T == 0 is a no-op)
 *   E            routed experts (columns of logits/probs/routing_map), 1..MR_MAX_EXPERTS
 *   topk         slots per token including shared slots; k_r = topk - n_shared routed
 *                slots with 1 <= k_r <= min(E, MR_MAX_TOPK)
 *   score_fn     MR_SOFTMAX (over all E) or MR_SIGMOID (elementwise)
 *   in_dtype     MR_F32 or MR_BF16 logits; probs has the same dtype
 *   renorm       non-zero: divide the k_r routed weights by their sum before scaling
 *   n_group      0 = no group limit; else E % n_group == 0, n_group <= MR_MAX_GROUPS
 *   topk_group   groups kept (1..n_group); k_r % topk_group == 0 ([TE] "Hardening")
 *                and k_r/topk_group <= min(E/n_group, MR_MAX_GROUP_TOPK)
 *   n_shared     shared experts, always selected, ids E..E+n_shared-1 in the last slots
 *   scaling      factor applied to routed weights after renormalisation
 *   shared_weight  weight written for shared slots (not renormalised, not scaled)
 *   bias         nullable device fp32[E]; added to the sigmoid score for SELECTION only
 * Softmax with a bias or a group limit is MR_EUNSUPPORTED: its selection key is the
 * logit, and a bias or group score on logits has no stated meaning.
 */
typedef struct {
    int32_t T, E, topk, score_fn, in_dtype, renorm, n_group, topk_group, n_shared;
    float scaling, shared_weight;
    const float* bias;
} mr_router_params;

/*
 * moe_router_fwd -- score, select, weight and emit ([TE] fused_topk_with_score_function
 * forward; flowchart "score fn -> radix_topk_and_mask -> write probs + routing_map").
 *
 * For each token t:  s = score_fn(logits[t, :])  (fp32 compute)
 *   selection key: softmax -> the logit; sigmoid -> s (+ bias[e])
 *   group limit (n_group > 0): a group's score is the fp32 sum of its k_r/topk_group
 *     largest keys (largest first); the topk_group best groups are kept
 *   the k_r largest keys win; equal keys go to the LOWER expert index
 *   w_j = s_j;  renorm: w_j /= sum of the k_r winners' s (0 if the sum is 0);  w_j *= scaling
 * Outputs (each nullable; at least one required):
 *   probs[T x E]        (in_dtype)  w at the winners, 0 elsewhere
 *   routing_map[T x E]  (uint8)     1 at the winners, 0 elsewhere
 *   intermediate[T x E] (fp32)      s, the input of moe_router_bwd
 *   topk_idx[T x topk]  (int32)     winners by descending key (ties: ascending index), then shared ids
 *   topk_w[T x topk]    (fp32)      their weights, then shared_weight
 * status: nullable device int32 (see "Device status words"). Rows wider than 1024
 * experts are staged in shared memory by bulk copies whose waits are bounded; a wait
 * that gives up raises *status to MR_ETIMEOUT (the library's per-device word when
 * status is NULL) and the call's outputs are not valid.
 * Errors: MR_EINVAL (null logits, no output, sizes out of range, T*E > INT_MAX,
 * n_group/topk_group inconsistent), MR_EUNSUPPORTED (limits above), MR_ECUDA.
 */
int moe_router_fwd(const mr_router_params* p, const void* logits, void* probs,
                   uint8_t* routing_map, float* intermediate, int32_t* topk_idx, float* topk_w,
                   int32_t* status, mr_stream_t stream);

/*
 * moe_router_bwd -- gradient of probs w.r.t. logits ([TE] top-k backward, "Two-pass
 * fused design"), selection held fixed; uses T, E, score_fn, renorm, scaling of p.
 *   ds_i = scaling * m_i * g_i                                   (no renorm)
 *   ds_i = (scaling * m_i / A) * (g_i - B / A),  A = sum m s, B = sum m s g   (renorm)
 *   softmax: dx_i = s_i * (ds_i - sum_j s_j ds_j);  sigmoid: dx_i = ds_i * s_i * (1 - s_i)
 * grad_probs, intermediate, grad_logits: fp32 [T x E]; routing_map: uint8 [T x E]
 * (as written by moe_router_fwd). grad_logits is written over all T x E.
 */
int moe_router_bwd(const mr_router_params* p, const float* grad_probs, const float* intermediate,
                   const uint8_t* routing_map, float* grad_logits, mr_stream_t stream);

/*
 * moe_router_bwd_dtype -- moe_router_bwd with grad_probs and grad_logits in grad_dtype:
 * MR_F32 (exactly moe_router_bwd) or MR_BF16, the dtype of bf16 logits and probs; the
 * intermediate stays fp32. The gradient is computed in fp32 and rounded once (round to
 * nearest even) when stored. 9 bytes per element moved instead of 13 ([TE]
 * "Performance": T x E x dtype). MR_EINVAL for another grad_dtype.
 */
int moe_router_bwd_dtype(const mr_router_params* p, int grad_dtype, const void* grad_probs,
                         const float* intermediate, const uint8_t* routing_map, void* grad_logits,
                         mr_stream_t stream);

/*
 * moe_aux_scores_fwd -- scores for the load-balancing loss ([TE]
 * fused_score_for_moe_aux_loss): scores[T x E] (fp32) = score_fn over all E (no bias,
 * no groups, no renorm) and routing_map[T x E] = the top-k of those scores (same key
 * and tie rule as moe_router_fwd). Either output may be NULL, not both.
 */
int moe_aux_scores_fwd(int T, int E, int topk, int score_fn, int in_dtype, const void* logits,
                       float* scores, uint8_t* routing_map, mr_stream_t stream);

/*
 * moe_aux_scores_bwd -- its gradient: softmax dx = s * (g - sum g s); sigmoid
 * dx = g * s * (1 - s). All arrays fp32 [T x E].
 */
int moe_aux_scores_bwd(int T, int E, int score_fn, const float* grad_scores, const float* scores,
                       float* grad_logits, mr_stream_t stream);

/*
 * The aux-loss scalar ([TE] names fused_moe_aux_loss, which consumes the scores and
 * routing map above, but prints no formula; it is read as the switch-style
 * load-balancing loss: coeff * E * sum_e f_e * P_e with f_e the fraction of routed
 * slots that chose e and P_e the mean probability of e):
 *   loss = C * sum_e tokens_per_expert[e] * sum_t probs[t][e],
 *   C = coeff * E / (topk * N^2),  N = total_num_tokens (the token count the counts and
 *   probabilities were taken over; it may exceed T when tokens span several devices)
 *   d loss / d probs[t][e] = C * tokens_per_expert[e] * grad_loss
 *
 * moe_tokens_per_expert -- tokens_per_expert[e] (int32 [E]) = number of rows t with
 *   routing_map[t][e] != 0 (routing_map uint8 [T x E]). Overwrites all E entries.
 * moe_aux_loss_workspace_bytes -- device scratch moe_aux_loss_fwd needs for these
 *   sizes (per-column partial sums; 0 for T == 0, or for invalid sizes).
 * moe_aux_loss_fwd -- *loss (one fp32, device) from probs fp32 [T x E] and
 *   tokens_per_expert int32 [E]. The column sums are Kahan-compensated fp32 in a fixed
 *   order and the dot product is taken in fp64: the result is deterministic.
 *   workspace: caller-owned device scratch of at least moe_aux_loss_workspace_bytes(),
 *   16-byte aligned, contents ignored on entry; calls that share a workspace must not
 *   overlap on the GPU.
 * moe_aux_loss_bwd -- grad_probs fp32 [T x E] from grad_loss (one fp32, device).
 * All three: MR_EINVAL for a NULL required pointer, T < 0, E < 1, topk < 1,
 *   total_num_tokens < 1, T*E > INT_MAX, or a too-small or misaligned workspace.
 */
int moe_tokens_per_expert(int T, int E, const uint8_t* routing_map, int32_t* tokens_per_expert,
                          mr_stream_t stream);
size_t moe_aux_loss_workspace_bytes(int T, int E);
int moe_aux_loss_fwd(int T, int E, int topk, float coeff, long long total_num_tokens, const float* probs,
                     const int32_t* tokens_per_expert, float* loss, void* workspace, size_t ws_bytes,
                     mr_stream_t stream);
int moe_aux_loss_bwd(int T, int E, int topk, float coeff, long long total_num_tokens,
                     const int32_t* tokens_per_expert, const float* grad_loss, float* grad_probs,
                     mr_stream_t stream);

/*
 * moe_sort -- bucket (token, slot) pairs by expert into block_m-padded blocks
 * ([FLY] moe_sorting; layout as consumed by [GEMM]).
 *   cnt[e] = pairs routed to e;  pad[e] = ceil(cnt[e]/block_m)*block_m (0 if empty)
 *   off[e] = sum_{e'<e} pad[e'];  *num_tokens_post_pad = sum_e pad[e]
 *   sorted_token_ids[off[e] + r] = t*topk + j, r-th pair of e in ascending (t, j);
 *     the rest of e's range holds the sentinel T*topk (one past the last valid row)
 *   sorted_weights: topk_w of the pair (nullable in and out together), 0 at sentinels
 *   expert_ids[b] = e for each block b of e's range
 * Inputs: topk_idx int32 [T x topk], topk_w fp32 [T x topk].
 * Outputs: sorted_token_ids / sorted_weights with room for moe_sort_capacity()
 *   entries, expert_ids with room for capacity/block_m entries, num_tokens_post_pad
 *   one int32. Only [0, num_tokens_post_pad) and [0, num_tokens_post_pad/block_m)
 *   are written.
 * workspace: device scratch of at least moe_sort_workspace_bytes(), contents
 *   ignored on entry (any state), owned by the caller; the call only writes into it.
 * status: nullable device int32; an id outside [0, E_tot) is dropped and *status is
 *   raised to MR_ERANGE (see "Device status words"; the caller zeroes it first).
 * Limits: T*topk < INT_MAX, E_tot <= MR_MAX_SORT_EXPERTS, block_m >= 1.
 */
size_t moe_sort_capacity(int T, int topk, int E_tot, int block_m);
size_t moe_sort_workspace_bytes(int T, int topk, int E_tot, int block_m);
int moe_sort(const int32_t* topk_idx, const float* topk_w, int T, int topk, int E_tot,
             int block_m, int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids,
             int32_t* num_tokens_post_pad, void* workspace, size_t ws_bytes, int32_t* status,
             mr_stream_t stream);

/*
 * moe_sort_noalloc -- moe_sort without a workspace argument, for callers that cannot
 * allocate device memory: code that is handed only a stream and its tensors (an
 * inference-engine plugin or custom op with no allocator handle), or code that must
 * not call cudaMalloc/cudaFree because those synchronise the device or are not
 * allowed at that point. The pages have no counterpart; this is a convenience of
 * this library.
 *
 * Same arguments, layout, outputs and errors as moe_sort, minus workspace/ws_bytes.
 * Its scratch (the per-chunk expert-count table, moe_sort_workspace_bytes() bytes)
 * is a file-scope device array of MR_SORT_NOALLOC_SCRATCH_BYTES inside the library,
 * held on every GPU that loads the library until the process exits; a call whose
 * table would not fit returns MR_EUNSUPPORTED before anything is enqueued. The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * The first call on a device looks up the array's device address (a
 * cudaGetSymbolAddress with that device current) and caches it: make that first
 * call outside any stream capture. All calls on a device share the one array and
 * every call rewrites the part it uses, so nothing needs clearing between calls, but
 * calls whose work overlaps on the GPU (different streams, no ordering) race on it
 * and give wrong results: order them, or use moe_sort with separate workspaces.
 */
#define MR_SORT_NOALLOC_SCRATCH_BYTES (1u << 20)
/* The size of that array in bytes, as this build of the library has it (the value of
 * MR_SORT_NOALLOC_SCRATCH_BYTES it was compiled with), for callers that load the
 * library at run time. */
size_t moe_sort_noalloc_scratch_bytes(void);
int moe_sort_noalloc(const int32_t* topk_idx, const float* topk_w, int T, int topk, int E_tot,
                     int block_m, int32_t* sorted_token_ids, float* sorted_weights,
                     int32_t* expert_ids, int32_t* num_tokens_post_pad, int32_t* status,
                     mr_stream_t stream);

/*
 * moe_router_fused_fwd_sort -- moe_router_fwd (compact outputs) followed by moe_sort
 * over E_tot = E + n_shared experts ([FLY] fused top-k + sorting). With rows of
 * E <= MR_MAX_FUSED_EXPERTS it is ONE launch: of one CTA for T <= MR_MAX_FUSED_TOKENS
 * (a warp per token; up to 128 pairs one warp sorts them), and of one thread-block
 * cluster for MR_MAX_FUSED_TOKENS < T <= 512 where the device schedules such a cluster
 * (else one CTA up to T <= MR_MAX_FUSED_TOKENS_SMALL_E when E <= MR_MAX_FUSED_EXPERTS_SMALL).
 * Otherwise (the pages report no gain from fusing beyond T = 16 and leave larger T open)
 * it runs as the separate forward and sort launches. Results are the same in every form.
 * topk_idx / topk_w are nullable (compact outputs written only when given). The
 * workspace (moe_router_fused_workspace_bytes, 0 for the one-launch sizes) holds
 * the compact outputs when those are NULL and the sort's scratch (0 bytes for the
 * one-launch case).
 * status: nullable device int32, as for moe_router_fwd (MR_ETIMEOUT from the staged
 * wide-row forward when the call runs as separate launches).
 */
size_t moe_router_fused_workspace_bytes(const mr_router_params* p, int block_m);
int moe_router_fused_fwd_sort(const mr_router_params* p, const void* logits, int block_m,
                              int32_t* topk_idx, float* topk_w, int32_t* sorted_token_ids,
                              float* sorted_weights, int32_t* expert_ids,
                              int32_t* num_tokens_post_pad, void* workspace, size_t ws_bytes,
                              int32_t* status, mr_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_router_strerror(int code);

/*
 * Top-k path selection ([TE] NVTE_RADIX_TOPK_THRESHOLD): k_r < select_threshold takes
 * the repeated-arg-max register path, otherwise the threshold-select path. force_path:
 * 0 = by threshold, 1 = always arg-max, 2 = always threshold-select. Both paths give
 * bit-identical results. Defaults: threshold 8 (or env MR_TOPK_SELECT_THRESHOLD),
 * force from env MR_FORCE_PATH=argmax|select. Process-wide; not thread-safe against
 * concurrent calls. Returns MR_EINVAL for a negative threshold or unknown force_path.
 */
int moe_router_set_topk_path(int select_threshold, int force_path);

/*
 * The library's per-device status word. Kernels that wait on an asynchronous copy
 * (the forward on rows staged in shared memory) bound every wait; if one gives up
 * and the call had no status argument (or was moe_aux_scores_fwd), the kernel
 * raises this word to MR_ETIMEOUT and stops. This call enqueues, on `stream`, a copy
 * of the current device's word into *out (a device int32) and, if clear != 0, resets
 * the word to 0 after copying it. Asynchronous like every other call: *out is valid
 * once the stream reaches this point.
 * Returns MR_EINVAL for a NULL out, MR_ECUDA on a failed launch.
 */
int moe_router_device_status(int32_t* out, int clear, mr_stream_t stream);

/*
 * Launch overlap (programmatic dependent launch). enable = 1 (the default; the
 * environment variable MR_LAUNCH_OVERLAP=0 starts the process with it off):
 * every kernel of the library is launched so that it may start while the
 * previous kernel in the stream is still running; it does only its own set-up
 * (shared memory, barriers) and then waits for that kernel to complete before
 * it touches global memory, so results and stream order are unchanged and only
 * the launch latency is hidden. enable = 0: plain stream order. Process-wide,
 * read by every later launch. Returns MR_EINVAL for another value.
 */
int moe_router_set_launch_overlap(int enable);

/*
 * Test hook for the bounded waits ([TE] "Hardening": device-side guards report
 * instead of trapping). tries: attempts of about a microsecond each before a wait of
 * the staged wide-row forward gives up (0 restores the default of 2^20, about a
 * second). drop_copies != 0: the kernel arms each row's barrier for the bytes of
 * the row but issues no copy, so every wait runs out while no copy is in flight;
 * the kernel then reports MR_ETIMEOUT and returns, and the outputs are not valid.
 * Process-wide, read by every later launch; not thread-safe against concurrent
 * calls. Returns MR_EINVAL for drop_copies outside {0, 1}.
 */
int moe_router_set_wait_test(unsigned int tries, int drop_copies);

/* Diagnostics (not part of the routing path):
 * moe_router_expf evaluates the library's device fp32 exponential on n values
 *   (x, y: device fp32 [n]); used to check it bit-for-bit against its specification.
 * moe_router_exp_value evaluates the exponential the softmax forward uses for its
 *   numerators exp(x - max) on n values (defined for x <= 0; x, y: device fp32 [n]);
 *   used to check its error against exp in double precision.
 * moe_router_noop launches an empty kernel through the same path as the other calls:
 *   the launch-latency floor the fused decode call is measured against. */
int moe_router_expf(const float* x, float* y, int n, mr_stream_t stream);
int moe_router_exp_value(const float* x, float* y, int n, mr_stream_t stream);
int moe_router_noop(mr_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ROUTER_H */
