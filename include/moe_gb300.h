/*
 * moe_gb300.h — C ABI of the routed fused-MoE expert GEMM for GB300 (sm_103a).
 *
 * Token rows arrive grouped by expert and padded to 128-row blocks, described
 * by four int32 dispatch tables.  For every valid row p of expert e
 *
 *     up_logits[p, :] = fp16( silu(x[p]·gate_w[e]ᵀ) ⊙ (x[p]·up_w[e]ᵀ) )
 *     out[p, :]       = fp16( (up_logits[p]·down_w[e]ᵀ) · routed_expert_weights[c] )
 *
 * with fp32 accumulation, c = group_offsets[e] + (p - group_padded_offsets[e])
 * the row's compact index, and padding rows neither computed nor written.
 * Source: "Fused MoE GEMM 提交说明", §算子来源 (the expert MLP), §实现要点
 * (padded vs compact indexing, padding rows untouched), §完整算子代码 (the
 * run_kernel argument list, block_token = 128, fp16 data with fp32
 * accumulation, up_logits as an fp16 workspace); "moe_dispatch_contract.py"
 * (TileLang tutorial, ch. 18) for the four tables; "MetaX-TileLang工具链"
 * §1.9 for the two launches and their arguments.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - fp16 data is passed as `uint16_t` bit patterns (IEEE binary16).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous: it validates its arguments on the host, enqueues
 *     kernels and returns without synchronising.
 *   - A negative return value (MOE_ERR_*) means nothing was enqueued.
 *   - `status_dev` (nullable) is a device int32 into which kernels OR
 *     MOE_DEV_* bits when they meet inconsistent data (an expert id or table
 *     entry out of range, a bounded wait that ran out).  Offending work items
 *     are skipped; kernels never trap.  The caller zeroes it and reads it back.
 *   - Shapes are limited to hidden % 128 == 0, intermediate % 128 == 0,
 *     block_token == 128, 1 <= n_experts <= MOE_MAX_EXPERTS,
 *     num_blocks_m <= MOE_MAX_BLOCKS.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status_t;

#define MOE_OK            0
#define MOE_ERR_NULL     -1  /* a required pointer is NULL                          */
#define MOE_ERR_SHAPE    -2  /* a size is negative, inconsistent or not a multiple of 128 */
#define MOE_ERR_ALIGN    -3  /* a pointer is not 16-byte aligned (TMA needs it)      */
#define MOE_ERR_BLOCK    -4  /* block_token != 128                                   */
#define MOE_ERR_DEVICE   -5  /* no usable sm_103 device / driver entry point         */
#define MOE_ERR_LAUNCH   -6  /* a kernel launch failed (cudaGetLastError)            */
#define MOE_ERR_LIMIT    -7  /* n_experts or num_blocks_m above the library limits   */
#define MOE_ERR_WORKSPACE -8 /* workspace missing or smaller than required           */
#define MOE_ERR_STATIC_WORKSPACE -9 /* problem larger than the library's fixed workspace */

/* Bits OR-ed into *status_dev by kernels. */
#define MOE_DEV_BAD_EXPERT_ID 0x1  /* a topk id outside [0, n_experts)                 */
#define MOE_DEV_BAD_TABLE     0x2  /* a table entry points outside its array           */
#define MOE_DEV_TIMEOUT       0x4  /* a bounded pipeline wait ran out; tiles skipped    */
#define MOE_DEV_DEBUG_CHECK   0x8  /* MOE_DEBUG builds only: a kernel's own check of an
                                      index, coordinate or shared-memory canary failed */

#define MOE_BLOCK_TOKEN  128
#define MOE_MAX_EXPERTS  1024
#define MOE_MAX_BLOCKS   16384

/* Version of this ABI (bumped on any incompatible change). */
int32_t moe_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* Number of 128-row blocks of the padded layout:
 *     ceil(pairs / block_token) + n_experts
 * ("moe_dispatch_contract.py", build_contract step 4; "MetaX-TileLang工具链"
 * §1.9: M = ceil(group_sum / block_token) + group_count).  Every expert owns at
 * least one block because of the "+1" padding rule, so this bounds the padded
 * row count.  Returns -1 for negative arguments or block_token <= 0. */
int64_t moe_num_blocks(int64_t pairs, int32_t n_experts, int32_t block_token);

/* Build the four dispatch tables on the GPU from routing choices
 * ("moe_dispatch_contract.py", docstring and build_contract).
 *   topk_ids              [n_tokens, top_k] int32, row-major; the flat pair
 *                         index is t*top_k + j.  Ids must lie in [0, n_experts).
 *   group_sizes           [n_experts]   out: pairs routed to each expert
 *   group_offsets         [n_experts+1] out: exclusive prefix sum of the sizes
 *                         (compact rows); entry n_experts = total pairs
 *   group_padded_offsets  [n_experts+1] out: exclusive prefix sum of
 *                         ceil((size+1)/block_token)*block_token (padded rows);
 *                         entry n_experts = total padded rows
 *   group_idx_for_bx      [num_blocks_m] out: for block bx, the last expert e
 *                         with group_padded_offsets[e] <= bx*block_token
 *   num_blocks_m          must equal moe_num_blocks(n_tokens*top_k, n_experts, block_token)
 * Out-of-range ids are not counted and set MOE_DEV_BAD_EXPERT_ID.  One kernel
 * launch; no workspace. */
moe_status_t moe_build_dispatch(const int32_t* topk_ids, int64_t n_tokens, int32_t top_k,
                                int32_t n_experts, int32_t block_token,
                                int32_t* group_sizes, int32_t* group_offsets,
                                int32_t* group_padded_offsets, int32_t* group_idx_for_bx,
                                int64_t num_blocks_m, int32_t* status_dev, void* stream);

/* The fused forward: phase 1 (grouped gate+up GEMM, SiLU·up epilogue into the
 * fp16 up_logits workspace) then phase 2 (grouped down GEMM, routed weight
 * applied to the fp32 accumulator, fp16 store) — "Fused MoE GEMM 提交说明",
 * §完整算子代码, the page's run_kernel contract plus the explicit up_logits
 * argument of "MetaX-TileLang工具链" §1.9.
 *   stacked_expert_tokens [total_padded_tokens, hidden] fp16, padded rows
 *   gate_w, up_w          [n_experts, intermediate, hidden] fp16
 *   down_w                [n_experts, hidden, intermediate] fp16
 *   routed_expert_weights [total_valid_tokens] fp32, compact (expert-sorted) order
 *                         (may be NULL when total_valid_tokens == 0)
 *   group_*               the four tables above (only entries [0, n_experts) of
 *                         group_offsets / group_padded_offsets are read)
 *   up_logits             [total_padded_tokens, intermediate] fp16 workspace
 *   out                   [total_padded_tokens, hidden] fp16
 * Requirements: total_padded_tokens >= num_blocks_m*128; hidden and
 * intermediate multiples of 128; every pointer 16-byte aligned.  Rows that are
 * not valid rows of some block are never written, in up_logits or out.
 * Two kernel launches on `stream` (the second with programmatic dependent
 * launch); no workspace beyond up_logits. */
moe_status_t moe_fused_forward(const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens,
                               int32_t hidden,
                               const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
                               int32_t n_experts, int32_t intermediate,
                               const float* routed_expert_weights, int64_t total_valid_tokens,
                               const int32_t* group_sizes, const int32_t* group_offsets,
                               const int32_t* group_padded_offsets,
                               const int32_t* group_idx_for_bx, int64_t num_blocks_m,
                               uint16_t* up_logits, uint16_t* out,
                               int32_t* status_dev, void* stream);

/* Workspace bytes moe_pack_routed needs for `pairs` (token, expert) pairs
 * (per-chunk expert histograms and every pair's rank inside its chunk).
 * Returns -1 for invalid arguments. */
int64_t moe_pack_workspace_bytes(int64_t pairs, int32_t n_experts);

/* Pack: place every (token, expert) pair in the grouped, padded layout that
 * moe_fused_forward reads.  Pairs are stably sorted by expert
 * ("moe_dispatch_contract.py", build_contract), so the pair of rank r inside
 * expert e (counting pairs in flat order t*top_k + j) goes to padded row
 * group_padded_offsets[e] + r and compact index group_offsets[e] + r
 * ("Fused MoE GEMM 提交说明", §实现要点).
 *   topk_ids, topk_weights  [n_tokens, top_k] int32 / fp32 (weights may be NULL
 *                           when routed_expert_weights is NULL)
 *   x_tokens                [n_tokens, hidden] fp16 (may be NULL when
 *                           stacked_expert_tokens is NULL)
 *   group_offsets, group_padded_offsets  the tables of moe_build_dispatch
 *   stacked_expert_tokens   out, nullable: [total_padded_tokens, hidden]; row
 *                           pair_padded_rows[f] receives x_tokens[f / top_k];
 *                           padding rows are not written
 *   routed_expert_weights   out, nullable: [n_tokens*top_k] fp32, compact order
 *   pair_padded_rows        out: [n_tokens, top_k] int32 padded row of every
 *                           pair (-1 for an id outside [0, n_experts))
 *   workspace               device scratch of moe_pack_workspace_bytes() bytes
 * Three kernel launches; an out-of-range id sets MOE_DEV_BAD_EXPERT_ID. */
moe_status_t moe_pack_routed(const int32_t* topk_ids, const float* topk_weights, int64_t n_tokens,
                             int32_t top_k, int32_t n_experts, const uint16_t* x_tokens, int32_t hidden,
                             const int32_t* group_offsets, const int32_t* group_padded_offsets,
                             int64_t total_padded_tokens, uint16_t* stacked_expert_tokens,
                             float* routed_expert_weights, int32_t* pair_padded_rows,
                             void* workspace, size_t workspace_bytes, int32_t* status_dev, void* stream);

/* Combine: y[t, :] = fp16( sum over j = 0..top_k-1, in that order, of
 * out[pair_padded_rows[t*top_k + j], :] ) with the sum in fp32 and one
 * round-to-nearest-even.  The pages combine with a PyTorch scatter_reduce
 * ("MetaX-TileLang工具链", §2.7); the routed weight is already inside `out`.
 *   out               [total_padded_tokens, hidden] fp16 (moe_fused_forward's)
 *   pair_padded_rows  [n_tokens, top_k] int32 (moe_pack_routed's); negative
 *                     entries are skipped
 *   y                 out: [n_tokens, hidden] fp16
 * One kernel launch. */
moe_status_t moe_combine_routed(const uint16_t* out, int64_t total_padded_tokens, int32_t hidden,
                                const int32_t* pair_padded_rows, int64_t n_tokens, int32_t top_k,
                                uint16_t* y, void* stream);

#define MOE_ROUTER_MAX_EXPERTS 256
#define MOE_ROUTER_MAX_TOPK    16

/* Router ("MetaX-TileLang工具链", §2.4: logits = W_g(x), scores =
 * softmax(logits), topk_scores, topk_indices = topk(scores)).
 *   x_tokens      [n_tokens, hidden] fp16
 *   router_w      [n_experts, hidden] fp16 (W_g; a logit is a row of W_g
 *                 dotted with the token, accumulated in fp32)
 *   topk_ids      out: [n_tokens, top_k] int32, the top_k experts by logit in
 *                 descending order; equal logits: the lower expert index first
 *   topk_weights  out: [n_tokens, top_k] fp32, their softmax probabilities over
 *                 all n_experts (not renormalised over the k)
 * Limits: hidden % 128 == 0, n_experts <= MOE_ROUTER_MAX_EXPERTS, top_k <=
 * min(n_experts, MOE_ROUTER_MAX_TOPK).  One kernel launch: a tcgen05 MMA tile
 * of 128 tokens x all experts per cluster of 1-8 CTAs (hidden split over the
 * cluster when there are fewer tiles than SMs), softmax and top-k in its
 * epilogue.  Every wait inside it is bounded (2 s); one that runs out sets
 * MOE_DEV_TIMEOUT in status_dev (nullable) and leaves the outputs invalid. */
moe_status_t moe_router_topk(const uint16_t* x_tokens, int64_t n_tokens, int32_t hidden,
                             const uint16_t* router_w, int32_t n_experts, int32_t top_k,
                             int32_t* topk_ids, float* topk_weights, int32_t* status_dev, void* stream);

/* Flags of moe_fused_forward_ex. */
#define MOE_RUN_PHASE1   0x1u  /* gate+up GEMM and SiLU·up epilogue into up_logits   */
#define MOE_RUN_PHASE2   0x2u  /* down GEMM and routed-weight epilogue into out       */
#define MOE_NO_PDL       0x4u  /* launch phase 2 without programmatic dependent launch */
/* Test of the failure path: phase 1's MMA issuer skips its first "accumulator
 * ready" signal, so an epilogue wait runs out after its bound (2 s); the
 * kernel then stops, frees its resources and reports MOE_DEV_TIMEOUT in
 * status_dev.  The outputs of such a call are not valid. */
#define MOE_TEST_DROP_SIGNAL 0x100u

/* moe_fused_forward with a choice of phases: `flags` is a combination of
 * MOE_RUN_PHASE1 / MOE_RUN_PHASE2 (at least one) and optionally MOE_NO_PDL.
 * Running phase 2 alone reads up_logits as left by an earlier phase 1 on the
 * same tables (for example to time each phase by itself).  Same arguments,
 * requirements and errors as moe_fused_forward, which is this call with
 * flags = MOE_RUN_PHASE1 | MOE_RUN_PHASE2. */
moe_status_t moe_fused_forward_ex(const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens,
                                  int32_t hidden,
                                  const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
                                  int32_t n_experts, int32_t intermediate,
                                  const float* routed_expert_weights, int64_t total_valid_tokens,
                                  const int32_t* group_sizes, const int32_t* group_offsets,
                                  const int32_t* group_padded_offsets,
                                  const int32_t* group_idx_for_bx, int64_t num_blocks_m,
                                  uint16_t* up_logits, uint16_t* out,
                                  int32_t* status_dev, void* stream, uint32_t flags);

/* Workspace bytes of moe_fused_forward_single_launch (one int32 counter per
 * 128-row block, rounded up).  Returns -1 for a negative argument. */
int64_t moe_single_launch_workspace_bytes(int64_t num_blocks_m);

/* moe_fused_forward with both phases in ONE persistent launch (same
 * arguments, results and errors, plus a workspace).  Each cluster of two CTAs
 * runs its phase-1 tiles, then its phase-2 tiles; a phase-2 tile of a unit of
 * blocks starts as soon as every phase-1 tile of that unit has stored its
 * up_logits rows (per-unit counters in `workspace`, zeroed by this call with a
 * cudaMemsetAsync on `stream`), so the phase-1 tail and the kernel boundary
 * overlap phase-2 work.  The waits are bounded (MOE_DEV_TIMEOUT) and need all
 * clusters of the launch resident at once, which the grid size ensures when
 * no other kernel holds SMs for long.  Workspace: device memory of
 * moe_single_launch_workspace_bytes(num_blocks_m) bytes, caller-owned; calls
 * that overlap on the GPU must not share it. */
moe_status_t moe_fused_forward_single_launch(
    const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens, int32_t hidden,
    const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
    int32_t n_experts, int32_t intermediate,
    const float* routed_expert_weights, int64_t total_valid_tokens,
    const int32_t* group_sizes, const int32_t* group_offsets,
    const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx, int64_t num_blocks_m,
    uint16_t* up_logits, uint16_t* out, void* workspace, size_t workspace_bytes,
    int32_t* status_dev, void* stream);

/* Size of the fixed workspace used by moe_fused_forward_static_workspace. */
#define MOE_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)

/* The fused forward for callers that cannot allocate device memory (the pages
 * have no counterpart of this call).  A plugin inside an inference runtime
 * that owns every device allocation, or a latency-critical serving loop that
 * cannot afford cudaMalloc's possible device-wide synchronisation or its
 * failure under memory pressure, cannot provide the up_logits workspace that
 * moe_fused_forward needs.  This call takes the same arguments without
 * up_logits and keeps that workspace in a fixed array compiled into the
 * library: every GPU that loads the library holds MOE_STATIC_WORKSPACE_BYTES
 * (64 MiB) of device memory for it until the process exits.
 *   - Limit: total_padded_tokens * intermediate * 2 bytes must not exceed
 *     MOE_STATIC_WORKSPACE_BYTES; larger problems return
 *     MOE_ERR_STATIC_WORKSPACE and nothing is enqueued.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that
 *     first call before any stream capture.  The cache does not survive a
 *     device reset: do not use this call across cudaDeviceReset.
 *   - Argument checks: first the ones moe_fused_forward makes (same codes,
 *     same order), then the workspace limit (MOE_ERR_STATIC_WORKSPACE).
 *   - All calls in the process share the one array per device and it keeps
 *     the last call's contents.  Nothing in it has to start at zero.  Calls
 *     whose kernels overlap on the GPU (different streams, no ordering between
 *     them) race on the array and give wrong results; order them.
 * Otherwise the same arguments, requirements, results and errors as
 * moe_fused_forward. */
moe_status_t moe_fused_forward_static_workspace(
    const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens, int32_t hidden,
    const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
    int32_t n_experts, int32_t intermediate,
    const float* routed_expert_weights, int64_t total_valid_tokens,
    const int32_t* group_sizes, const int32_t* group_offsets,
    const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx, int64_t num_blocks_m,
    uint16_t* out, int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
