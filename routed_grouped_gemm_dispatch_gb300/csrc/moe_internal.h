// Declarations shared by the translation units of the library (host side).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

// MOE_DEBUG builds (-DMOE_DEBUG=1) compile the kernels' own invariant checks;
// a failed one ORs MOE_DEV_DEBUG_CHECK into the status word and the kernel
// carries on (no trap).  In release builds the checks compile to nothing.
#ifndef MOE_DEBUG
#define MOE_DEBUG 0
#endif
#define MOE_DCHECK(cond, status_ptr)                                              \
    do {                                                                          \
        if (MOE_DEBUG && !(cond) && (status_ptr)) atomicOr((status_ptr), MOE_DEV_DEBUG_CHECK); \
    } while (0)

namespace moe {

struct ForwardArgs {
    const uint16_t* x;            // [rows_total, H]
    int64_t rows_total;
    int32_t hidden;
    const uint16_t* gate_w;       // [E, I, H]
    const uint16_t* up_w;         // [E, I, H]
    const uint16_t* down_w;       // [E, H, I]
    int32_t n_experts;
    int32_t intermediate;
    const float* rw;              // [valid_total]
    int64_t valid_total;
    const int32_t* sizes;
    const int32_t* offsets;
    const int32_t* padded;
    const int32_t* gidx;
    int64_t num_blocks_m;
    uint16_t* up_logits;          // [rows_total, I]
    uint16_t* out;                // [rows_total, H]
    int32_t* status;
};

// Host-side checks shared by the forward entry points: NULL pointers,
// shapes, library limits, padded row count and 16-byte alignment, in that
// order; the up_logits pointer only when `check_up_logits`.  Returns MOE_OK or
// the first MOE_ERR_* that applies.  No device call.
int32_t check_forward_args(const ForwardArgs& a, bool check_up_logits);

// Enqueue the dispatch-table builder.  Arguments already validated.
cudaError_t launch_build_dispatch(const int32_t* topk_ids, int64_t pairs, int32_t n_experts,
                                  int32_t block_token, int32_t* sizes, int32_t* offsets,
                                  int32_t* padded, int32_t* gidx, int64_t num_blocks_m,
                                  int32_t* status, cudaStream_t stream);

// Enqueue phase 1 and/or phase 2 (MOE_RUN_* flags).  Arguments already validated.  Returns
// cudaErrorNotSupported when the driver entry point for tensor maps is missing.
// With `ready_ws` (zeroed here, single_launch_workspace_bytes() bytes) and both
// phases requested, both phases run in one persistent launch.
cudaError_t launch_fused_forward(const ForwardArgs& a, uint32_t flags, cudaStream_t stream,
                                 void* ready_ws = nullptr);
int64_t single_launch_workspace_bytes(int64_t num_blocks_m);

// Pack: pair ranks, padded rows, compact routed weights, activation rows.
int64_t pack_workspace_bytes(int64_t pairs, int32_t n_experts);
cudaError_t launch_pack(const int32_t* topk_ids, const float* topk_weights, int64_t n_tokens, int32_t top_k,
                        int32_t n_experts, const uint16_t* x_tokens, int32_t hidden, const int32_t* offsets,
                        const int32_t* padded, int64_t rows_total, int64_t valid_total, uint16_t* x_packed,
                        float* rw_compact, int32_t* pair_rows, void* workspace, int32_t* status,
                        cudaStream_t stream);
// Combine: y[t] = fp16(sum_j out[pair_rows[t*k + j]]) in fp32, j in order.
cudaError_t launch_combine(const uint16_t* out, int64_t rows_total, int32_t hidden, const int32_t* pair_rows,
                           int64_t n_tokens, int32_t top_k, uint16_t* y, cudaStream_t stream);

// Router: logits, softmax, top-k.
cudaError_t launch_router(const uint16_t* x, int64_t n_tokens, int32_t hidden, const uint16_t* router_w,
                          int32_t n_experts, int32_t top_k, int32_t* topk_ids, float* topk_weights,
                          int32_t* status, cudaStream_t stream);

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

}  // namespace moe
