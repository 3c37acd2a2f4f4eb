// C ABI of the library: argument validation and dispatch to the launchers.
// Every check here runs on the host before anything is enqueued; a failed
// check returns a MOE_ERR_* code and launches nothing.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"

namespace {

constexpr int32_t ABI_VERSION = 1;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_device() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_DEVICE;
    // The library is compiled for sm_103a only.
    if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
    return MOE_OK;
}

moe_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    if (e == cudaErrorNotSupported || e == cudaErrorNoDevice) return MOE_ERR_DEVICE;
    return MOE_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_NULL: return "MOE_ERR_NULL: a required pointer is NULL";
        case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: a size is negative, inconsistent or not a multiple of 128";
        case MOE_ERR_ALIGN: return "MOE_ERR_ALIGN: a pointer is not 16-byte aligned";
        case MOE_ERR_BLOCK: return "MOE_ERR_BLOCK: block_token must be 128";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: no usable sm_103 device or driver entry point";
        case MOE_ERR_LAUNCH: return "MOE_ERR_LAUNCH: a kernel launch failed";
        case MOE_ERR_LIMIT: return "MOE_ERR_LIMIT: n_experts or num_blocks_m above the library limits";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
        case MOE_ERR_STATIC_WORKSPACE:
            return "MOE_ERR_STATIC_WORKSPACE: total_padded_tokens * intermediate * 2 bytes exceeds the "
                   "library's fixed workspace (MOE_STATIC_WORKSPACE_BYTES)";
        default: return "unknown moe status";
    }
}

int64_t moe_num_blocks(int64_t pairs, int32_t n_experts, int32_t block_token) {
    if (pairs < 0 || n_experts < 0 || block_token <= 0) return -1;
    return (pairs + block_token - 1) / block_token + n_experts;
}

moe_status_t moe_build_dispatch(const int32_t* topk_ids, int64_t n_tokens, int32_t top_k,
                                int32_t n_experts, int32_t block_token, int32_t* group_sizes,
                                int32_t* group_offsets, int32_t* group_padded_offsets,
                                int32_t* group_idx_for_bx, int64_t num_blocks_m, int32_t* status_dev,
                                void* stream) {
    if (n_tokens < 0 || top_k <= 0) return MOE_ERR_SHAPE;
    if (block_token != MOE_BLOCK_TOKEN) return MOE_ERR_BLOCK;
    if (n_experts <= 0 || n_experts > MOE_MAX_EXPERTS) return MOE_ERR_LIMIT;
    const int64_t pairs = n_tokens * static_cast<int64_t>(top_k);
    if (num_blocks_m != moe_num_blocks(pairs, n_experts, block_token)) return MOE_ERR_SHAPE;
    if (num_blocks_m > MOE_MAX_BLOCKS) return MOE_ERR_LIMIT;
    if ((pairs > 0 && !topk_ids) || !group_sizes || !group_offsets || !group_padded_offsets ||
        !group_idx_for_bx)
        return MOE_ERR_NULL;
    if (moe_status_t s = check_device()) return s;
    return from_cuda(moe::launch_build_dispatch(topk_ids, pairs, n_experts, block_token, group_sizes,
                                                group_offsets, group_padded_offsets, group_idx_for_bx,
                                                num_blocks_m, status_dev,
                                                static_cast<cudaStream_t>(stream)));
}

int64_t moe_pack_workspace_bytes(int64_t pairs, int32_t n_experts) {
    if (pairs < 0 || n_experts <= 0) return -1;
    return moe::pack_workspace_bytes(pairs, n_experts);
}

moe_status_t moe_pack_routed(const int32_t* topk_ids, const float* topk_weights, int64_t n_tokens, int32_t top_k,
                             int32_t n_experts, const uint16_t* x_tokens, int32_t hidden,
                             const int32_t* group_offsets, const int32_t* group_padded_offsets,
                             int64_t total_padded_tokens, uint16_t* stacked_expert_tokens,
                             float* routed_expert_weights, int32_t* pair_padded_rows, void* workspace,
                             size_t workspace_bytes, int32_t* status_dev, void* stream) {
    if (n_tokens < 0 || top_k <= 0 || hidden <= 0 || hidden % 128 != 0 || total_padded_tokens < 0)
        return MOE_ERR_SHAPE;
    if (n_experts <= 0 || n_experts > MOE_MAX_EXPERTS) return MOE_ERR_LIMIT;
    const int64_t pairs = n_tokens * static_cast<int64_t>(top_k);
    if (pairs == 0) return MOE_OK;
    if (!topk_ids || !group_offsets || !group_padded_offsets || !pair_padded_rows) return MOE_ERR_NULL;
    if (stacked_expert_tokens && !x_tokens) return MOE_ERR_NULL;
    if (routed_expert_weights && !topk_weights) return MOE_ERR_NULL;
    if ((stacked_expert_tokens && (!aligned16(stacked_expert_tokens) || !aligned16(x_tokens))))
        return MOE_ERR_ALIGN;
    if (!workspace || static_cast<int64_t>(workspace_bytes) < moe::pack_workspace_bytes(pairs, n_experts))
        return MOE_ERR_WORKSPACE;
    if (moe_status_t s = check_device()) return s;
    return from_cuda(moe::launch_pack(topk_ids, topk_weights, n_tokens, top_k, n_experts, x_tokens, hidden,
                                      group_offsets, group_padded_offsets, total_padded_tokens, pairs,
                                      stacked_expert_tokens, routed_expert_weights, pair_padded_rows, workspace,
                                      status_dev, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine_routed(const uint16_t* out, int64_t total_padded_tokens, int32_t hidden,
                                const int32_t* pair_padded_rows, int64_t n_tokens, int32_t top_k, uint16_t* y,
                                void* stream) {
    if (n_tokens < 0 || top_k <= 0 || hidden <= 0 || hidden % 128 != 0 || total_padded_tokens < 0)
        return MOE_ERR_SHAPE;
    if (n_tokens == 0) return MOE_OK;
    if (!out || !pair_padded_rows || !y) return MOE_ERR_NULL;
    if (!aligned16(out) || !aligned16(y)) return MOE_ERR_ALIGN;
    if (moe_status_t s = check_device()) return s;
    return from_cuda(moe::launch_combine(out, total_padded_tokens, hidden, pair_padded_rows, n_tokens, top_k, y,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_router_topk(const uint16_t* x_tokens, int64_t n_tokens, int32_t hidden,
                             const uint16_t* router_w, int32_t n_experts, int32_t top_k, int32_t* topk_ids,
                             float* topk_weights, int32_t* status_dev, void* stream) {
    if (n_tokens < 0 || hidden <= 0 || hidden % 128 != 0) return MOE_ERR_SHAPE;
    if (n_experts <= 0 || n_experts > MOE_ROUTER_MAX_EXPERTS) return MOE_ERR_LIMIT;
    if (top_k <= 0 || top_k > n_experts || top_k > MOE_ROUTER_MAX_TOPK) return MOE_ERR_LIMIT;
    if (n_tokens == 0) return MOE_OK;
    if (!x_tokens || !router_w || !topk_ids || !topk_weights) return MOE_ERR_NULL;
    if (!aligned16(x_tokens) || !aligned16(router_w)) return MOE_ERR_ALIGN;
    if (moe_status_t s = check_device()) return s;
    return from_cuda(moe::launch_router(x_tokens, n_tokens, hidden, router_w, n_experts, top_k, topk_ids,
                                        topk_weights, status_dev, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace moe {

int32_t check_forward_args(const ForwardArgs& a, bool check_up_logits) {
    if (!a.x || !a.gate_w || !a.up_w || !a.down_w || (a.valid_total > 0 && !a.rw) || !a.sizes || !a.offsets ||
        !a.padded || !a.gidx || (check_up_logits && !a.up_logits) || !a.out)
        return MOE_ERR_NULL;
    if (a.hidden <= 0 || a.intermediate <= 0 || a.hidden % 128 != 0 || a.intermediate % 128 != 0)
        return MOE_ERR_SHAPE;
    if (a.rows_total < 0 || a.valid_total < 0 || a.num_blocks_m < 0) return MOE_ERR_SHAPE;
    if (a.n_experts <= 0 || a.n_experts > MOE_MAX_EXPERTS) return MOE_ERR_LIMIT;
    if (a.num_blocks_m > MOE_MAX_BLOCKS) return MOE_ERR_LIMIT;
    if (a.rows_total < a.num_blocks_m * MOE_BLOCK_TOKEN) return MOE_ERR_SHAPE;
    if (!aligned16(a.x) || !aligned16(a.gate_w) || !aligned16(a.up_w) || !aligned16(a.down_w) ||
        (check_up_logits && !aligned16(a.up_logits)) || !aligned16(a.out))
        return MOE_ERR_ALIGN;
    return MOE_OK;
}

}  // namespace moe

namespace {

moe_status_t forward_impl(const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens, int32_t hidden,
                          const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w, int32_t n_experts,
                          int32_t intermediate, const float* routed_expert_weights, int64_t total_valid_tokens,
                          const int32_t* group_sizes, const int32_t* group_offsets,
                          const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx,
                          int64_t num_blocks_m, uint16_t* up_logits, uint16_t* out, int32_t* status_dev,
                          void* stream, uint32_t flags, void* ready_ws) {
    const uint32_t phases = flags & (MOE_RUN_PHASE1 | MOE_RUN_PHASE2);
    if (phases == 0 || (flags & ~(MOE_RUN_PHASE1 | MOE_RUN_PHASE2 | MOE_NO_PDL | MOE_TEST_DROP_SIGNAL)) != 0)
        return MOE_ERR_SHAPE;
    moe::ForwardArgs a{};
    a.x = stacked_expert_tokens;
    a.rows_total = total_padded_tokens;
    a.hidden = hidden;
    a.gate_w = gate_w;
    a.up_w = up_w;
    a.down_w = down_w;
    a.n_experts = n_experts;
    a.intermediate = intermediate;
    a.rw = routed_expert_weights;
    a.valid_total = total_valid_tokens;
    a.sizes = group_sizes;
    a.offsets = group_offsets;
    a.padded = group_padded_offsets;
    a.gidx = group_idx_for_bx;
    a.num_blocks_m = num_blocks_m;
    a.up_logits = up_logits;
    a.out = out;
    a.status = status_dev;
    if (moe_status_t s = moe::check_forward_args(a, true)) return s;
    if (moe_status_t s = check_device()) return s;
    if (num_blocks_m == 0) return MOE_OK;
    return from_cuda(moe::launch_fused_forward(a, flags, static_cast<cudaStream_t>(stream), ready_ws));
}

}  // namespace

extern "C" {

moe_status_t moe_fused_forward_ex(const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens,
                                  int32_t hidden, const uint16_t* gate_w, const uint16_t* up_w,
                                  const uint16_t* down_w, int32_t n_experts, int32_t intermediate,
                                  const float* routed_expert_weights, int64_t total_valid_tokens,
                                  const int32_t* group_sizes, const int32_t* group_offsets,
                                  const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx,
                                  int64_t num_blocks_m, uint16_t* up_logits, uint16_t* out,
                                  int32_t* status_dev, void* stream, uint32_t flags) {
    return forward_impl(stacked_expert_tokens, total_padded_tokens, hidden, gate_w, up_w, down_w, n_experts,
                        intermediate, routed_expert_weights, total_valid_tokens, group_sizes, group_offsets,
                        group_padded_offsets, group_idx_for_bx, num_blocks_m, up_logits, out, status_dev, stream,
                        flags, nullptr);
}

int64_t moe_single_launch_workspace_bytes(int64_t num_blocks_m) {
    if (num_blocks_m < 0) return -1;
    return moe::single_launch_workspace_bytes(num_blocks_m);
}

moe_status_t moe_fused_forward_single_launch(
    const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens, int32_t hidden, const uint16_t* gate_w,
    const uint16_t* up_w, const uint16_t* down_w, int32_t n_experts, int32_t intermediate,
    const float* routed_expert_weights, int64_t total_valid_tokens, const int32_t* group_sizes,
    const int32_t* group_offsets, const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx,
    int64_t num_blocks_m, uint16_t* up_logits, uint16_t* out, void* workspace, size_t workspace_bytes,
    int32_t* status_dev, void* stream) {
    if (num_blocks_m < 0) return MOE_ERR_SHAPE;
    if (!workspace || static_cast<int64_t>(workspace_bytes) < moe::single_launch_workspace_bytes(num_blocks_m))
        return MOE_ERR_WORKSPACE;
    return forward_impl(stacked_expert_tokens, total_padded_tokens, hidden, gate_w, up_w, down_w, n_experts,
                        intermediate, routed_expert_weights, total_valid_tokens, group_sizes, group_offsets,
                        group_padded_offsets, group_idx_for_bx, num_blocks_m, up_logits, out, status_dev, stream,
                        MOE_RUN_PHASE1 | MOE_RUN_PHASE2, workspace);
}

moe_status_t moe_fused_forward(const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens,
                               int32_t hidden, const uint16_t* gate_w, const uint16_t* up_w,
                               const uint16_t* down_w, int32_t n_experts, int32_t intermediate,
                               const float* routed_expert_weights, int64_t total_valid_tokens,
                               const int32_t* group_sizes, const int32_t* group_offsets,
                               const int32_t* group_padded_offsets, const int32_t* group_idx_for_bx,
                               int64_t num_blocks_m, uint16_t* up_logits, uint16_t* out,
                               int32_t* status_dev, void* stream) {
    return moe_fused_forward_ex(stacked_expert_tokens, total_padded_tokens, hidden, gate_w, up_w, down_w,
                                n_experts, intermediate, routed_expert_weights, total_valid_tokens,
                                group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                                num_blocks_m, up_logits, out, status_dev, stream,
                                MOE_RUN_PHASE1 | MOE_RUN_PHASE2);
}

}  // extern "C"
