// moe_fused_forward_static_workspace: the fused forward for callers that must
// not allocate device memory.
//
// moe_fused_forward needs an fp16 up_logits workspace of
// total_padded_tokens x intermediate elements, which the caller normally
// allocates.  Some callers cannot call cudaMalloc on the path that runs the
// forward: a plugin inside an inference runtime that owns every device
// allocation itself, or a latency-critical serving loop where cudaMalloc's
// possible device-wide synchronisation and its failure under memory pressure
// are not acceptable.  This entry point gives them a forward that allocates
// nothing: up_logits lives in a fixed array compiled into the library.
//
// The array below is a file-scope __device__ object: every GPU on which the
// library's module is loaded holds it (STATIC_UP_LOGITS_BYTES) until the
// process exits.  In host code its name is only a host-side stand-in, so the
// device address is looked up with cudaGetSymbolAddress, once per device with
// that device current, on the first call made on that device, and cached.
// The cache is not told about a device reset: after cudaDeviceReset (or any
// re-creation of the device's primary context) the cached address is stale,
// so this entry point must not be used across a reset.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"

namespace {

constexpr size_t STATIC_UP_LOGITS_BYTES = static_cast<size_t>(MOE_STATIC_WORKSPACE_BYTES);
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) uint16_t g_static_up_logits[STATIC_UP_LOGITS_BYTES / sizeof(uint16_t)];

std::mutex g_mutex;
void* g_addr[MAX_DEVICES] = {};

// Device address of g_static_up_logits on the current device (looked up once
// per device).  Returns nullptr if the lookup fails.
void* static_workspace_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_up_logits) != cudaSuccess) {
            cudaGetLastError();   // leave no pending error behind for the caller's next check
            return nullptr;
        }
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" moe_status_t moe_fused_forward_static_workspace(
    const uint16_t* stacked_expert_tokens, int64_t total_padded_tokens, int32_t hidden,
    const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w, int32_t n_experts,
    int32_t intermediate, const float* routed_expert_weights, int64_t total_valid_tokens,
    const int32_t* group_sizes, const int32_t* group_offsets, const int32_t* group_padded_offsets,
    const int32_t* group_idx_for_bx, int64_t num_blocks_m, uint16_t* out, int32_t* status_dev,
    void* stream) {
    // The checks every forward makes come first (same codes, same order as
    // moe_fused_forward), then the limit of the fixed workspace.
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
    a.out = out;
    if (moe_status_t s = moe::check_forward_args(a, false)) return s;
    const double need = static_cast<double>(total_padded_tokens) * intermediate * sizeof(uint16_t);
    if (need > static_cast<double>(STATIC_UP_LOGITS_BYTES)) return MOE_ERR_STATIC_WORKSPACE;
    void* ws = static_workspace_address();
    if (ws == nullptr) return MOE_ERR_DEVICE;
    // Nothing in the workspace has to start at zero: phase 1 writes every
    // valid row before phase 2 reads it, and rows phase 2 reads but phase 1
    // never wrote only feed padding rows, whose results are not stored.
    return moe_fused_forward(stacked_expert_tokens, total_padded_tokens, hidden, gate_w, up_w, down_w,
                             n_experts, intermediate, routed_expert_weights, total_valid_tokens,
                             group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                             num_blocks_m, static_cast<uint16_t*>(ws), out, status_dev, stream);
}
