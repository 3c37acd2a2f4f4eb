// The steps on either side of the grouped GEMM: pack (token-major rows into
// the grouped, padded layout the forward reads) and combine (the k expert rows
// of every token summed back into token order).
//
// "moe_dispatch_contract.py" (TileLang tutorial, ch. 18), build_contract: the
// pairs are stably sorted by expert, so the pair of rank r inside expert e goes
// to padded row group_padded_offsets[e] + r and compact row group_offsets[e] + r
// ("Fused MoE GEMM 提交说明", §实现要点: x / out use padded rows, the routed
// weights compact rows).  "MetaX-TileLang工具链" §2.7: the pages pack with a
// Python loop and combine with a PyTorch scatter_reduce; here both are kernels.
//
// Pack runs in three launches:
//   1. rank_chunks_kernel: for each chunk of PACK_CHUNK (1024) pairs, every pair's
//      rank among the chunk's earlier pairs of the same expert (warp match_any
//      inside a warp, shared-memory per-warp counts across warps) and the
//      chunk's per-expert histogram (workspace);
//   2. scan_chunks_kernel: per expert (one warp each), exclusive prefix of the
//      histograms over chunks (in place);
//   3. place_pairs_kernel: row = padded[e] + chunk prefix + rank; writes the
//      pair's padded row, its routed weight at the compact index, and copies
//      the token's activation row (one warp per pair, 16-byte vectors).
// Combine: one CTA per token, fp32 sum over j = 0..k-1 in order, one rounding.
// Every launch here uses programmatic dependent launch: a kernel may start
// during the tail of the previous one on the stream, and waits for it
// (griddepcontrol.wait) before its first global access.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int RANK_THREADS = 1024;
constexpr int RANK_WARPS = RANK_THREADS / 32;
constexpr int PACK_CHUNK = RANK_THREADS;           // pairs per chunk (one pass per CTA)

__global__ void __launch_bounds__(RANK_THREADS)
rank_chunks_kernel(const int32_t* __restrict__ topk_ids, int64_t pairs, int32_t n_experts,
                   int32_t* __restrict__ local_rank, int32_t* __restrict__ chunk_hist, int32_t* status) {
    extern __shared__ int32_t sh[];
    int32_t* running = sh;                                    // [E] pairs of e seen so far in the chunk
    uint8_t* wcnt = reinterpret_cast<uint8_t*>(sh + n_experts);   // [RANK_WARPS][E] per-warp counts
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched with programmatic dependent launch: the shared-memory set-up
    // may overlap the previous kernel; global reads come after its completion
    pdl_launch_dependents();
    for (int e = tid; e < n_experts; e += RANK_THREADS) running[e] = 0;
    for (int i = tid; i < RANK_WARPS * n_experts; i += RANK_THREADS) wcnt[i] = 0;
    pdl_wait_prior_grid();
    __syncthreads();
    const int64_t chunk0 = static_cast<int64_t>(blockIdx.x) * PACK_CHUNK;
    bool bad = false;
    for (int r = 0; r < PACK_CHUNK / RANK_THREADS; ++r) {
        const int64_t f = chunk0 + r * RANK_THREADS + tid;
        int32_t e = -1;
        if (f < pairs) {
            e = __ldg(topk_ids + f);
            if (static_cast<uint32_t>(e) >= static_cast<uint32_t>(n_experts)) {
                bad = true;
                e = -1;
            }
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int32_t rank_w = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank_w == 0) wcnt[warp * n_experts + e] = static_cast<uint8_t>(__popc(peers));
        __syncthreads();
        if (e >= 0) {
            int32_t before = running[e];
            for (int w = 0; w < warp; ++w) before += wcnt[w * n_experts + e];
            local_rank[f] = before + rank_w;
        }
        __syncthreads();
        for (int ee = tid; ee < n_experts; ee += RANK_THREADS) {
            int32_t s = 0;
            for (int w = 0; w < RANK_WARPS; ++w) {
                s += wcnt[w * n_experts + ee];
                wcnt[w * n_experts + ee] = 0;
            }
            running[ee] += s;
        }
        __syncthreads();
    }
    for (int e = tid; e < n_experts; e += RANK_THREADS)
        chunk_hist[static_cast<int64_t>(blockIdx.x) * n_experts + e] = running[e];
    if (bad && status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
}

// One warp per expert: exclusive prefix of that expert's chunk histograms
// (in place), 32 chunks per step with a warp-shuffle scan.
__global__ void scan_chunks_kernel(int32_t* chunk_hist, int32_t n_chunks, int32_t n_experts) {
    const int32_t e = static_cast<int32_t>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait_prior_grid();
    if (e >= n_experts) return;
    int32_t carry = 0;
    for (int32_t c0 = 0; c0 < n_chunks; c0 += 32) {
        const int32_t c = c0 + lane;
        int32_t* p = chunk_hist + static_cast<int64_t>(c) * n_experts + e;
        const int32_t v = c < n_chunks ? *p : 0;
        int32_t incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        if (c < n_chunks) *p = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// One warp per pair.
__global__ void place_pairs_kernel(const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_weights,
                                   int64_t pairs, int32_t top_k, int32_t n_experts,
                                   const int32_t* __restrict__ local_rank, const int32_t* __restrict__ chunk_base,
                                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ padded,
                                   const uint16_t* __restrict__ x_tokens, int32_t hidden, int64_t rows_total,
                                   int64_t valid_total, uint16_t* __restrict__ x_packed,
                                   float* __restrict__ rw_compact, int32_t* __restrict__ pair_rows, int32_t* status) {
    const int64_t f = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait_prior_grid();
    if (f >= pairs) return;
    const int32_t e = __ldg(topk_ids + f);
    if (static_cast<uint32_t>(e) >= static_cast<uint32_t>(n_experts)) {
        if (lane == 0) pair_rows[f] = -1;
        return;
    }
    const int32_t c = static_cast<int32_t>(f / PACK_CHUNK);
    const int32_t rank = __ldg(chunk_base + static_cast<int64_t>(c) * n_experts + e) + __ldg(local_rank + f);
    const int64_t row = static_cast<int64_t>(__ldg(padded + e)) + rank;
    const int64_t compact = static_cast<int64_t>(__ldg(offsets + e)) + rank;
    if (row >= rows_total || compact >= valid_total) {
        if (lane == 0) {
            pair_rows[f] = -1;
            if (status) atomicOr(status, MOE_DEV_BAD_TABLE);
        }
        return;
    }
    // the pair lands inside its expert's padded range, before the padding rows
    MOE_DCHECK(row < __ldg(padded + e + 1) && rank >= 0, status);
    if (lane == 0) {
        pair_rows[f] = static_cast<int32_t>(row);
        if (rw_compact) rw_compact[compact] = __ldg(topk_weights + f);
    }
    if (x_packed) {
        // eight 16-byte loads in flight per lane before their stores
        const uint4* src = reinterpret_cast<const uint4*>(x_tokens + (f / top_k) * static_cast<int64_t>(hidden));
        uint4* dst = reinterpret_cast<uint4*>(x_packed + row * static_cast<int64_t>(hidden));
        const int32_t n16 = hidden / 8;
        for (int32_t i0 = 0; i0 < n16; i0 += 8 * 32) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t i = i0 + u * 32 + lane;
                if (i < n16) v[u] = __ldg(src + i);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t i = i0 + u * 32 + lane;
                if (i < n16) dst[i] = v[u];
            }
        }
    }
}

constexpr int COMBINE_THREADS = 256;

// One CTA per token; each thread sums 8 consecutive columns of the token's k
// expert rows in j order, with up to JB rows' loads in flight before the sums
// (JB follows top_k, so a small k keeps few registers and many CTAs per SM).
template <int JB>
__global__ void __launch_bounds__(COMBINE_THREADS)
combine_kernel(const uint16_t* __restrict__ out, int64_t rows_total, int32_t hidden,
               const int32_t* __restrict__ pair_rows, int32_t top_k, uint16_t* __restrict__ y) {
    const int64_t t = blockIdx.x;
    pdl_launch_dependents();
    pdl_wait_prior_grid();
    for (int32_t c8 = threadIdx.x; c8 < hidden / 8; c8 += COMBINE_THREADS) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int32_t j0 = 0; j0 < top_k; j0 += JB) {
            uint4 v[JB];
            bool ok[JB];
#pragma unroll
            for (int u = 0; u < JB; ++u) {
                const int32_t j = j0 + u;
                const int64_t row = j < top_k ? static_cast<int64_t>(__ldg(pair_rows + t * top_k + j)) : -1;
                ok[u] = row >= 0 && row < rows_total;
                if (ok[u]) v[u] = __ldg(reinterpret_cast<const uint4*>(out + row * hidden) + c8);
            }
#pragma unroll
            for (int u = 0; u < JB; ++u) {
                if (!ok[u]) continue;
                const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f2 = __half22float2(h[i]);
                    acc[2 * i] += f2.x;
                    acc[2 * i + 1] += f2.y;
                }
            }
        }
        uint4 o;
        __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) oh[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        reinterpret_cast<uint4*>(y + t * hidden)[c8] = o;
    }
}

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream finishes; every kernel here waits for it
// (griddepcontrol.wait) before its first global access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace

int64_t pack_workspace_bytes(int64_t pairs, int32_t n_experts) {
    const int64_t chunks = (pairs + PACK_CHUNK - 1) / PACK_CHUNK;
    // chunk histograms, then every pair's rank inside its chunk
    return 4 * (chunks * n_experts + pairs) + 256;
}

cudaError_t launch_pack(const int32_t* topk_ids, const float* topk_weights, int64_t n_tokens, int32_t top_k,
                        int32_t n_experts, const uint16_t* x_tokens, int32_t hidden, const int32_t* offsets,
                        const int32_t* padded, int64_t rows_total, int64_t valid_total, uint16_t* x_packed,
                        float* rw_compact, int32_t* pair_rows, void* workspace, int32_t* status,
                        cudaStream_t stream) {
    const int64_t pairs = n_tokens * top_k;
    if (pairs == 0) return cudaSuccess;
    const int32_t chunks = static_cast<int32_t>((pairs + PACK_CHUNK - 1) / PACK_CHUNK);
    int32_t* hist = static_cast<int32_t*>(workspace);
    int32_t* local_rank = hist + static_cast<int64_t>(chunks) * n_experts;
    const size_t smem = 4 * static_cast<size_t>(n_experts) + RANK_WARPS * static_cast<size_t>(n_experts);
    cudaError_t err = cudaFuncSetAttribute(rank_chunks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    if ((err = launch_pdl(rank_chunks_kernel, dim3(chunks), dim3(RANK_THREADS), smem, stream, topk_ids, pairs,
                          n_experts, local_rank, hist, status)) != cudaSuccess)
        return err;
    if ((err = launch_pdl(scan_chunks_kernel, dim3((n_experts + 7) / 8), dim3(256), 0, stream, hist, chunks,
                          n_experts)) != cudaSuccess)
        return err;
    const int64_t warps = pairs;
    const int64_t blocks = (warps * 32 + 255) / 256;
    return launch_pdl(place_pairs_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, topk_ids,
                      topk_weights, pairs, top_k, n_experts, local_rank, hist, offsets, padded, x_tokens, hidden,
                      rows_total, valid_total, x_packed, rw_compact, pair_rows, status);
}

cudaError_t launch_combine(const uint16_t* out, int64_t rows_total, int32_t hidden, const int32_t* pair_rows,
                           int64_t n_tokens, int32_t top_k, uint16_t* y, cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(n_tokens));
    auto kernel = top_k <= 2 ? combine_kernel<2> : top_k <= 4 ? combine_kernel<4> : combine_kernel<8>;
    return launch_pdl(kernel, grid, dim3(COMBINE_THREADS), 0, stream, out, rows_total, hidden, pair_rows, top_k, y);
}

}  // namespace moe
