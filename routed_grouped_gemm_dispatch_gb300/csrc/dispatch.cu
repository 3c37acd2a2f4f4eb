// Dispatch-table builder: histogram + exclusive scans + block -> expert map,
// in one CTA ("moe_dispatch_contract.py", TileLang tutorial ch. 18: module
// docstring and build_contract; the padded step is ceil((count+1)/padding_M) *
// padding_M with padding_M = block_token).
//
// One CTA of 1024 threads: the counts of up to MOE_MAX_EXPERTS experts live in
// shared memory (for at most 256 experts one histogram per warp, summed
// afterwards, so that a popular expert's increments do not all queue on one
// address), the scans are warp-shuffle scans over one expert per thread,
// and each block finds its expert by binary search over the padded offsets
// (the page scans linearly; both give the last expert whose padded start is
// <= bx * block_token).  No workspace and no host synchronisation: the tables
// never leave the device.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int DISPATCH_THREADS = 1024;
constexpr int PRIV_EXPERTS = 256;   // per-warp histograms up to this many experts

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

__global__ void __launch_bounds__(DISPATCH_THREADS)
build_dispatch_kernel(const int32_t* __restrict__ topk_ids, int64_t pairs, int32_t n_experts,
                      int32_t block_token, int32_t* __restrict__ sizes, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ padded, int32_t* __restrict__ gidx, int64_t num_blocks_m,
                      int32_t* status) {
    __shared__ int32_t cnt[MOE_MAX_EXPERTS];
    __shared__ int32_t pad_s[MOE_MAX_EXPERTS + 1];
    __shared__ int32_t wsum_c[DISPATCH_THREADS / 32];
    __shared__ int32_t wsum_p[DISPATCH_THREADS / 32];
    __shared__ int32_t hist_w[DISPATCH_THREADS / 32][PRIV_EXPERTS];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // A forward launched right behind this kernel may start its own set-up
    // now; it reads the tables only after this grid has completed.
    pdl_launch_dependents();
    // This kernel is itself launched with programmatic dependent launch, so
    // it may start during the tail of the previous kernel on the stream (for
    // example the previous step's phase 2, which still reads the tables, or a
    // router that writes topk_ids).  Only the shared-memory set-up overlaps
    // that kernel: griddepcontrol.wait is the one point after which its
    // writes are visible, so every global read and write comes after it.
    const bool priv = n_experts <= PRIV_EXPERTS;
    if (priv) {
        for (int i = tid; i < (DISPATCH_THREADS / 32) * PRIV_EXPERTS; i += DISPATCH_THREADS)
            (&hist_w[0][0])[i] = 0;
    } else {
        for (int e = tid; e < n_experts; e += DISPATCH_THREADS) cnt[e] = 0;
    }
    pdl_wait_prior_grid();
    __syncthreads();

    // histogram of the flattened expert ids: 16-byte loads, eight per thread
    // in flight before their atomics, so a few memory round trips cover the
    // whole input; a scalar loop takes the unaligned case and the tail
    bool bad = false;
    int32_t* hist = priv ? hist_w[warp] : cnt;
    auto count = [&](int32_t v) {
        if (static_cast<uint32_t>(v) < static_cast<uint32_t>(n_experts)) atomicAdd(&hist[v], 1);
        else bad = true;
    };
    int64_t done = 0;
    if ((reinterpret_cast<uintptr_t>(topk_ids) & 15) == 0) {
        constexpr int U = 8;
        const int64_t n4 = pairs / 4;
        const int4* ids4 = reinterpret_cast<const int4*>(topk_ids);
        for (int64_t base = 0; base < n4; base += U * DISPATCH_THREADS) {
            int4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + u * DISPATCH_THREADS + tid;
                if (i < n4) v[u] = __ldg(ids4 + i);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (base + u * DISPATCH_THREADS + tid < n4) {
                    count(v[u].x);
                    count(v[u].y);
                    count(v[u].z);
                    count(v[u].w);
                }
            }
        }
        done = 4 * n4;
    }
    for (int64_t f = done + tid; f < pairs; f += DISPATCH_THREADS) count(__ldg(topk_ids + f));
    if (bad && status) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();
    if (priv) {
        for (int e = tid; e < n_experts; e += DISPATCH_THREADS) {
            int32_t sum = 0;
#pragma unroll 8
            for (int w = 0; w < DISPATCH_THREADS / 32; ++w) sum += hist_w[w][e];
            cnt[e] = sum;
        }
        __syncthreads();
    }

    // exclusive scans of the counts (compact offsets) and of the padded steps
    const int e = tid;                                  // n_experts <= 1024 threads
    const int32_t c = e < n_experts ? cnt[e] : 0;
    const int32_t step = e < n_experts ? ((c + 1 + block_token - 1) / block_token) * block_token : 0;
    const int32_t ic = warp_incl_scan(c, lane);
    const int32_t ip = warp_incl_scan(step, lane);
    if (lane == 31) {
        wsum_c[warp] = ic;
        wsum_p[warp] = ip;
    }
    __syncthreads();
    if (warp == 0) {
        const int32_t sc = warp_incl_scan(wsum_c[lane], lane);
        const int32_t sp = warp_incl_scan(wsum_p[lane], lane);
        wsum_c[lane] = sc;
        wsum_p[lane] = sp;
    }
    __syncthreads();
    const int32_t base_c = warp > 0 ? wsum_c[warp - 1] : 0;
    const int32_t base_p = warp > 0 ? wsum_p[warp - 1] : 0;
    const int32_t excl_c = base_c + ic - c;
    const int32_t excl_p = base_p + ip - step;
    if (e < n_experts) {
        sizes[e] = c;
        offsets[e] = excl_c;
        padded[e] = excl_p;
        pad_s[e] = excl_p;
    }
    if (e == n_experts - 1) {
        offsets[n_experts] = excl_c + c;
        padded[n_experts] = excl_p + step;
        pad_s[n_experts] = excl_p + step;
    }
    __syncthreads();

    // block -> expert: last e in [0, E) with pad_s[e] <= bx * block_token
    for (int64_t bx = tid; bx < num_blocks_m; bx += DISPATCH_THREADS) {
        const int64_t start = bx * block_token;
        int32_t lo = 0, hi = n_experts - 1;             // pad_s[0] = 0 <= start
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (static_cast<int64_t>(pad_s[mid]) <= start) lo = mid;
            else hi = mid - 1;
        }
        gidx[bx] = lo;
        // the found expert's padded range holds the block (or it is the last expert)
        MOE_DCHECK(lo >= 0 && lo < n_experts && pad_s[lo] <= start &&
                       (lo == n_experts - 1 || start < static_cast<int64_t>(pad_s[lo + 1])),
                   status);
    }
    // every padded range holds its rows plus at least one padding row, in whole blocks
    MOE_DCHECK(e >= n_experts || (excl_p % block_token == 0 && step >= c + 1), status);
}

}  // namespace

cudaError_t launch_build_dispatch(const int32_t* topk_ids, int64_t pairs, int32_t n_experts,
                                  int32_t block_token, int32_t* sizes, int32_t* offsets,
                                  int32_t* padded, int32_t* gidx, int64_t num_blocks_m,
                                  int32_t* status, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(DISPATCH_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, build_dispatch_kernel, topk_ids, pairs, n_experts, block_token, sizes, offsets,
                              padded, gidx, num_blocks_m, status);
}

}  // namespace moe
