// Router: logits = x · W_gᵀ (fp32), softmax over all experts, top-k
// ("MetaX-TileLang工具链", §2.4: logits = W_g(x), scores = softmax(logits),
// topk_scores, topk_indices = topk(scores)).
//
// One cluster of S CTAs per 128-token tile, one tcgen05 MMA tile of M = 128
// tokens and N = n_experts rounded up to 16 (at most 256).  When there are
// fewer tiles than SMs the tile's K (hidden) is split over the S CTAs of its
// cluster, so that tiles x S SMs stream x instead of one per tile.  Warp 0
// streams the CTA's K range of x and W_g with TMA (4 stages of 64-wide K),
// warp 1 owns TMEM and issues the MMAs, warps 2-17 are the epilogue:
//  1. CTA r of the cluster owns tokens r*128/S .. (r+1)*128/S - 1 of the
//     tile.  Every CTA stores its fp32 logits (partial sums over its K range
//     when S > 1) from TMEM into its owners' shared memory, one slot per
//     source CTA (distributed shared memory stores, no round trips);
//  2. after a cluster barrier each owner sums the S slots of its tokens in
//     rank order, T consecutive lanes per token (expert e to lane e % T; T
//     the smaller of 4*S and n_pad / KMAX): every lane keeps a sorted list of
//     its best KMAX logits
//     (descending, ties to the lower expert index), built from bitonic sorts
//     of KMAX logits at a time; the token's lanes merge their lists in
//     butterfly rounds (a bitonic top-KMAX merge of two sorted lists), then
//     sum exp(l - max) against the known maximum and write the top-k.
// The top-k is decided on the logits (softmax preserves their order).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int R_BM = 128;
constexpr int R_BK = 64;
constexpr int R_STAGES = 4;
constexpr int R_A_BYTES = R_BM * R_BK * 2;           // 16 KB
constexpr int R_B_MAX_BYTES = 256 * R_BK * 2;        // 32 KB
constexpr int R_STAGE_BYTES = R_A_BYTES + R_B_MAX_BYTES;
constexpr int R_EPI_WARPS = 16;
constexpr int R_THREADS = 64 + 32 * R_EPI_WARPS;     // producer, MMA, epilogue warps
constexpr int R_MAX_E = 256;                         // MOE_ROUTER_MAX_EXPERTS
constexpr uint64_t R_WAIT_NS = 2000000000ull;
constexpr uint64_t R_DRAIN_NS = 200000000ull;
constexpr int R_OFF_BARS = R_STAGES * R_STAGE_BYTES;
constexpr int R_OFF_TMEM = R_OFF_BARS + (2 * R_STAGES + 2) * 8;
constexpr int R_OFF_ABORT = R_OFF_TMEM + 4;
constexpr size_t R_SMEM = 1024 + R_OFF_ABORT + 16;
constexpr int R_MAX_SPLIT = 8;   // CTAs per cluster (the portable cluster size)

static_assert(R_MAX_E == MOE_ROUTER_MAX_EXPERTS, "router expert limit");

struct RouterParams {
    int64_t n_tokens;
    int32_t n_experts;
    int32_t n_pad;         // n_experts rounded up to 16
    int32_t tmem_cols;     // power of two >= max(32, n_pad)
    int32_t top_k;
    int32_t k_blocks;      // hidden / 64
    int32_t lanes;         // T: lanes per token in the top-k (a power of two, 4*S at most)
    int32_t rs;            // slot_stride(S, T)
    int32_t* topk_ids;
    float* topk_weights;
    int32_t* status;
};

// Row stride of the owners' slots for S CTAs per cluster and T lanes per
// token: at least the 128 / S tokens a CTA owns, and congruent to 32 / T
// modulo 32, so that the 32 lanes of a warp (32 / T tokens x T experts) hit
// 32 banks.
__host__ __device__ constexpr int slot_stride(int S, int T) {
    return R_BM / S + (((32 / T - R_BM / S) % 32) + 32) % 32;
}

// (l, e) ranks above (lo, eo): a larger logit, or an equal one with a lower
// expert index (an empty entry is (-inf, INT_MAX))
__device__ __forceinline__ bool ranks_above(float l, int32_t e, float lo, int32_t eo) {
    return l > lo || (l == lo && e < eo);
}

// compare-exchange: the better of entries i and l ends at i
template <int K>
__device__ __forceinline__ void cex(float (&v)[K], int32_t (&e)[K], int i, int l) {
    if (ranks_above(v[l], e[l], v[i], e[i])) {
        const float tv = v[i];
        const int32_t te = e[i];
        v[i] = v[l];
        e[i] = e[l];
        v[l] = tv;
        e[l] = te;
    }
}

// bitonic sort into descending order (K a power of two, fully unrolled)
template <int K>
__device__ __forceinline__ void bitonic_sort_desc(float (&v)[K], int32_t (&e)[K]) {
#pragma unroll
    for (int k = 2; k <= K; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    if ((i & k) == 0) cex<K>(v, e, i, l);
                    else cex<K>(v, e, l, i);
                }
            }
        }
    }
}

// v <- the best K of v and w (both sorted descending), sorted descending:
// the elementwise better of v[q] and w[K-1-q] holds the best K as a bitonic
// sequence, which one merge network sorts
template <int K>
__device__ __forceinline__ void merge_topk(float (&v)[K], int32_t (&e)[K], const float (&w)[K],
                                           const int32_t (&f)[K]) {
#pragma unroll
    for (int q = 0; q < K; ++q)
        if (ranks_above(w[K - 1 - q], f[K - 1 - q], v[q], e[q])) {
            v[q] = w[K - 1 - q];
            e[q] = f[K - 1 - q];
        }
#pragma unroll
    for (int j = K >> 1; j > 0; j >>= 1) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int l = i ^ j;
            if (l > i) cex<K>(v, e, i, l);
        }
    }
}

// S: CTAs per cluster (1, 2, 4 or 8); CTA r runs K blocks k_blocks*r/S ..
// k_blocks*(r+1)/S.  KMAX: the length of the top-k lists (>= top_k).
template <int S, int KMAX>
__global__ void __launch_bounds__(R_THREADS, 1)
router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
              const RouterParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + R_OFF_BARS;
    const uint32_t bar_empty = bar_full + 8 * R_STAGES;
    const uint32_t bar_tfull = bar_empty + 8 * R_STAGES;
    const uint32_t bar_drain = bar_tfull + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + R_OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + R_OFF_ABORT);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b_bytes = static_cast<uint32_t>(p.n_pad) * R_BK * 2;

    if (tid == 0) {
        for (int s = 0; s < R_STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_x);
        tma_prefetch_map(&map_w);
    }
    if (warp == 1) {
        tmem_alloc(sbase + R_OFF_TMEM, static_cast<uint32_t>(p.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t rank = S > 1 ? cluster_cta_rank() : 0u;
    const int32_t row0 = static_cast<int32_t>(blockIdx.x / S) * R_BM;
    const int32_t kb_begin = static_cast<int32_t>((static_cast<int64_t>(p.k_blocks) * rank) / S);
    const int32_t kb_end = static_cast<int32_t>((static_cast<int64_t>(p.k_blocks) * (rank + 1)) / S);
    // The owner's slots, in the stage area (free once the cluster's MMAs have
    // all completed): slot of source CTA s, expert e, owned token j at
    // (s * n_pad + e) * RS + j.
    constexpr int ROWS = R_BM / S;                       // tokens a CTA owns
    const int RS = p.rs;
    const int T = p.lanes;                               // lanes per owned token
    float* slots = reinterpret_cast<float*>(smem);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_normal();
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int32_t kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_full + 8 * stage;
                const uint32_t sa = sbase + stage * R_STAGE_BYTES;
                mbar_arrive_expect_tx(fb, R_A_BYTES + b_bytes);
                tma_load_2d(sa, &map_x, fb, kb * R_BK, row0, pol);
                tma_load_2d(sa + R_A_BYTES, &map_w, fb, kb * R_BK, 0, pol);
                ++issued;
                if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                volatile int never = 0;
                const int64_t n = issued < R_STAGES ? issued : R_STAGES;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t idx = issued - 1 - i;
                    mbar_wait_bounded(bar_full + 8 * static_cast<uint32_t>(idx % R_STAGES),
                                      static_cast<uint32_t>((idx / R_STAGES) & 1), &never, R_DRAIN_NS);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32acc(R_BM, static_cast<uint32_t>(p.n_pad));
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int32_t kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sa = sbase + stage * R_STAGE_BYTES;
                const uint32_t sb = sa + R_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < R_BK / 16; ++kk)
                    tc_mma_f16(tmem_base, smem_desc_k_sw128(sa + kk * 32), smem_desc_k_sw128(sb + kk * 32), idesc,
                               (kb != kb_begin || kk != 0) ? 1u : 0u);
                tc_commit(bar_empty + 8 * stage);
                if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
            }
            if (ok) tc_commit(bar_tfull);
            volatile int never = 0;
            tc_commit(bar_drain);
            mbar_wait_bounded(bar_drain, 0, &never, R_DRAIN_NS);
        }
        __syncwarp();
    } else {
        if (mbar_wait_bounded(bar_tfull, 0, abort_flag, R_WAIT_NS)) tc_fence_after_sync();
        __syncwarp();
    }
    // every CTA of the cluster has finished its MMAs (its stage area is free)
    if (S > 1) cluster_sync_all();
    else __syncthreads();

    if (warp >= 2 && !*abort_flag) {
        // step 1: TMEM -> the owners' slots.  Warp w reads TMEM lanes
        // 32*(w%4) .. +31 (one token each); the four warps of a lane quarter
        // take every fourth group of 8 columns.
        const int quarter = warp & 3;
        const int cpart = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const int owner = row / ROWS;
        const uint32_t dst = (S > 1 ? mapa_shared(smem_u32(slots), static_cast<uint32_t>(owner)) : smem_u32(slots)) +
                             4u * static_cast<uint32_t>(static_cast<int>(rank) * p.n_pad * RS + (row - owner * ROWS));
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const bool token = static_cast<int64_t>(row0) + row < p.n_tokens;   // rows past the last token stay unread
        for (int32_t c0 = 8 * cpart; c0 < p.n_pad; c0 += 32) {
            uint32_t v[8];
            tmem_ld_32x32b_x8(taddr + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t a = dst + 4u * static_cast<uint32_t>((c0 + j) * RS);
                if (!token) continue;
                if (S > 1) st_shared_cluster_f32(a, __uint_as_float(v[j]));
                else slots[(c0 + j) * RS + row] = __uint_as_float(v[j]);
            }
        }
    }
    // every slot is written (and every CTA's abort flag is final)
    tc_fence_before_sync();
    __syncwarp();
    if (S > 1) cluster_sync_all();
    else __syncthreads();

    if (warp >= 2 && tid - 64 < ROWS * p.lanes) {        // whole warps: ROWS * T is a multiple of 32
        bool ok = true;
        const uint32_t abort_addr = smem_u32(const_cast<int*>(abort_flag));
#pragma unroll
        for (int r = 0; r < S; ++r)
            if ((S > 1 ? ld_shared_cluster_s32(mapa_shared(abort_addr, static_cast<uint32_t>(r))) : *abort_flag) != 0)
                ok = false;
        // step 2: T lanes per owned token; lane j takes experts j, j + T, ...
        const int et = tid - 64;
        const int g = et / T;                               // owned token
        const int j = et - g * T;
        const int64_t t = static_cast<int64_t>(row0) + static_cast<int>(rank) * ROWS + g;
        const bool live = ok && t < p.n_tokens;
        // the token's logit of expert e: the sum of its S partial slots in rank order
        auto logit = [&](int32_t e) {
            float l = 0.0f;
#pragma unroll
            for (int s = 0; s < S; ++s) l += slots[(s * p.n_pad + e) * RS + g];
            return l;
        };
        float bv[KMAX];
        int32_t bi[KMAX];
#pragma unroll
        for (int q = 0; q < KMAX; ++q) {
            bv[q] = -INFINITY;
            bi[q] = 0x7fffffff;
        }
        // pass 1: this lane's best KMAX, KMAX experts at a time
        for (int32_t e0 = j; live && e0 < p.n_experts; e0 += KMAX * T) {
            float cv[KMAX];
            int32_t ci[KMAX];
#pragma unroll
            for (int q = 0; q < KMAX; ++q) {
                const int32_t e = e0 + q * T;
                cv[q] = e < p.n_experts ? logit(e) : -INFINITY;
                ci[q] = e < p.n_experts ? e : 0x7fffffff;
            }
            bitonic_sort_desc<KMAX>(cv, ci);
            merge_topk<KMAX>(bv, bi, cv, ci);
        }
        // merge over the token's T lanes (both partners end with the same list)
#pragma unroll 1
        for (int d = 1; d < T; d <<= 1) {
            float ov[KMAX];
            int32_t oi[KMAX];
#pragma unroll
            for (int q = 0; q < KMAX; ++q) {
                ov[q] = __shfl_xor_sync(0xffffffffu, bv[q], d);
                oi[q] = __shfl_xor_sync(0xffffffffu, bi[q], d);
            }
            merge_topk<KMAX>(bv, bi, ov, oi);
        }
        // pass 2: sum of exp(l - max) over the token's experts
        const float m = bv[0];
        float sum = 0.0f;
        for (int32_t e = j; live && e < p.n_experts; e += T) sum += __expf(logit(e) - m);
#pragma unroll 1
        for (int d = 1; d < T; d <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
        sum = __shfl_sync(0xffffffffu, sum, lane & ~(T - 1));   // the token's first lane's value for all
        if (live && j == 0) {
#pragma unroll
            for (int q = 0; q < KMAX; ++q) {
                if (q < p.top_k) {
                    // an id in range: a finite logit ranked q-th (NaN logits never rank)
                    MOE_DCHECK(bi[q] >= 0 && bi[q] < p.n_experts, p.status);
                    p.topk_ids[t * p.top_k + q] = bi[q] < p.n_experts ? bi[q] : -1;
                    p.topk_weights[t * p.top_k + q] = __expf(bv[q] - m) / sum;
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn router_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
    });
    return fn;
}

bool router_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {R_BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return router_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_router(const uint16_t* x, int64_t n_tokens, int32_t hidden, const uint16_t* router_w,
                          int32_t n_experts, int32_t top_k, int32_t* topk_ids, float* topk_weights,
                          int32_t* status, cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    if (!router_encode_fn()) return cudaErrorNotSupported;
    RouterParams p{};
    p.n_tokens = n_tokens;
    p.n_experts = n_experts;
    p.n_pad = ((n_experts + 15) / 16) * 16;
    int cols = 32;
    while (cols < p.n_pad) cols <<= 1;
    p.tmem_cols = cols;
    p.top_k = top_k;
    p.k_blocks = hidden / R_BK;
    p.topk_ids = topk_ids;
    p.topk_weights = topk_weights;
    p.status = status;
    CUtensorMap map_x, map_w;
    if (!router_map(&map_x, x, static_cast<uint64_t>(n_tokens), static_cast<uint64_t>(hidden), R_BM) ||
        !router_map(&map_w, router_w, static_cast<uint64_t>(n_experts), static_cast<uint64_t>(hidden),
                    static_cast<uint32_t>(p.n_pad)))
        return cudaErrorInvalidValue;
    const int64_t tiles = (n_tokens + R_BM - 1) / R_BM;
    // K split: the largest power of two S <= R_MAX_SPLIT with tiles x S
    // within the SM count, at most one CTA per 64-wide K block, and the
    // owners' slots (S x n_pad x the slot stride, fp32) within the stage area
    int64_t split = 1;
    const int kmax = top_k <= 4 ? 4 : top_k <= 8 ? 8 : 16;
    // lanes per token: one list of kmax logits each, at most the 4*S the
    // epilogue warps give every owned token
    auto lanes_for = [&](int64_t sp) {
        int t = 1;
        while (t * 2 <= 4 * sp && t * 2 * kmax <= p.n_pad) t *= 2;
        return t < 4 ? 4 : t;
    };
    while (split * 2 <= R_MAX_SPLIT && tiles * split * 2 <= device_sm_count() && split * 2 <= p.k_blocks &&
           static_cast<int64_t>(split * 2) * p.n_pad *
                   slot_stride(static_cast<int>(split * 2), lanes_for(split * 2)) * 4 <= R_OFF_BARS)
        split *= 2;
    auto kernel_for = [kmax](int64_t sp) {
        if (kmax == 4)
            return sp >= 8 ? router_kernel<8, 4> : sp == 4 ? router_kernel<4, 4> : sp == 2 ? router_kernel<2, 4>
                                                                                          : router_kernel<1, 4>;
        if (kmax == 8)
            return sp >= 8 ? router_kernel<8, 8> : sp == 4 ? router_kernel<4, 8> : sp == 2 ? router_kernel<2, 8>
                                                                                          : router_kernel<1, 8>;
        return sp >= 8 ? router_kernel<8, 16> : sp == 4 ? router_kernel<4, 16> : sp == 2 ? router_kernel<2, 16>
                                                                                        : router_kernel<1, 16>;
    };
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(R_THREADS);
    cfg.dynamicSmemBytes = R_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a cluster size the device can place (clusters live inside one GPC);
    // the answer is cached per device and size
    static std::mutex mu;
    static std::map<std::tuple<int, int, int64_t>, bool> placeable;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNoDevice;
    for (; split >= 1; split /= 2) {
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_tuple(dev, kmax, split);
        auto it = placeable.find(key);
        if (it == placeable.end()) {
            cudaError_t e = cudaFuncSetAttribute(kernel_for(split), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(R_SMEM));
            if (e != cudaSuccess) return e;
            attr[0].val.clusterDim.x = static_cast<unsigned>(split);
            cfg.gridDim = dim3(static_cast<unsigned>(split));
            int n = 0;
            const bool ok = split == 1 || (cudaOccupancyMaxActiveClusters(&n, kernel_for(split), &cfg) == cudaSuccess &&
                                           n > 0);
            if (!ok) cudaGetLastError();
            it = placeable.emplace(key, ok).first;
        }
        if (it->second) break;
    }
    p.lanes = lanes_for(split);
    p.rs = slot_stride(static_cast<int>(split), p.lanes);
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * split));
    return cudaLaunchKernelEx(&cfg, kernel_for(split), map_x, map_w, p);
}

}  // namespace moe
