// Router: logits = x · W_gᵀ (fp32), softmax over all experts, top-k
// ("MetaX-TileLang工具链", §2.4: logits = W_g(x), scores = softmax(logits),
// topk_scores, topk_indices = topk(scores)).
//
// One CTA per 128-token tile, one tcgen05 MMA tile of M = 128 tokens and
// N = n_experts rounded up to 16 (at most 256), so a token's whole logit row
// sits in one TMEM lane.  Warp 0 streams x and W_g with TMA (4 stages of
// 64-wide K), warp 1 owns TMEM and issues the MMAs, warps 2-9 split each
// token's row in two halves of the expert columns: per half a register top-k
// (ties to the lower expert index, descending order) and the softmax sum
// against the half's maximum, then the first half's thread merges the two.
// The top-k is decided on the logits (softmax preserves their order).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

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
constexpr int R_THREADS = 320;                       // producer, MMA, 8 epilogue warps
constexpr int R_EPI_THREADS = 256;
constexpr int R_MAX_TOPK = 16;
constexpr uint64_t R_WAIT_NS = 2000000000ull;
constexpr uint64_t R_DRAIN_NS = 200000000ull;
constexpr int R_OFF_BARS = R_STAGES * R_STAGE_BYTES;
constexpr int R_OFF_TMEM = R_OFF_BARS + (2 * R_STAGES + 2) * 8;
constexpr int R_OFF_ABORT = R_OFF_TMEM + 4;
// the second half-row's partial results, handed to the first half's thread:
// top-k values [R_MAX_TOPK][128], ids [R_MAX_TOPK][128], max [128], sum [128]
constexpr int R_OFF_XCH = ((R_OFF_ABORT + 4 + 15) / 16) * 16;
constexpr int R_XCH_BYTES = (2 * R_MAX_TOPK + 2) * R_BM * 4;
constexpr size_t R_SMEM = 1024 + R_OFF_XCH + R_XCH_BYTES;

struct RouterParams {
    int64_t n_tokens;
    int32_t n_experts;
    int32_t n_pad;         // n_experts rounded up to 16
    int32_t tmem_cols;     // power of two >= max(32, n_pad)
    int32_t top_k;
    int32_t k_blocks;      // hidden / 64
    int32_t* topk_ids;
    float* topk_weights;
    int32_t* status;
};

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
    const int32_t row0 = static_cast<int32_t>(blockIdx.x) * R_BM;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_normal();
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
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
            for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
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
                               (kb | kk) != 0 ? 1u : 0u);
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
        // Warps 2-9: warp w reads TMEM lanes 32*(w%4) .. +31 (one token per
        // thread); warps 2-5 take the first half of the expert columns and
        // warps 6-9 the second half, then the second half's thread hands its
        // partial top-k, max and sum to the first half's thread of the same
        // token, which merges them and writes the token's outputs.
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const int64_t t = static_cast<int64_t>(row0) + row;
        const int32_t n_half = p.n_pad / 2;              // a multiple of 8
        const int32_t c_begin = half * n_half;
        float* xv = reinterpret_cast<float*>(smem + R_OFF_XCH);
        int32_t* xi = reinterpret_cast<int32_t*>(xv + R_MAX_TOPK * R_BM);
        float* xm = reinterpret_cast<float*>(xi + R_MAX_TOPK * R_BM);
        float* xs = xm + R_BM;
        float best_v[R_MAX_TOPK];
        int32_t best_i[R_MAX_TOPK];
#pragma unroll
        for (int q = 0; q < R_MAX_TOPK; ++q) {
            best_v[q] = -INFINITY;
            best_i[q] = -1;
        }
        float s = 0.0f;
        // Insert (l, e) into the descending list (everything in registers: all
        // loops over the list are unrolled with compile-time indices).  A new
        // value goes in after any equal one, so the lower expert index stays
        // first, and every slot is updated from the old list at once.
        auto insert = [&](float l, int32_t e) {
            bool gt[R_MAX_TOPK];
#pragma unroll
            for (int q = 0; q < R_MAX_TOPK; ++q) gt[q] = best_i[q] < 0 || l > best_v[q];
#pragma unroll
            for (int q = R_MAX_TOPK - 1; q > 0; --q) {
                best_v[q] = gt[q - 1] ? best_v[q - 1] : (gt[q] ? l : best_v[q]);
                best_i[q] = gt[q - 1] ? best_i[q - 1] : (gt[q] ? e : best_i[q]);
            }
            if (gt[0]) {
                best_v[0] = l;
                best_i[0] = e;
            }
        };
        const bool ok = mbar_wait_bounded(bar_tfull, 0, abort_flag, R_WAIT_NS);
        if (ok) {
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            // pass 1: the R_MAX_TOPK largest logits of this half (8 columns per
            // TMEM load keeps the unrolled code within the instruction cache)
            for (int32_t c0 = c_begin; c0 < c_begin + n_half; c0 += 8) {
                uint32_t v[8];
                tmem_ld_32x32b_x8(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int32_t e = c0 + j;
                    const float l = __uint_as_float(v[j]);
                    if (e < p.n_experts && (best_i[R_MAX_TOPK - 1] < 0 || l > best_v[R_MAX_TOPK - 1])) insert(l, e);
                }
            }
            // pass 2: sum of exp(l - this half's max), independent partial sums
            const float mh = best_v[0];
            float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int32_t c0 = c_begin; c0 < c_begin + n_half; c0 += 8) {
                uint32_t v[8];
                tmem_ld_32x32b_x8(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + j < p.n_experts) part[j & 3] += expf(__uint_as_float(v[j]) - mh);
            }
            s = (part[0] + part[1]) + (part[2] + part[3]);
            if (half == 1) {
#pragma unroll
                for (int q = 0; q < R_MAX_TOPK; ++q) {
                    xv[q * R_BM + row] = best_v[q];
                    xi[q * R_BM + row] = best_i[q];
                }
                xm[row] = mh;
                xs[row] = s;
            }
        }
        // every epilogue thread meets here, whatever its wait returned
        asm volatile("bar.sync 1, %0;" ::"r"(R_EPI_THREADS) : "memory");
        if (half == 0 && ok && !*abort_flag) {
            // merge: the other half's experts all have higher indices, so its
            // entries go after equal values already in the list
            const float m0 = best_v[0], m1 = xm[row];
            for (int q = 0; q < R_MAX_TOPK; ++q) {
                const int32_t e = xi[q * R_BM + row];
                const float l = xv[q * R_BM + row];
                if (e < 0) break;
                if (best_i[R_MAX_TOPK - 1] >= 0 && !(l > best_v[R_MAX_TOPK - 1])) break;
                insert(l, e);
            }
            const float mx = best_v[0];                   // = max(m0, m1)
            const float st = s * expf(m0 - mx) + (m1 == -INFINITY ? 0.0f : xs[row] * expf(m1 - mx));
            if (t < p.n_tokens) {
#pragma unroll
                for (int q = 0; q < R_MAX_TOPK; ++q) {
                    if (q < p.top_k) {
                        // ids in range and the list in descending order
                        MOE_DCHECK(best_i[q] >= 0 && best_i[q] < p.n_experts, p.status);
                        MOE_DCHECK(q == 0 || !(best_v[q] > best_v[q > 0 ? q - 1 : 0]), p.status);
                        p.topk_ids[t * p.top_k + q] = best_i[q];
                        p.topk_weights[t * p.top_k + q] = expf(best_v[q] - mx) / st;
                    }
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
    cudaError_t err = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(R_SMEM));
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>((n_tokens + R_BM - 1) / R_BM);
    router_kernel<<<grid, R_THREADS, R_SMEM, stream>>>(map_x, map_w, p);
    return cudaGetLastError();
}

}  // namespace moe
