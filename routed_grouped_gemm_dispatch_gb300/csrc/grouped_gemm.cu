// Grouped expert GEMMs of the routed fused MoE forward, for sm_103a.
//
// Phase 1 ("Fused MoE GEMM 提交说明", §完整算子代码, first launch): for every
// 128-row block bx with actual_rows > 0 and every 128-wide slice n of the
// intermediate dimension,
//     G = X[bx] · gate_w[e][n]ᵀ,  U = X[bx] · up_w[e][n]ᵀ      (fp32)
//     up_logits[row, n·128 + j] = fp16( silu(G[i,j]) · U[i,j] )  for i < actual_rows
// Phase 2 (second launch): for every active block and 256-wide slice of hidden,
//     C = U_logits[bx] · down_w[e][slice]ᵀ                      (fp32)
//     out[row, col] = fp16( C[i,col] · routed_expert_weights[offsets[e] + token_offset + i] )
// with e = group_idx_for_bx[bx], token_offset = bx·128 − group_padded_offsets[e],
// actual_rows = max(0, min(128, group_sizes[e] − token_offset)).
//
// GB300 design (not the page's): one persistent CTA per SM walks a compacted
// list of active (block, slice) tiles, so padding-only blocks cost nothing.
// Warp roles: warp 0 issues TMA loads (128-byte swizzled tiles, 4-stage
// ring), warp 1 owns TMEM and issues tcgen05.mma (M=128, N=256, K=16, fp32
// accumulators in TMEM, double buffered so the epilogue of tile t overlaps the
// MMAs of tile t+1), warps 2-5 run the epilogue from TMEM through registers.
// Phase 1 stacks the gate and up slices as one N=256 B operand so the x tile
// is loaded once for both products.  Every pipeline wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                       // rows per block (block_token)
constexpr int BK = 64;                        // K per stage: one 128-byte swizzle row
constexpr int BN = 256;                       // N per MMA
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_TILE_BYTES = BN * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators of 128 x 256
constexpr int NUM_THREADS = 192;              // 6 warps
constexpr int NUM_EPI_THREADS = 128;          // warps 2..5
constexpr int PANEL = 16;                     // active blocks per rasterisation panel
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;   // 0.2 s per drain wait
constexpr uint32_t IDESC = idesc_f16_f32acc(BM, BN);

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int OFF_STAGES = 0;
constexpr int OFF_BARS = STAGES * STAGE_BYTES;                 // 8-byte mbarriers
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;               // full, empty, tfull, tempty, drain
constexpr int OFF_TMEM_SLOT = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int OFF_NACT = OFF_ABORT + 4;
constexpr int OFF_WSUM = OFF_NACT + 4;                         // NUM_THREADS/32 ints
constexpr int OFF_LIST = ((OFF_WSUM + (NUM_THREADS / 32) * 4 + 15) / 16) * 16;  // uint16 bx list

size_t smem_bytes_for(int64_t num_blocks_m) {
    return 1024 /* alignment slack */ + OFF_LIST + 2 * static_cast<size_t>(num_blocks_m);
}

struct GemmParams {
    const int32_t* sizes;
    const int32_t* offsets;
    const int32_t* padded;
    const int32_t* gidx;
    const float* rw;          // phase 2 only
    uint16_t* dst;            // up_logits (phase 1) or out (phase 2)
    int32_t* status;
    int64_t rows_total;
    int64_t valid_total;
    int32_t num_blocks_m;
    int32_t n_experts;
    int32_t k_blocks;         // K / 64
    int32_t n_tiles;          // N slices per block
    int32_t n_extent;         // I (phase 1) or H (phase 2): columns of dst
};

struct TileInfo {
    int32_t bx;
    int32_t n;
};

__device__ __forceinline__ TileInfo decode_tile(int32_t t, int32_t nact, int32_t n_tiles,
                                                const uint16_t* list) {
    const int32_t per_panel = PANEL * n_tiles;
    const int32_t pi = t / per_panel;
    const int32_t r = t - pi * per_panel;
    const int32_t first = pi * PANEL;
    const int32_t width = min(PANEL, nact - first);
    const int32_t n = r / width;
    const int32_t b = r - n * width;
    return TileInfo{static_cast<int32_t>(list[first + b]), n};
}

// Rows of block bx that belong to its expert ("Fused MoE GEMM 提交说明",
// §完整算子代码: actual_rows).  Also returns the expert and the row's
// token_offset.  Blocks whose table entries point outside their arrays count
// as empty and raise MOE_DEV_BAD_TABLE.
__device__ __forceinline__ int32_t block_rows(const GemmParams& p, int32_t bx, int32_t* e_out,
                                              int32_t* tok_off_out) {
    const int32_t e = __ldg(p.gidx + bx);
    if (e < 0 || e >= p.n_experts) {
        if (p.status) atomicOr(p.status, MOE_DEV_BAD_TABLE);
        return 0;
    }
    const int64_t tok_off = static_cast<int64_t>(bx) * BM - __ldg(p.padded + e);
    int64_t actual = static_cast<int64_t>(__ldg(p.sizes + e)) - tok_off;
    actual = actual > BM ? BM : (actual < 0 ? 0 : actual);
    if (actual > 0) {
        const int64_t c0 = static_cast<int64_t>(__ldg(p.offsets + e)) + tok_off;
        if (tok_off < 0 || c0 < 0 || c0 + actual > p.valid_total ||
            static_cast<int64_t>(bx) * BM + actual > p.rows_total) {
            if (p.status) atomicOr(p.status, MOE_DEV_BAD_TABLE);
            return 0;
        }
    }
    *e_out = e;
    *tok_off_out = static_cast<int32_t>(tok_off);
    return static_cast<int32_t>(actual);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int PHASE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1,
                    const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + OFF_BARS;                   // [STAGES]
    const uint32_t bar_empty = bar_full + 8 * STAGES;             // [STAGES]
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;            // [2]
    const uint32_t bar_tempty = bar_tfull + 16;                   // [2]
    const uint32_t bar_drain = bar_tempty + 16;                   // [1]
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* wsum = reinterpret_cast<int32_t*>(smem + OFF_WSUM);
    uint16_t* list = reinterpret_cast<uint16_t*>(smem + OFF_LIST);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (PHASE == 1) pdl_launch_dependents();

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, 1);
            mbar_init(bar_tempty + 8 * a, NUM_EPI_THREADS);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b0);
        if (PHASE == 1) tma_prefetch_map(&map_b1);
    }
    if (warp == 1) {
        tmem_alloc(sbase + OFF_TMEM_SLOT, TMEM_COLS);
        tmem_relinquish();
    }

    // ---- compacted list of active blocks (same order as bx) ----------------
    int32_t nact = 0;
    for (int32_t base = 0; base < p.num_blocks_m; base += NUM_THREADS) {
        const int32_t bx = base + tid;
        int32_t flag = 0;
        if (bx < p.num_blocks_m) {
            int32_t e, tok;
            flag = block_rows(p, bx, &e, &tok) > 0;
        }
        const uint32_t ballot = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) wsum[warp] = __popc(ballot);
        __syncthreads();
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < NUM_THREADS / 32; ++w) {
            const int32_t c = wsum[w];
            before += (w < warp) ? c : 0;
            total += c;
        }
        if (flag) list[nact + before + __popc(ballot & ((1u << lane) - 1u))] = static_cast<uint16_t>(bx);
        nact += total;
        __syncthreads();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const int32_t total_tiles = nact * p.n_tiles;

    // Phase 2 reads up_logits written by phase 1: wait for that grid here
    // (everything above only touched the dispatch tables).
    if (PHASE == 2) pdl_wait_prior_grid();

    if (warp == 0) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_normal();
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, nact, p.n_tiles, list);
                const int32_t e = __ldg(p.gidx + ti.bx);
                for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t sa = sbase + OFF_STAGES + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE_BYTES;
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(sa, &map_a, fb, kb * BK, ti.bx * BM, pol);
                    if (PHASE == 1) {
                        tma_load_3d(sb, &map_b0, fb, kb * BK, ti.n * 128, e, pol);
                        tma_load_3d(sb + B_TILE_BYTES / 2, &map_b1, fb, kb * BK, ti.n * 128, e, pol);
                    } else {
                        tma_load_3d(sb, &map_b0, fb, kb * BK, ti.n * BN, e, pol);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // Let the copies already in flight land before the CTA exits.
                volatile int never = 0;
                const int64_t n = issued < STAGES ? issued : STAGES;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t idx = issued - 1 - i;
                    mbar_wait_bounded(bar_full + 8 * static_cast<uint32_t>(idx % STAGES),
                                      static_cast<uint32_t>((idx / STAGES) & 1), &never, DRAIN_LIMIT_NS);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, aphase = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                if (!mbar_wait_bounded(bar_tempty + 8 * acc, aphase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int32_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = sbase + OFF_STAGES + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_f16(d_tmem, smem_desc_k_sw128(sa + kk * 32), smem_desc_k_sw128(sb + kk * 32),
                                   IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(bar_empty + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(bar_tfull + 8 * acc);
                acc ^= 1u;
                if (acc == 0) aphase ^= 1u;
            }
            // Every MMA this thread issued has finished once this arrives.
            volatile int never = 0;
            tc_commit(bar_drain);
            mbar_wait_bounded(bar_drain, 0, &never, DRAIN_LIMIT_NS);
        }
        __syncwarp();
    } else {
        // ===================== epilogue (warps 2..5) =====================
        const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;         // row of the 128-row tile
        uint32_t acc = 0, aphase = 0;
        for (int32_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const TileInfo ti = decode_tile(t, nact, p.n_tiles, list);
            int32_t e = 0, tok = 0;
            const int32_t actual = block_rows(p, ti.bx, &e, &tok);
            if (!mbar_wait_bounded(bar_tfull + 8 * acc, aphase, abort_flag, WAIT_LIMIT_NS)) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            const int64_t grow = static_cast<int64_t>(ti.bx) * BM + row;
            if (PHASE == 1) {
                uint16_t* dst_row = p.dst + grow * p.n_extent + static_cast<int64_t>(ti.n) * 128;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, g);
                    tmem_ld_32x32b_x32(taddr + 128 + c * 32, u);
                    tmem_ld_wait();
                    if (row < actual) {
                        uint32_t h[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g0 = __uint_as_float(g[2 * j]);
                            const float g1 = __uint_as_float(g[2 * j + 1]);
                            const float s0 = __fdividef(g0, 1.0f + __expf(-g0));
                            const float s1 = __fdividef(g1, 1.0f + __expf(-g1));
                            h[j] = pack_half2(s0 * __uint_as_float(u[2 * j]),
                                              s1 * __uint_as_float(u[2 * j + 1]));
                        }
                        uint4* d4 = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                    }
                }
            } else {
                float w = 0.0f;
                if (row < actual) w = __ldg(p.rw + (__ldg(p.offsets + e) + tok + row));
                uint16_t* dst_row = p.dst + grow * p.n_extent;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int32_t col0 = ti.n * BN + c * 32;
                    if (col0 >= p.n_extent) break;              // partial last slice of H
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, v);
                    tmem_ld_wait();
                    if (row < actual) {
                        uint32_t h[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            h[j] = pack_half2(__uint_as_float(v[2 * j]) * w, __uint_as_float(v[2 * j + 1]) * w);
                        uint4* d4 = reinterpret_cast<uint4*>(dst_row + col0);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(bar_tempty + 8 * acc);
            acc ^= 1u;
            if (acc == 0) aphase ^= 1u;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D fp16 map over a row-major [rows, cols] array, box {64, box_rows}, 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp16 map over [experts, rows, cols], box {64, box_rows, 1}: the expert is
// a coordinate, so a tile never crosses into the next expert (rows past the end
// of one expert read as zero).
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t experts, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
    const cuuint64_t dims[3] = {cols, rows, experts};
    const cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    const cuuint32_t box[3] = {BK, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attr(const void* fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

}  // namespace

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

cudaError_t launch_fused_forward(const ForwardArgs& a, uint32_t flags, cudaStream_t stream) {
    if (!encode_fn()) return cudaErrorNotSupported;
    CUtensorMap map_x, map_gate, map_up, map_u, map_down;
    const uint64_t rows = static_cast<uint64_t>(a.rows_total);
    const uint64_t H = static_cast<uint64_t>(a.hidden), I = static_cast<uint64_t>(a.intermediate);
    const uint64_t E = static_cast<uint64_t>(a.n_experts);
    if (!make_map_2d(&map_x, a.x, rows, H, BM) || !make_map_3d(&map_gate, a.gate_w, E, I, H, 128) ||
        !make_map_3d(&map_up, a.up_w, E, I, H, 128) || !make_map_2d(&map_u, a.up_logits, rows, I, BM) ||
        !make_map_3d(&map_down, a.down_w, E, H, I, BN))
        return cudaErrorInvalidValue;

    GemmParams p1{};
    p1.sizes = a.sizes;
    p1.offsets = a.offsets;
    p1.padded = a.padded;
    p1.gidx = a.gidx;
    p1.rw = a.rw;
    p1.status = a.status;
    p1.rows_total = a.rows_total;
    p1.valid_total = a.valid_total;
    p1.num_blocks_m = static_cast<int32_t>(a.num_blocks_m);
    p1.n_experts = a.n_experts;
    GemmParams p2 = p1;
    p1.dst = a.up_logits;
    p1.k_blocks = a.hidden / BK;
    p1.n_tiles = a.intermediate / 128;
    p1.n_extent = a.intermediate;
    p2.dst = a.out;
    p2.k_blocks = a.intermediate / BK;
    p2.n_tiles = (a.hidden + BN - 1) / BN;
    p2.n_extent = a.hidden;

    const size_t smem = smem_bytes_for(a.num_blocks_m);
    cudaError_t err;
    if ((err = set_smem_attr(reinterpret_cast<const void*>(&grouped_gemm_kernel<1>), smem)) != cudaSuccess) return err;
    if ((err = set_smem_attr(reinterpret_cast<const void*>(&grouped_gemm_kernel<2>), smem)) != cudaSuccess) return err;

    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorNoDevice;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    if (flags & MOE_RUN_PHASE1) {
        err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<1>, map_x, map_gate, map_up, p1);
        if (err != cudaSuccess) return err;
    }
    if (flags & MOE_RUN_PHASE2) {
        // Phase 2 may start its prologue (tables, TMEM, barriers) while phase 1
        // drains; it waits for phase 1's results before its first load.
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = (flags & MOE_NO_PDL) ? 0 : 1;
        err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<2>, map_u, map_down, map_down, p2);
    }
    return err;
}

}  // namespace moe
