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
// GB300 design (not the page's):
//  * Persistent clusters of two CTAs (one CTA per SM) walk a compacted list of
//    work units built from the active blocks (actual_rows > 0), so padding-only
//    blocks cost nothing.  A unit is a PAIR — two consecutive active blocks of
//    the same expert — or a SINGLE block.
//  * Each (unit, N slice) tile is one 2-SM MMA tile: tcgen05.mma.cta_group::2
//    with M = 256 (rows 0..127 = the first block, held by the even CTA; rows
//    128..255 = the second block, held by the odd CTA) and N = 256, where each
//    CTA's shared memory holds only half of the weight tile (128 of its 256
//    rows) and the pair shares it.  Per SM this halves the weight bytes that
//    TMA writes into and the tensor core reads out of shared memory, which is
//    what limits a one-SM 128 x 256 tile.  A SINGLE block runs as a 2-SM tile
//    with M = 128: each CTA holds 64 of the block's rows, so no MMA work goes
//    to a second, empty block.  The M = 128 accumulator of a CTA sits in 128
//    TMEM columns: lanes 0-63 hold its rows' columns 0-127 of N, lanes 64-127
//    the same rows' columns 128-255.  In phase 1 each CTA's half of B is then
//    64 gate rows followed by the same 64 up rows, so a thread finds the gate
//    and up values of its outputs in its own lane.
//  * Tiles are ordered in groups of units, slice by slice inside a group, so
//    concurrent clusters share each weight slice in L2 instead of re-reading
//    it once per unit.  One-phase launches split each expert's units evenly
//    into as few groups as the L2 budget allows (decode_tile_groups); the
//    single launch, and one-phase launches whose group table does not fit in
//    shared memory, use groups of the average units per expert (decode_tile).
//  * Inside a CTA: warp 0 issues TMA loads (128-byte swizzled tiles; a ring of
//    three 64 KB stages, each two adjacent 64-wide K boxes of A and of B; both
//    CTAs' copies complete on the even CTA's "full" barrier), warp 1
//    owns TMEM (allocated for the pair) and, in the even CTA only, issues the
//    MMAs (K = 16 each, fp32 accumulators in TMEM, double buffered so the
//    epilogue of one tile overlaps the MMAs of the next), warps 2-5 run the
//    epilogue of the CTA's own 128 rows from TMEM through registers.  Phase 1
//    stacks the gate slice (even CTA) and the up slice (odd CTA) as the N=256 B
//    operand, so the x tile is read once for both products.  Every pipeline
//    wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/moe_gb300.h"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                       // rows per block (block_token)
constexpr int BK = 64;                        // K per box: one 128-byte swizzle row
constexpr int KSUB = 2;                       // boxes (adjacent 64-wide K chunks) per stage
constexpr int BN = 256;                       // N per MMA
constexpr int STAGES = 6 / KSUB;
constexpr int A_BOX_BYTES = BM * BK * 2;      // 16 KB: this CTA's 128 rows of A, one box
constexpr int B_BOX_BYTES = (BN / 2) * BK * 2;  // 16 KB: this CTA's 128 rows of B, one box
constexpr int A_TILE_BYTES = KSUB * A_BOX_BYTES;
constexpr int B_HALF_BYTES = KSUB * B_BOX_BYTES;
constexpr int STAGE_BYTES = A_TILE_BYTES + B_HALF_BYTES;
constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators of 128 lanes x 256
constexpr int NUM_THREADS = 192;              // 6 warps
constexpr int NUM_EPI_THREADS = 128;          // warps 2..5
constexpr int CLUSTER = 2;
constexpr uint16_t CLUSTER_MASK = 0x3;
constexpr uint16_t PAIR_BIT = 0x8000;
constexpr int SMALL_ROWS = 32;                // blocks with at most this many rows load 16-row boxes
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;   // 0.2 s per drain wait
constexpr uint32_t IDESC = idesc_f16_f32acc(2 * BM, BN);   // M = 256 across the pair
constexpr uint32_t IDESC_M128 = idesc_f16_f32acc(BM, BN);  // M = 128 across the pair (a lone block)
constexpr int HALF_ROWS = BM / 2;                          // rows of a lone block each CTA holds
constexpr uint32_t A16_BYTES = A_BOX_BYTES / 8;            // a 16-row box of A
constexpr uint32_t A64_BYTES = A_BOX_BYTES / 2;            // a 64-row box of A
constexpr int64_t GROUP_A_BYTES = 64ll << 20;     // A rows a tile-order group keeps hot in L2

static_assert(MOE_MAX_BLOCKS <= 0x7FFF, "block indices must leave the pair bit free");

// Shared-memory layout (offsets from a 1024-byte aligned base).  During the
// prologue the stage area also holds the active-block list and its experts.
constexpr int OFF_STAGES = 0;
constexpr int OFF_BARS = STAGES * STAGE_BYTES;                 // 8-byte mbarriers
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;               // full, empty, tfull, tempty, drain
constexpr int OFF_TMEM_SLOT = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
constexpr int OFF_COUNTS = OFF_ABORT + 4;                      // runs, units, groups, (spare)
constexpr int OFF_WSUM = OFF_COUNTS + 16;                      // NUM_THREADS/32 ints
constexpr int OFF_UNITS = ((OFF_WSUM + (NUM_THREADS / 32) * 4 + 15) / 16) * 16;

// After the unit list (one uint16 per unit, at most one unit per block)
// comes, when the tile order uses per-expert groups, the first unit of every
// group (one uint16 per group, at most one group per unit).
__host__ __device__ inline size_t units_bytes(int64_t m) { return ((2 * static_cast<size_t>(m) + 15) / 16) * 16; }
size_t smem_bytes_for(int64_t m, bool expert_groups) {
    return 1024 /* alignment slack */ + OFF_UNITS + units_bytes(m) * (expert_groups ? 2 : 1) + (MOE_DEBUG ? 16 : 0);
}
constexpr uint32_t SMEM_CANARY = 0xC0FFEE11u;

struct PhaseParams {
    uint16_t* dst;            // up_logits (phase 1) or out (phase 2)
    int32_t k_blocks;         // K / (64 * KSUB)
    int32_t n_tiles;          // N slices per block
    int32_t n_extent;         // I (phase 1) or H (phase 2): columns of dst
    int32_t group;            // most units of a tile-order group the L2 budget allows (>= 1)
};

struct GemmParams {
    const int32_t* sizes;
    const int32_t* offsets;
    const int32_t* padded;
    const int32_t* gidx;
    const float* rw;          // phase 2 only
    int32_t* status;
    int64_t rows_total;
    int64_t valid_total;
    int32_t num_blocks_m;
    int32_t n_experts;
    PhaseParams ph[2];        // [0]: phase 1 (gate+up), [1]: phase 2 (down)
    int32_t tables_before_wait;  // phase 2 right behind phase 1: the tables may be read before
                                 // waiting for phase 1 (phase 1 lets it start only after its own wait)
    int32_t* ready;           // both phases in one launch: per unit, finished phase-1 tile stores
                              // (zero at launch)
    int32_t drop_first_signal;   // failure-path test: skip the first "accumulator ready" commit
    int32_t expert_groups;    // one-phase launches: tile-order groups follow the experts (see decode_tile_groups)
};

// Rows of block bx that belong to its expert ("Fused MoE GEMM 提交说明",
// §完整算子代码: actual_rows).  Also returns the expert and the block's
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

// One cluster tile as seen by the CTA of rank `rank`.  Tile order: the unit
// list (expert-sorted) is cut into groups of consecutive units, and inside a
// group the tiles run slice by slice, each slice over all the group's units.
// Concurrent clusters then share each weight slice across an expert's units
// while the group's A rows stay in L2.  decode_tile: groups of `group` units
// (about the average number of units per expert; group = 1 is plain
// unit-major order).  decode_tile_groups: groups that follow the experts,
// each expert's units split evenly into as few groups as the L2 budget
// allows, so an expert with many units streams its weights a few times
// instead of once per average-sized group.
struct Tile {
    int32_t u;        // unit
    int32_t bx0;      // first block of the unit (the expert comes from it)
    int32_t bx;       // block whose rows this CTA holds (a lone block: both CTAs hold half of it)
    int32_t n;        // N slice
    bool pair;        // true: M = 256 over two blocks; false: M = 128 over one block
};

__device__ __forceinline__ Tile decode_tile(int32_t t, const uint16_t* units, int32_t n_tiles,
                                            int32_t nunits, int32_t group, uint32_t rank) {
    const int32_t per_group = group * n_tiles;
    const int32_t g = t / per_group;
    const int32_t l = t - g * per_group;
    const int32_t left = nunits - g * group;
    const int32_t gsize = left < group ? left : group;
    Tile ti;
    ti.n = l / gsize;
    const int32_t u = g * group + (l - ti.n * gsize);
    ti.u = u;
    ti.bx0 = units[u] & 0x7FFF;
    ti.pair = (units[u] & PAIR_BIT) != 0;
    ti.bx = ti.pair ? ti.bx0 + static_cast<int32_t>(rank) : ti.bx0;
    return ti;
}

// Group g starts at unit gstart[g] and its tiles at gstart[g] * n_tiles.
__device__ __forceinline__ Tile decode_tile_groups(int32_t t, const uint16_t* units, const uint16_t* gstart,
                                                   int32_t ngroups, int32_t n_tiles, int32_t nunits, uint32_t rank) {
    int32_t lo = 0, hi = ngroups - 1;            // the last group that starts at or before tile t
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (static_cast<int32_t>(gstart[mid]) * n_tiles <= t) lo = mid;
        else hi = mid - 1;
    }
    const int32_t g0 = gstart[lo];
    const int32_t gsize = (lo + 1 < ngroups ? static_cast<int32_t>(gstart[lo + 1]) : nunits) - g0;
    const int32_t l = t - g0 * n_tiles;
    Tile ti;
    ti.n = l / gsize;
    const int32_t u = g0 + (l - ti.n * gsize);
    ti.u = u;
    ti.bx0 = units[u] & 0x7FFF;
    ti.pair = (units[u] & PAIR_BIT) != 0;
    ti.bx = ti.pair ? ti.bx0 + static_cast<int32_t>(rank) : ti.bx0;
    return ti;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Epilogue stores in whole 128-byte lines.  Each thread holds 64 fp16 columns
// of its own row as eight 16-byte pieces.  Inside every group of 8 lanes the
// 8 x 8 grid of pieces is transposed with three rounds of butterfly shuffles
// (round m swaps the pieces whose index bit m differs from the lane's bit m),
// after which lane 8g + i holds piece i of rows 8g .. 8g + 7; one store per
// row then writes a full 128-byte line from 8 lanes, 4 lines per warp
// instruction, instead of 32 half-filled sectors.
__device__ __forceinline__ void transpose8_pieces(uint4 (&el)[8], int lane) {
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (e & m) continue;
            const int f = e | m;
            const uint4 send = hi ? el[e] : el[f];
            uint4 recv;
            recv.x = __shfl_xor_sync(0xffffffffu, send.x, m);
            recv.y = __shfl_xor_sync(0xffffffffu, send.y, m);
            recv.z = __shfl_xor_sync(0xffffffffu, send.z, m);
            recv.w = __shfl_xor_sync(0xffffffffu, send.w, m);
            if (hi) el[e] = recv;
            else el[f] = recv;
        }
    }
}

// Store the 64 columns the warp's threads hold for their rows (el[k] = columns
// 8k .. 8k+7 of row warp_row0 + lane), rows below `actual` only.  `dst0`
// points at the first column in row warp_row0; `stride` is the row stride.
// A warp with at least 16 valid rows transposes first and writes whole lines;
// a sparser warp (decode-like blocks) stores each thread's row directly.
__device__ __forceinline__ void store_rows64(uint4 (&el)[8], uint16_t* dst0, int64_t stride, int lane,
                                            int warp_row0, int32_t actual) {
    if (warp_row0 + 16 <= actual) {
        transpose8_pieces(el, lane);
        const int g8 = lane & ~7;
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (warp_row0 + g8 + r < actual)
                *reinterpret_cast<uint4*>(dst0 + static_cast<int64_t>(g8 + r) * stride + (lane & 7) * 8) = el[r];
    } else if (warp_row0 + lane < actual) {
        uint4* d = reinterpret_cast<uint4*>(dst0 + static_cast<int64_t>(lane) * stride);
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = el[k];
    }
}

// Which phase a tile of the launch belongs to, and its index inside that
// phase.  PHASE 1 or 2 launches run one phase; PHASE 3 runs both: the first
// nunits * n_tiles(phase 1) tiles are phase 1, the rest phase 2.
struct PhaseTile {
    int ph;
    int32_t t;
};

template <int PHASE>
__device__ __forceinline__ PhaseTile phase_of(int32_t t, int32_t tiles1) {
    if (PHASE == 1) return PhaseTile{1, t};
    if (PHASE == 2) return PhaseTile{2, t};
    return t < tiles1 ? PhaseTile{1, t} : PhaseTile{2, t - tiles1};
}

// Wait (bounded) until *counter >= need, with acquire ordering.
__device__ __forceinline__ bool counter_wait_bounded(const int32_t* counter, int32_t need, volatile int* abort,
                                                     uint64_t limit_ns) {
    auto load = [&]() {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
        return v;
    };
    if (load() >= need) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(64);
        if (load() >= need) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}

// map_x / map_x64 / map_x16: x (boxes of 128, 64 and 16 rows, 64 wide);
// map_gate / map_up: phase-1 weights (boxes of 128 rows), map_gate64 /
// map_up64 (64 rows, for M = 128 tiles); map_u / map_u64 / map_u16:
// up_logits; map_down: phase-2 weights (128 rows).  A launch of one phase gets
// placeholders for the other phase's maps.
template <int PHASE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_x64,
                    const __grid_constant__ CUtensorMap map_x16,
                    const __grid_constant__ CUtensorMap map_gate,
                    const __grid_constant__ CUtensorMap map_up,
                    const __grid_constant__ CUtensorMap map_gate64,
                    const __grid_constant__ CUtensorMap map_up64,
                    const __grid_constant__ CUtensorMap map_u,
                    const __grid_constant__ CUtensorMap map_u64,
                    const __grid_constant__ CUtensorMap map_u16,
                    const __grid_constant__ CUtensorMap map_down,
                    const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + OFF_BARS;                   // [STAGES] (used in the even CTA)
    const uint32_t bar_empty = bar_full + 8 * STAGES;             // [STAGES]
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;            // [2]
    const uint32_t bar_tempty = bar_tfull + 16;                   // [2] (used in the even CTA)
    const uint32_t bar_drain = bar_tempty + 16;                   // [1]
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* counts = reinterpret_cast<int32_t*>(smem + OFF_COUNTS);
    int32_t* wsum = reinterpret_cast<int32_t*>(smem + OFF_WSUM);
    uint16_t* units = reinterpret_cast<uint16_t*>(smem + OFF_UNITS);
    // prologue scratch in the (still unused) stage area
    uint16_t* act_bx = reinterpret_cast<uint16_t*>(smem + OFF_STAGES);
    uint16_t* act_e = act_bx + p.num_blocks_m;
    uint16_t* unit_rs = act_e + p.num_blocks_m;            // each unit's run (its first list entry)
    uint16_t* unit_pos = unit_rs + p.num_blocks_m;         // and its position among the run's units
    uint16_t* run_nb = unit_pos + p.num_blocks_m;          // at a run's first entry: the run's blocks
    uint16_t* gstart = units + units_bytes(p.num_blocks_m) / 2;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_cta_rank();
    const bool leader = rank == 0;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);           // the even CTA's arrive.expect_tx
            mbar_init(bar_empty + 8 * s, 1);          // the MMA's commit, multicast to both CTAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8 * a, 1);
            mbar_init(bar_tempty + 8 * a, CLUSTER * NUM_EPI_THREADS);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if (PHASE != 2) {
            tma_prefetch_map(&map_x);
            tma_prefetch_map(&map_x64);
            tma_prefetch_map(&map_x16);
            tma_prefetch_map(&map_gate);
            tma_prefetch_map(&map_up);
            tma_prefetch_map(&map_gate64);
            tma_prefetch_map(&map_up64);
        }
        if (PHASE != 1) {
            tma_prefetch_map(&map_u);
            tma_prefetch_map(&map_u64);
            tma_prefetch_map(&map_u16);
            tma_prefetch_map(&map_down);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(sbase + OFF_TMEM_SLOT, TMEM_COLS);
        tmem_relinquish_pair();
    }

    // Launched with programmatic dependent launch: everything above overlaps
    // the previous kernel; every global read below comes after its completion.
    // Phase 2 directly behind phase 1 may read the dispatch tables earlier
    // (phase 1 only lets it start once phase 1 itself has waited).
    if (PHASE != 2 || !p.tables_before_wait) pdl_wait_prior_grid();
    // Let the next kernel on the stream launch: phase 2 behind phase 1, or
    // the next step's table builder behind phase 2 (it waits for this grid
    // before it writes anything).
    pdl_launch_dependents();

    // ---- 1. compacted list of active blocks and their experts (bx order) ---
    int32_t nact = 0;
    for (int32_t base = 0; base < p.num_blocks_m; base += NUM_THREADS) {
        const int32_t bx = base + tid;
        int32_t flag = 0, e = 0, tok = 0;
        if (bx < p.num_blocks_m) flag = block_rows(p, bx, &e, &tok) > 0;
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
        if (flag) {
            const int32_t i = nact + before + __popc(ballot & ((1u << lane) - 1u));
            act_bx[i] = static_cast<uint16_t>(bx);
            act_e[i] = static_cast<uint16_t>(e);
        }
        nact += total;
        __syncthreads();
    }

    // ---- 2. units: pair up consecutive blocks of one expert ----------------
    // A run is a maximal stretch of consecutive list entries with the same
    // expert and consecutive block indices; inside a run, entries at even
    // positions start a unit, which is a pair when the run continues.
    if (warp == 0) {
        int32_t nu = 0, run_start = 0, nruns = 0;
        int32_t run_min = 0x7fffffff, run_max = 0;          // units per run (this lane's run ends)
        for (int32_t base = 0; base < nact; base += 32) {
            const int32_t i = base + lane;
            const bool in = i < nact;
            const int32_t bxi = in ? act_bx[i] : 0;
            const int32_t ei = in ? act_e[i] : -1;
            const bool cont = in && i > 0 && act_e[i - 1] == ei && act_bx[i - 1] + 1 == bxi;
            const uint32_t starts = __ballot_sync(0xffffffffu, in && !cont);
            const uint32_t le = starts & (lane == 31 ? 0xffffffffu : ((2u << lane) - 1u));
            const int32_t rs = le ? base + 31 - __clz(le) : run_start;
            const bool ustart = in && (((i - rs) & 1) == 0);
            const bool next_cont = (i + 1 < nact) && act_e[i + 1] == ei && act_bx[i + 1] == bxi + 1;
            const uint32_t ub = __ballot_sync(0xffffffffu, ustart);
            if (ustart) {
                const int32_t idx = nu + __popc(ub & ((1u << lane) - 1u));
                units[idx] = static_cast<uint16_t>(bxi | (next_cont ? PAIR_BIT : 0));
                unit_rs[idx] = static_cast<uint16_t>(rs);
                unit_pos[idx] = static_cast<uint16_t>((i - rs) >> 1);
            }
            if (in && !next_cont) {                           // the run ends here
                run_nb[rs] = static_cast<uint16_t>(i - rs + 1);
                const int32_t ru = (i - rs + 2) >> 1;
                run_min = ru < run_min ? ru : run_min;
                run_max = ru > run_max ? ru : run_max;
            }
            nu += __popc(ub);
            nruns += __popc(starts);
            if (starts) run_start = base + 31 - __clz(starts);
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
            const int32_t a = __shfl_xor_sync(0xffffffffu, run_min, d);
            const int32_t b = __shfl_xor_sync(0xffffffffu, run_max, d);
            run_min = a < run_min ? a : run_min;
            run_max = b > run_max ? b : run_max;
        }
        if (lane == 0) {
            counts[0] = nruns;
            counts[1] = nu;
            counts[2] = 0;
            // every run has the same number of units, within the L2 budget:
            // per-expert groups are the runs, which the fixed-size order
            // with groups of about one run already gives
            counts[3] = run_min == run_max && run_max <= p.ph[PHASE == 2 ? 1 : 0].group ? -1 : 0;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (PHASE != 3 && p.expert_groups && counts[3] == 0) {
        // ---- 3. per-expert groups of the tile order -------------------------
        // A run's (an expert's) n units are split evenly into k = ceil(n / cap)
        // groups: group j starts at its unit floor(j * n / k).  Every thread
        // flags the units that start a group; the flags are compacted in unit
        // order.  When every group has the same size the cheaper fixed-size
        // decode gives the same order and is used instead.
        const int32_t cap = p.ph[PHASE == 2 ? 1 : 0].group;
        const int32_t nu = counts[1];
        int32_t ng = 0;
        for (int32_t base = 0; base < nu; base += NUM_THREADS) {
            const int32_t u = base + tid;
            int32_t flag = 0;
            if (u < nu) {
                const int32_t pos = unit_pos[u];
                const int32_t n = (run_nb[unit_rs[u]] + 1) >> 1;                 // the run's units
                flag = u == 0 || pos == 0;
                if (!flag && pos < n) {
                    const int32_t k = (n + cap - 1) / cap;
                    const int32_t j = (pos * k + n - 1) / n;                     // first group at or after pos
                    flag = j < k && (j * n) / k == pos;
                }
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
            if (flag) gstart[ng + before + __popc(ballot & ((1u << lane) - 1u))] = static_cast<uint16_t>(u);
            ng += total;
            __syncthreads();
        }
        const int32_t g0 = ng >= 2 ? gstart[1] : nu;                             // the first group's size
        int32_t same = 1;
        for (int32_t g = tid; g < ng; g += NUM_THREADS)
            if (gstart[g] != g * g0) same = 0;
        same = __syncthreads_and(same) && nu - (ng - 1) * g0 <= g0;
        if (tid == 0) {
            counts[2] = same ? 0 : ng;
            counts[3] = same ? g0 : 0;
        }
        __syncthreads();
    }
    const uint32_t tmem_base = *tmem_slot;
    volatile uint32_t* canary = reinterpret_cast<volatile uint32_t*>(
        smem + OFF_UNITS + units_bytes(p.num_blocks_m) * (PHASE != 3 && p.expert_groups ? 2 : 1));
    if (MOE_DEBUG && tid == 0) *canary = SMEM_CANARY;
    MOE_DCHECK(counts[1] <= p.num_blocks_m && counts[0] <= counts[1], p.status);
    const int32_t tiles1 = PHASE == 2 ? 0 : counts[1] * p.ph[0].n_tiles;
    const int32_t total_tiles = PHASE == 1 ? tiles1
                              : PHASE == 2 ? counts[1] * p.ph[1].n_tiles
                                           : tiles1 + counts[1] * p.ph[1].n_tiles;
    // With about one unit per expert run every weight byte is used once:
    // stream the weights through L2 with evict-first; otherwise keep them for
    // the expert's other units.
    const bool weights_streamed = 4 * counts[1] <= 5 * counts[0];
    // Tile-order group: about one expert's units (so a weight slice is shared
    // by all of them at once), at most what the host's L2 budget allows.
    const int32_t upe = counts[0] > 0 ? (counts[1] + counts[0] - 1) / counts[0] : 1;
    int32_t grp[2] = {p.ph[0].group < upe ? p.ph[0].group : upe, p.ph[1].group < upe ? p.ph[1].group : upe};
    if (PHASE != 3 && p.expert_groups && counts[3] > 0) grp[PHASE - 1] = counts[3];   // equal per-expert groups
    const int32_t ngroups = counts[2];
    MOE_DCHECK(ngroups == 0 || (ngroups <= counts[1] && gstart[0] == 0), p.status);
    auto tile_of = [&](const PhaseTile& pt) -> Tile {
        const PhaseParams& q = p.ph[pt.ph - 1];
        return ngroups > 0 ? decode_tile_groups(pt.t, units, gstart, ngroups, q.n_tiles, counts[1], rank)
                           : decode_tile(pt.t, units, q.n_tiles, counts[1], grp[pt.ph - 1], rank);
    };
    // Both CTAs' barriers are initialised and their prologue scratch in the
    // stage area is dead before either CTA's copies or commits reach the other.
    cluster_sync_all();

    // Phase 2 reads up_logits written by phase 1: wait for that grid here
    // (everything above only touched the dispatch tables).
    if (PHASE == 2 && p.tables_before_wait) pdl_wait_prior_grid();

    const int32_t cluster_id = static_cast<int32_t>(blockIdx.x) / CLUSTER;
    const int32_t n_clusters = static_cast<int32_t>(gridDim.x) / CLUSTER;

    if (warp == 0) {
        // ===================== TMA producer (both CTAs) =====================
        if (lane == 0) {
            const uint64_t pol_a = l2_policy_evict_normal();   // activations
            const uint64_t pol_b = weights_streamed ? l2_policy_evict_first() : l2_policy_evict_normal();
            const uint32_t leader_full = mapa_shared(bar_full, 0);
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            // Tile metadata is fetched ahead of use so that no global-memory
            // round trip sits between two tiles' copies: the expert of tile
            // t + 2C and that expert's size and padded offset for tile t + C
            // are loaded while tile t streams (C = number of clusters).
            auto expert_of = [&](int32_t tt) -> int32_t {
                if (tt >= total_tiles) return 0;
                const PhaseTile pt = phase_of<PHASE>(tt, tiles1);
                return __ldg(p.gidx + tile_of(pt).bx0);
            };
            int32_t e_cur = expert_of(cluster_id);
            int32_t size_cur = __ldg(p.sizes + e_cur), pad_cur = __ldg(p.padded + e_cur);
            int32_t e_next = expert_of(cluster_id + n_clusters);
            for (int32_t t = cluster_id; t < total_tiles && ok; t += n_clusters) {
                const PhaseTile pt = phase_of<PHASE>(t, tiles1);
                const PhaseParams& pp = p.ph[pt.ph - 1];
                const Tile ti = tile_of(pt);
                const int32_t e = e_cur;
                MOE_DCHECK(ti.u >= 0 && ti.u < counts[1] && ti.n >= 0 && ti.n < pp.n_tiles, p.status);
                MOE_DCHECK(ti.bx >= 0 && ti.bx < p.num_blocks_m && e >= 0 && e < p.n_experts, p.status);
                MOE_DCHECK(e == __ldg(p.gidx + ti.bx), p.status);
                MOE_DCHECK(pt.ph == 1 ? ti.n * 128 + 128 <= p.ph[0].n_extent
                                      : ti.n * BN + static_cast<int32_t>(rank) * 128 < p.ph[1].n_extent,
                           p.status);
                const CUtensorMap* a_map = pt.ph == 1 ? &map_x : &map_u;
                const CUtensorMap* a64_map = pt.ph == 1 ? &map_x64 : &map_u64;
                const CUtensorMap* a16_map = pt.ph == 1 ? &map_x16 : &map_u16;
                if (PHASE == 3 && pt.ph == 2) {
                    // this tile reads the unit's up_logits rows: wait until every
                    // phase-1 tile of the unit has stored them (both CTAs store
                    // rows of every tile), then order those generic stores before
                    // this thread's TMA (async proxy) reads
                    const int32_t u = ti.u;
                    const int32_t need = p.ph[0].n_tiles * CLUSTER;
                    if (!counter_wait_bounded(p.ready + u, need, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const int32_t size_next = __ldg(p.sizes + e_next), pad_next = __ldg(p.padded + e_next);
                const int32_t e_next2 = expert_of(t + 2 * n_clusters);
                // Rows of A to load, per CTA.  A pair (M = 256): this CTA's
                // block, as one 128-row box, or as 16-row boxes when it has at
                // most SMALL_ROWS valid rows (decode-like blocks; every other
                // block the full box, which moves faster than many small
                // boxes).  A lone block (M = 128): this CTA's 64 rows of it, as
                // one 64-row box, as 16-row boxes when at most SMALL_ROWS of
                // them are valid, or, when none is, a box that lies wholly past
                // the tensor's last row: it reads no memory and lands as
                // zeros, so the discarded rows multiply zeros (on a
                // power-capped GPU zeros measured ~2% faster than whatever the
                // stage last held).  Rows not loaded only feed discarded rows
                // of D.  The even CTA sets the expected byte count of both.
                struct APlan {
                    const CUtensorMap* map;
                    int32_t row;       // first row of the first box
                    int32_t boxes;     // boxes per K box of the stage
                    uint32_t bytes;    // bytes per K box
                };
                auto a_plan = [&](uint32_t r) -> APlan {
                    if (ti.pair) {
                        const int32_t bx = ti.bx0 + static_cast<int32_t>(r);
                        int32_t rows = size_cur - (bx * BM - pad_cur);
                        rows = rows > BM ? BM : (rows < 0 ? 0 : rows);
                        if (rows > SMALL_ROWS) return APlan{a_map, bx * BM, 1, static_cast<uint32_t>(A_BOX_BYTES)};
                        const int32_t n16 = (rows + 15) / 16;
                        return APlan{a16_map, bx * BM, n16, n16 * A16_BYTES};
                    }
                    int32_t rows = size_cur - (ti.bx0 * BM - pad_cur) - static_cast<int32_t>(r) * HALF_ROWS;
                    rows = rows > HALF_ROWS ? HALF_ROWS : (rows < 0 ? 0 : rows);
                    const int32_t row0 = ti.bx0 * BM + static_cast<int32_t>(r) * HALF_ROWS;
                    if (rows == 0) return APlan{a64_map, static_cast<int32_t>(p.rows_total), 1, A64_BYTES};
                    if (rows > SMALL_ROWS) return APlan{a64_map, row0, 1, A64_BYTES};
                    const int32_t n16 = (rows + 15) / 16;
                    return APlan{a16_map, row0, n16, n16 * A16_BYTES};
                };
                const APlan own = a_plan(rank);
                const uint32_t bytes_peer = leader ? a_plan(1).bytes : 0u;
                const uint32_t stage_tx = KSUB * (own.bytes + bytes_peer + 2 * B_BOX_BYTES);
                MOE_DCHECK(own.row == p.rows_total ||
                               static_cast<int64_t>(own.row) + (own.map == a_map ? BM : own.map == a64_map
                                                                                        ? HALF_ROWS
                                                                                        : 16 * own.boxes) <=
                                   p.rows_total,
                           p.status);
                MOE_DCHECK(own.boxes >= 1 && own.boxes <= (ti.pair ? SMALL_ROWS / 16 : HALF_ROWS / 16), p.status);
                for (int32_t kb = 0; kb < pp.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = leader_full + 8 * stage;
                    const uint32_t sa = sbase + OFF_STAGES + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE_BYTES;
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, stage_tx);
#pragma unroll
                    for (int ks = 0; ks < KSUB; ++ks) {
                        const int32_t k0 = (kb * KSUB + ks) * BK;
                        for (int32_t b = 0; b < own.boxes; ++b)
                            tma_load_2d_pair(sa + ks * A_BOX_BYTES + b * A16_BYTES, own.map, fb, k0, own.row + b * 16,
                                             pol_a);
                        if (pt.ph == 1) {
                            if (ti.pair) {
                                tma_load_3d_pair(sb + ks * B_BOX_BYTES, leader ? &map_gate : &map_up, fb, k0,
                                                 ti.n * 128, e, pol_b);
                            } else {
                                // this CTA's half of N: 64 gate rows, then the same 64 up rows
                                const int32_t wrow = ti.n * 128 + static_cast<int32_t>(rank) * HALF_ROWS;
                                tma_load_3d_pair(sb + ks * B_BOX_BYTES, &map_gate64, fb, k0, wrow, e, pol_b);
                                tma_load_3d_pair(sb + ks * B_BOX_BYTES + B_BOX_BYTES / 2, &map_up64, fb, k0, wrow, e,
                                                 pol_b);
                            }
                        } else {
                            tma_load_3d_pair(sb + ks * B_BOX_BYTES, &map_down, fb, k0,
                                             ti.n * BN + static_cast<int32_t>(rank) * 128, e, pol_b);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                e_cur = e_next;
                size_cur = size_next;
                pad_cur = pad_next;
                e_next = e_next2;
            }
            if (!ok) {
                // Let the copies already in flight land before the CTA exits.
                volatile int never = 0;
                if (leader) {
                    const int64_t n = issued < STAGES ? issued : STAGES;
                    for (int64_t i = 0; i < n; ++i) {
                        const int64_t idx = issued - 1 - i;
                        mbar_wait_bounded(bar_full + 8 * static_cast<uint32_t>(idx % STAGES),
                                          static_cast<uint32_t>((idx / STAGES) & 1), &never, DRAIN_LIMIT_NS);
                    }
                } else {
                    // the odd CTA's copies report to the even CTA's barriers:
                    // give them a bounded moment to land
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 1000000ull) { }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================== MMA issuer (even CTA only) =====================
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, acc = 0, aphase = 0;
            bool ok = true;
            for (int32_t t = cluster_id; t < total_tiles && ok; t += n_clusters) {
                if (!mbar_wait_bounded(bar_tempty + 8 * acc, aphase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const PhaseTile pt = phase_of<PHASE>(t, tiles1);
                const PhaseParams& pp = p.ph[pt.ph - 1];
                const int32_t k_blocks = pp.k_blocks;
                const uint32_t idesc = tile_of(pt).pair ? IDESC : IDESC_M128;
                for (int32_t kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = sbase + OFF_STAGES + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < KSUB * (BK / 16); ++kk) {
                        const uint32_t off = (kk / (BK / 16)) * A_BOX_BYTES + (kk % (BK / 16)) * 32;
                        const uint32_t offb = (kk / (BK / 16)) * B_BOX_BYTES + (kk % (BK / 16)) * 32;
                        tc_mma_f16_pair(d_tmem, smem_desc_k_sw128(sa + off), smem_desc_k_sw128(sb + offb),
                                        idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    // the slot may be refilled in both CTAs once these MMAs are done
                    tc_commit_pair_mc(bar_empty + 8 * stage, CLUSTER_MASK);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (!(p.drop_first_signal && t == cluster_id)) tc_commit_pair_mc(bar_tfull + 8 * acc, CLUSTER_MASK);
                acc ^= 1u;
                if (acc == 0) aphase ^= 1u;
            }
            // Every MMA this thread issued has finished once this arrives.
            volatile int never = 0;
            tc_commit_pair(bar_drain);
            mbar_wait_bounded(bar_drain, 0, &never, DRAIN_LIMIT_NS);
        }
        __syncwarp();
    } else {
        // ===================== epilogue (warps 2..5, both CTAs) =====================
        // A pair (M = 256): this CTA's block, row = TMEM lane, all 256 columns
        // of N.  A lone block (M = 128): this CTA's 64 rows (rank 0: rows
        // 0-63, rank 1: rows 64-127); lane quarters 0/1 hold rows 0-31 / 32-63
        // with N columns 0-127 and quarters 2/3 the same rows with N columns
        // 128-255, all in the first 128 TMEM columns of the accumulator.
        const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
        const uint32_t leader_tempty = mapa_shared(bar_tempty, 0);
        uint32_t acc = 0, aphase = 0;
        for (int32_t t = cluster_id; t < total_tiles; t += n_clusters) {
            const PhaseTile pt = phase_of<PHASE>(t, tiles1);
            const PhaseParams& pp = p.ph[pt.ph - 1];
            const Tile ti = tile_of(pt);
            int32_t e = 0, tok = 0;
            const int32_t actual = block_rows(p, ti.bx, &e, &tok);
            const int half = ti.pair ? 0 : (quarter >> 1);             // which 128 columns of N (M = 128)
            // rows [warp_row0, warp_row0 + 32) of the block are this warp's
            const int warp_row0 = ti.pair ? quarter * 32 : static_cast<int>(rank) * HALF_ROWS + (quarter & 1) * 32;
            const int row = warp_row0 + lane;                            // row of the block
            if (!mbar_wait_bounded(bar_tfull + 8 * acc, aphase, abort_flag, WAIT_LIMIT_NS)) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            const int64_t grow = static_cast<int64_t>(ti.bx) * BM + row;
            MOE_DCHECK(actual >= 0 && actual <= BM && grow < p.rows_total, p.status);
            MOE_DCHECK(!ti.pair || actual == 0 || __ldg(p.gidx + ti.bx0) == __ldg(p.gidx + ti.bx), p.status);
            const int64_t wrow = static_cast<int64_t>(ti.bx) * BM + warp_row0;
            if (pt.ph == 1) {
                // gate and up of output column j: TMEM columns j and j + 128
                // (pair), or, for this thread's half of N, columns j and j + 64
                // (M = 128), whose outputs are columns 64*half + j of the slice
                const int up_off = ti.pair ? 128 : 64;
                uint16_t* dst_row = pp.dst + grow * pp.n_extent + static_cast<int64_t>(ti.n) * 128 + half * 64;
                MOE_DCHECK(ti.n * 128 + 128 <= pp.n_extent, p.status);
#pragma unroll 1
                for (int c = 0; c < (warp_row0 < actual ? up_off / 32 : 0); ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, g);
                    tmem_ld_32x32b_x32(taddr + up_off + c * 32, u);
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
                uint16_t* dst0 = pp.dst + wrow * pp.n_extent;
                const int ncols = ti.pair ? BN : BN / 2;                 // TMEM columns this thread holds
#pragma unroll 1
                for (int c = 0; c < (warp_row0 < actual ? ncols / 32 : 0); c += 2) {   // 64 columns per pass
                    const int32_t col0 = ti.n * BN + half * (BN / 2) + c * 32;
                    MOE_DCHECK(col0 >= pp.n_extent || col0 + 64 <= pp.n_extent, p.status);
                    if (col0 >= pp.n_extent) break;             // partial last slice of H
                    uint4 el[8];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(taddr + (c + hh) * 32, v);
                        tmem_ld_wait();
                        uint32_t h[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            h[j] = pack_half2(__uint_as_float(v[2 * j]) * w, __uint_as_float(v[2 * j + 1]) * w);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            el[4 * hh + q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                    }
                    store_rows64(el, dst0 + col0, pp.n_extent, lane, warp_row0, actual);
                }
            }
            tc_fence_before_sync();
            // the accumulator may be reused once both CTAs have read their rows
            if (leader) mbar_arrive(bar_tempty + 8 * acc);
            else mbar_arrive_cluster(leader_tempty + 8 * acc);
            acc ^= 1u;
            if (acc == 0) aphase ^= 1u;
            if (PHASE == 3 && pt.ph == 1) {
                // Publish this CTA's up_logits rows of the tile to the phase-2
                // tiles of the unit, which read them with TMA: every storing
                // thread orders its stores before later async-proxy reads, the
                // four epilogue warps meet, then one thread releases a count.
                asm volatile("fence.proxy.async.global;" ::: "memory");
                asm volatile("bar.sync 1, %0;" ::"r"(NUM_EPI_THREADS) : "memory");
                if (warp == 2 && lane == 0) {
                    __threadfence();
                    atomicAdd(p.ready + ti.u, 1);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // Neither CTA leaves (or frees the pair's TMEM) while the other may still
    // write into its shared memory, arrive on its barriers or use the TMEM.
    cluster_sync_all();
    if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
    if (MOE_DEBUG && tid == 0) MOE_DCHECK(*canary == SMEM_CANARY, p.status);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

// Clusters of two that can be resident at once for a kernel with `smem`
// bytes of dynamic shared memory (cached per device, kernel and size).
template <int PHASE>
int max_clusters(size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(dev, smem);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(CLUSTER * 64);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<PHASE>, &cfg) != cudaSuccess) n = 0;
    cache[key] = n;
    return n;
}

}  // namespace

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

int64_t single_launch_workspace_bytes(int64_t num_blocks_m) {
    return ((4 * num_blocks_m + 255) / 256) * 256;
}

cudaError_t launch_fused_forward(const ForwardArgs& a, uint32_t flags, cudaStream_t stream, void* ready_ws) {
    if (!encode_fn()) return cudaErrorNotSupported;
    CUtensorMap map_x, map_x64, map_x16, map_gate, map_up, map_gate64, map_up64, map_u, map_u64, map_u16, map_down;
    const uint64_t rows = static_cast<uint64_t>(a.rows_total);
    const uint64_t H = static_cast<uint64_t>(a.hidden), I = static_cast<uint64_t>(a.intermediate);
    const uint64_t E = static_cast<uint64_t>(a.n_experts);
    if (!make_map_2d(&map_x, a.x, rows, H, BM) || !make_map_2d(&map_x64, a.x, rows, H, HALF_ROWS) ||
        !make_map_2d(&map_x16, a.x, rows, H, 16) ||
        !make_map_3d(&map_gate, a.gate_w, E, I, H, 128) || !make_map_3d(&map_up, a.up_w, E, I, H, 128) ||
        !make_map_3d(&map_gate64, a.gate_w, E, I, H, HALF_ROWS) ||
        !make_map_3d(&map_up64, a.up_w, E, I, H, HALF_ROWS) ||
        !make_map_2d(&map_u, a.up_logits, rows, I, BM) || !make_map_2d(&map_u64, a.up_logits, rows, I, HALF_ROWS) ||
        !make_map_2d(&map_u16, a.up_logits, rows, I, 16) || !make_map_3d(&map_down, a.down_w, E, H, I, 128))
        return cudaErrorInvalidValue;

    GemmParams p{};
    p.sizes = a.sizes;
    p.offsets = a.offsets;
    p.padded = a.padded;
    p.gidx = a.gidx;
    p.rw = a.rw;
    p.status = a.status;
    p.rows_total = a.rows_total;
    p.valid_total = a.valid_total;
    p.num_blocks_m = static_cast<int32_t>(a.num_blocks_m);
    p.n_experts = a.n_experts;
    p.ph[0].dst = a.up_logits;
    p.ph[0].k_blocks = a.hidden / (BK * KSUB);
    p.ph[0].n_tiles = a.intermediate / 128;
    p.ph[0].n_extent = a.intermediate;
    p.ph[1].dst = a.out;
    p.ph[1].k_blocks = a.intermediate / (BK * KSUB);
    p.ph[1].n_tiles = (a.hidden + BN - 1) / BN;
    p.ph[1].n_extent = a.hidden;
    // Group size of the tile order: as many units as keep their A rows
    // (256 rows x K fp16 per unit) within GROUP_A_BYTES, 1 to 32.
    auto group_for = [](int64_t k) {
        const int64_t per_unit = 2 * BM * k * 2;
        int64_t g = GROUP_A_BYTES / per_unit;
        return static_cast<int32_t>(g < 1 ? 1 : (g > 32 ? 32 : g));
    };
    p.ph[0].group = group_for(a.hidden);
    p.ph[1].group = group_for(a.intermediate);
    p.tables_before_wait = (flags & MOE_RUN_PHASE1) ? 1 : 0;
    p.ready = static_cast<int32_t*>(ready_ws);
    p.drop_first_signal = (flags & MOE_TEST_DROP_SIGNAL) ? 1 : 0;

    // One-phase launches order their tiles in per-expert groups when the
    // group table fits in shared memory beside the unit list (up to several
    // thousand blocks); otherwise, and for the single launch, in groups of
    // the average units per expert.
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return cudaErrorNoDevice;
    const bool groups_fit = smem_bytes_for(a.num_blocks_m, true) <= static_cast<size_t>(max_smem);
    const size_t smem = smem_bytes_for(a.num_blocks_m, groups_fit);
    const size_t smem3 = smem_bytes_for(a.num_blocks_m, false);
    p.expert_groups = groups_fit ? 1 : 0;
    cudaError_t err = cudaSuccess;
    if ((err = cudaFuncSetAttribute(grouped_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem))) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grouped_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem))) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grouped_gemm_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem3))) != cudaSuccess)
        return err;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    const bool both = (flags & (MOE_RUN_PHASE1 | MOE_RUN_PHASE2)) == (MOE_RUN_PHASE1 | MOE_RUN_PHASE2);
    if (ready_ws != nullptr && both) {
        // both phases in one persistent launch; the per-unit counters start at zero
        err = cudaMemsetAsync(ready_ws, 0, static_cast<size_t>(single_launch_workspace_bytes(a.num_blocks_m)),
                              stream);
        if (err != cudaSuccess) return err;
        const int nc = max_clusters<3>(smem3);
        if (nc <= 0) return cudaErrorNoDevice;
        cfg.gridDim = dim3(static_cast<unsigned>(CLUSTER * nc));
        cfg.dynamicSmemBytes = smem3;
        cfg.numAttrs = 2;
        p.expert_groups = 0;
        return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<3>, map_x, map_x64, map_x16, map_gate, map_up,
                                  map_gate64, map_up64, map_u, map_u64, map_u16, map_down, p);
    }
    if (flags & MOE_RUN_PHASE1) {
        const int nc = max_clusters<1>(smem);
        if (nc <= 0) return cudaErrorNoDevice;
        cfg.gridDim = dim3(static_cast<unsigned>(CLUSTER * nc));
        cfg.numAttrs = 2;   // cluster + programmatic dependent launch
        err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<1>, map_x, map_x64, map_x16, map_gate, map_up,
                                 map_gate64, map_up64, map_x, map_x64, map_x16, map_gate, p);
        if (err != cudaSuccess) return err;
        p.drop_first_signal = 0;
    }
    if (flags & MOE_RUN_PHASE2) {
        // Phase 2 may start its prologue (tables, TMEM, barriers) while phase 1
        // drains; it waits for phase 1's results before its first load.  Both
        // phases are launched with programmatic dependent launch.
        const int nc = max_clusters<2>(smem);
        if (nc <= 0) return cudaErrorNoDevice;
        cfg.gridDim = dim3(static_cast<unsigned>(CLUSTER * nc));
        cfg.numAttrs = (flags & MOE_NO_PDL) ? 1 : 2;
        err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<2>, map_u, map_u64, map_u16, map_down, map_down,
                                 map_down, map_down, map_u, map_u64, map_u16, map_down, p);
    }
    return err;
}

}  // namespace moe
