// Router: logits = x · W_gᵀ (fp32), softmax over all experts, top-k
// ("MetaX-TileLang工具链", §2.4: logits = W_g(x), scores = softmax(logits),
// topk_scores, topk_indices = topk(scores)).
//
// One cluster of S CTAs per 128-token tile, one tcgen05 MMA tile of M = 128
// tokens and N = n_experts rounded up to 16 (at most 256).  When there are
// fewer tiles than SMs the tile's K (hidden) is split over the S CTAs of its
// cluster, so that tiles x S SMs stream x instead of one per tile.  Warp 0
// streams the CTA's K range of x and W_g with TMA through a ring of up to
// eight 64-wide K stages (as many as shared memory holds beside the slots),
// warp 1 owns TMEM and issues the MMAs, warps 2-17 are the epilogue.  With
// as many tiles as SMs or more there is no K split; tiles then pair up on
// 2-SM MMAs (M = 256) in which each CTA holds its own tile's x and half of
// W_g's rows, so each SM receives a third fewer bytes.  The epilogue:
//  1. The tile's valid tokens are shared out evenly: CTA r owns tokens
//     r*R .. r*R + R - 1 (R = the valid tokens / S, rounded up).  Every CTA
//     writes its fp32 logits (partial sums over its K range when S > 1) from
//     TMEM into the owners' shared memory, one row per (source CTA, token):
//     rows for other CTAs as st.async stores that count their bytes on the
//     owner's mbarrier, so an owner waits for exactly its own rows and no
//     cluster-wide barrier sits between the MMAs and the top-k.
//  2. Each owner sums the S partial rows of its tokens in rank order, T lanes
//     per token, and selects the top-k in three steps.  (a) Every lane takes
//     the maxima of m groups of its logits; the k-th largest of the token's
//     T*m group maxima, theta, is at most the k-th largest logit, because k
//     distinct logits (the group maxima) reach it.  (b) The logits >= theta
//     are the candidates (typically k to 2k of them); the same pass sums
//     exp(l - max) for the softmax.  (c) Each candidate's rank is the number
//     of candidates that rank above it (a larger logit, or an equal one with
//     a lower expert index), and a candidate of rank q < k is output q.  A
//     token whose candidates overflow the list (many equal logits) takes the
//     general path instead: per-lane sorted lists of the best KMAX logits
//     (bitonic sorts), merged over the token's lanes in butterfly rounds.
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
constexpr int R_A_BYTES = R_BM * R_BK * 2;           // 16 KB of x per stage
constexpr int R_MAX_STAGES = 8;
constexpr int R_MIN_STAGES = 2;
constexpr int R_EPI_WARPS = 16;
constexpr int R_EPI_THREADS = 32 * R_EPI_WARPS;
constexpr int R_THREADS = 64 + R_EPI_THREADS;        // producer, MMA, epilogue warps
constexpr int R_MAX_E = 256;                         // MOE_ROUTER_MAX_EXPERTS
constexpr int R_CMAX = 32;                           // candidate list length per token
constexpr int R_CSTRIDE = 2 * R_CMAX + 4;            // words per token's list (16-byte rows, == 4 mod 32)
constexpr int R_MMAX = 8;                            // group maxima per lane
constexpr uint64_t R_WAIT_NS = 2000000000ull;
constexpr uint64_t R_DRAIN_NS = 200000000ull;
constexpr int R_MAX_SPLIT = 8;                       // CTAs per cluster (the portable cluster size)
constexpr int R_SMEM_MAX = 227 * 1024;               // dynamic shared memory asked for at most
constexpr int R_NUM_BARS = 2 * R_MAX_STAGES + 3;     // full, empty, tfull, drain, slots
constexpr int R_MISC_BYTES = R_NUM_BARS * 8 + 16;    // barriers, TMEM slot, abort flag
constexpr int R_CAND_BYTES = R_BM * R_CSTRIDE * 4;  // the lists of 128 tokens

static_assert(R_MAX_E == MOE_ROUTER_MAX_EXPERTS, "router expert limit");

struct RouterParams {
    int64_t n_tokens;
    int32_t n_experts;
    int32_t n_pad;         // n_experts rounded up to 16
    int32_t tmem_cols;     // power of two >= max(32, n_pad)
    int32_t top_k;
    int32_t k_blocks;      // hidden / 64
    int32_t stages;        // ring stages (R_MIN_STAGES .. R_MAX_STAGES)
    int32_t stage_bytes;   // 16 KB of x + n_pad rows of W_g, 64 wide
    int32_t rs;            // floats per slot row: >= n_pad, == 4 mod 32
    int32_t off_slots;     // byte offsets from the 1024-aligned base
    int32_t off_cand;
    int32_t off_bars;
    int32_t* topk_ids;
    float* topk_weights;
    int32_t* status;
};

// Shared-memory layout for n_pad experts, S CTAs per cluster (or a pair that
// splits W_g's rows) and at most kb K blocks per CTA.  The ring comes first.  With S = 1 the slots and the
// candidate lists reuse the ring (the CTA's own MMAs are done before they are
// written); with S > 1 other CTAs write the slots while this CTA's MMAs may
// still run, so the slots get their own region and only the lists reuse the
// ring.  Returns false when no layout with R_MIN_STAGES stages fits in
// smem_max bytes.
struct RouterLayout {
    int stages, stage_bytes, rs, off_slots, off_cand, off_bars;
    size_t smem;           // dynamic shared memory to request (with alignment slack)
};

__host__ __device__ constexpr int slot_stride(int n_pad) {
    return n_pad + (((4 - n_pad) % 32) + 32) % 32;
}

bool router_layout(int n_pad, int S, bool pair, int kb, int smem_max, RouterLayout* L) {
    L->stage_bytes = R_A_BYTES + (pair ? n_pad / 2 : n_pad) * R_BK * 2;
    L->rs = slot_stride(n_pad);
    const int slot_bytes = R_BM * L->rs * 4;
    const int budget = smem_max - 1024 - R_MISC_BYTES;
    int ring_cap = budget - (S > 1 ? slot_bytes : 0);
    int stages = ring_cap / L->stage_bytes;
    if (stages > R_MAX_STAGES) stages = R_MAX_STAGES;
    if (stages > kb) stages = kb < R_MIN_STAGES ? R_MIN_STAGES : kb;
    if (stages < R_MIN_STAGES) return false;
    L->stages = stages;
    int ring = stages * L->stage_bytes;
    if (S > 1) {
        L->off_slots = ring;
        L->off_cand = 0;
        if (ring < R_CAND_BYTES) return false;   // the lists must stay clear of the slots
        ring += slot_bytes;
    } else {
        L->off_slots = 0;
        L->off_cand = slot_bytes;
        if (ring < slot_bytes + R_CAND_BYTES) ring = slot_bytes + R_CAND_BYTES;
    }
    L->off_bars = ring;
    L->smem = 1024 + static_cast<size_t>(ring) + R_MISC_BYTES;
    return L->smem <= static_cast<size_t>(smem_max);
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
// k_blocks*(r+1)/S.  KMAX: the list length of the general top-k path
// (>= top_k).  PAIR (with S = 1): clusters of two CTAs, each with its own
// tile, share one 2-SM MMA of M = 256 tokens: each CTA loads its tile's x
// and half of W_g's rows, so each SM receives a third fewer bytes.
template <int S, int KMAX, bool PAIR>
__global__ void __launch_bounds__(R_THREADS, 1)
router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
              const RouterParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + static_cast<uint32_t>(p.off_bars);
    const uint32_t bar_empty = bar_full + 8 * R_MAX_STAGES;
    const uint32_t bar_tfull = bar_empty + 8 * R_MAX_STAGES;
    const uint32_t bar_drain = bar_tfull + 8;
    const uint32_t bar_slots = bar_drain + 8;   // the owner's rows from the other CTAs have landed
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + p.off_bars + R_NUM_BARS * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_bars + R_NUM_BARS * 8 + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b_bytes = static_cast<uint32_t>(PAIR ? p.n_pad / 2 : p.n_pad) * R_BK * 2;   // W_g rows per stage
    static_assert(!PAIR || S == 1, "a pair splits W_g, not K");
    const uint32_t rank = S > 1 ? cluster_cta_rank() : 0u;          // K-split rank
    const uint32_t prank = PAIR ? cluster_cta_rank() : 0u;         // rank in the pair
    const bool leader = prank == 0;
    const int32_t row0 = static_cast<int32_t>(blockIdx.x / S) * R_BM;
    // the tile's valid tokens, shared out evenly over the cluster's CTAs
    const int64_t left = p.n_tokens - row0;                       // <= 0: a pair's spare CTA
    const int32_t rows_valid = left < 0 ? 0 : (left < R_BM ? static_cast<int32_t>(left) : R_BM);
    const int32_t rows_own = (rows_valid + S - 1) / S;
    int32_t own_n = rows_valid - static_cast<int32_t>(rank) * rows_own;
    own_n = own_n < 0 ? 0 : (own_n > rows_own ? rows_own : own_n);
    const int RS = p.rs;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_slots, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (S > 1) {
            // the bytes of the rows the other S - 1 CTAs store here
            const uint32_t bytes = static_cast<uint32_t>((S - 1) * own_n * p.n_pad * 4);
            if (bytes) mbar_arrive_expect_tx(bar_slots, bytes);
            else mbar_arrive(bar_slots);
        }
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_x);
        tma_prefetch_map(&map_w);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(sbase + static_cast<uint32_t>(p.off_bars + R_NUM_BARS * 8),
                            static_cast<uint32_t>(p.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(sbase + static_cast<uint32_t>(p.off_bars + R_NUM_BARS * 8), static_cast<uint32_t>(p.tmem_cols));
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // every CTA's slot barrier is initialised before any CTA stores into it
    // (waited for just before the stores)
    if (S > 1) cluster_arrive_relaxed();
    // a pair: both CTAs' barriers exist before the odd CTA's copies or the
    // leader's commits reach them
    if (PAIR) cluster_sync_all();
    const uint32_t tmem_base = *tmem_slot;
    const int32_t kb_begin = static_cast<int32_t>((static_cast<int64_t>(p.k_blocks) * rank) / S);
    const int32_t kb_end = static_cast<int32_t>((static_cast<int64_t>(p.k_blocks) * (rank + 1)) / S);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_normal();
            int32_t stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int32_t kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = sbase + static_cast<uint32_t>(stage * p.stage_bytes);
                if (PAIR) {
                    // both CTAs' copies complete on the leader's barrier
                    const uint32_t fb = mapa_shared(bar_full + 8 * stage, 0);
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * (R_A_BYTES + b_bytes));
                    tma_load_2d_pair(sa, &map_x, fb, kb * R_BK, row0, pol);
                    tma_load_2d_pair(sa + R_A_BYTES, &map_w, fb, kb * R_BK,
                                     static_cast<int32_t>(prank) * (p.n_pad / 2), pol);
                } else {
                    const uint32_t fb = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(fb, R_A_BYTES + b_bytes);
                    tma_load_2d(sa, &map_x, fb, kb * R_BK, row0, pol);
                    tma_load_2d(sa + R_A_BYTES, &map_w, fb, kb * R_BK, 0, pol);
                }
                ++issued;
                if (++stage == p.stages) { stage = 0; phase ^= 1u; }
            }
            if (!ok && leader) {
                volatile int never = 0;
                const int64_t n = issued < p.stages ? issued : p.stages;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t idx = issued - 1 - i;
                    mbar_wait_bounded(bar_full + 8 * static_cast<uint32_t>(idx % p.stages),
                                      static_cast<uint32_t>((idx / p.stages) & 1), &never, R_DRAIN_NS);
                }
            } else if (!ok) {
                // the odd CTA's copies report to the leader's barriers: give
                // them a bounded moment to land
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) { }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_f16_f32acc(PAIR ? 2 * R_BM : R_BM, static_cast<uint32_t>(p.n_pad));
            int32_t stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int32_t kb = kb_begin; kb < kb_end; ++kb) {
                if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sa = sbase + static_cast<uint32_t>(stage * p.stage_bytes);
                const uint32_t sb = sa + R_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < R_BK / 16; ++kk) {
                    const uint64_t ad = smem_desc_k_sw128(sa + kk * 32), bd = smem_desc_k_sw128(sb + kk * 32);
                    const uint32_t acc = (kb != kb_begin || kk != 0) ? 1u : 0u;
                    if (PAIR) tc_mma_f16_pair(tmem_base, ad, bd, idesc, acc);
                    else tc_mma_f16(tmem_base, ad, bd, idesc, acc);
                }
                // the stage may be refilled (in both CTAs of a pair) once these MMAs are done
                if (PAIR) tc_commit_pair_mc(bar_empty + 8 * stage, 0x3);
                else tc_commit(bar_empty + 8 * stage);
                if (++stage == p.stages) { stage = 0; phase ^= 1u; }
            }
            if (ok) {
                if (PAIR) tc_commit_pair_mc(bar_tfull, 0x3);
                else tc_commit(bar_tfull);
            }
            volatile int never = 0;
            if (PAIR) tc_commit_pair(bar_drain);
            else tc_commit(bar_drain);
            mbar_wait_bounded(bar_drain, 0, &never, R_DRAIN_NS);
        }
        __syncwarp();
    } else {
        if (mbar_wait_bounded(bar_tfull, 0, abort_flag, R_WAIT_NS)) tc_fence_after_sync();
        __syncwarp();
    }
    if (S > 1) cluster_wait_acquire();

    // ---- step 1: TMEM -> the owners' slot rows.  Warp w reads TMEM lanes
    // 32*(w%4) .. +31 (one token each); the four warps of a lane quarter take
    // every fourth group of 8 columns.  Slot row (source rank s, owned token
    // g) starts at float (s * rows_own + g) * RS of the slot region.
    if (warp >= 2 && !*abort_flag) {
        const int quarter = warp & 3;
        const int cpart = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const bool valid = row < rows_valid;                 // rows past the last token are not stored
        const int owner = valid ? row / rows_own : 0;
        const int g = row - owner * rows_own;
        const uint32_t off = static_cast<uint32_t>(p.off_slots) +
                             4u * static_cast<uint32_t>((static_cast<int>(rank) * rows_own + g) * RS);
        const bool remote = S > 1 && owner != static_cast<int>(rank);
        const uint32_t raddr = remote ? mapa_shared(sbase + off, static_cast<uint32_t>(owner)) : 0u;
        const uint32_t rbar = remote ? mapa_shared(bar_slots, static_cast<uint32_t>(owner)) : 0u;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        // all of the warp's column groups (at most 8: n_pad <= 256) in flight at once
        uint32_t v[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (8 * cpart + 32 * i < p.n_pad) tmem_ld_32x32b_x8(taddr + 8 * cpart + 32 * i, v[i]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int32_t c0 = 8 * cpart + 32 * i;
            if (!valid || c0 >= p.n_pad) continue;
            const float f0 = __uint_as_float(v[i][0]), f1 = __uint_as_float(v[i][1]), f2 = __uint_as_float(v[i][2]),
                        f3 = __uint_as_float(v[i][3]), f4 = __uint_as_float(v[i][4]), f5 = __uint_as_float(v[i][5]),
                        f6 = __uint_as_float(v[i][6]), f7 = __uint_as_float(v[i][7]);
            if (remote) {
                st_async_v4_f32(raddr + 4u * c0, f0, f1, f2, f3, rbar);
                st_async_v4_f32(raddr + 4u * c0 + 16u, f4, f5, f6, f7, rbar);
            } else {
                float4* d = reinterpret_cast<float4*>(smem + off + 4u * c0);
                d[0] = make_float4(f0, f1, f2, f3);
                d[1] = make_float4(f4, f5, f6, f7);
            }
        }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (warp >= 2) named_bar_sync(1, R_EPI_THREADS);        // this CTA's own rows are in place
    // waited for at the end: no CTA exits while another may still store into it
    if (S > 1) cluster_arrive_relaxed();

    // ---- step 2: the top-k of each owned token, T lanes per token
    if (warp >= 2) {
        bool ok = !*abort_flag;
        if (S > 1 && own_n > 0 && ok) ok = mbar_wait_bounded<true>(bar_slots, 0, abort_flag, R_WAIT_NS);
        ok = __all_sync(0xffffffffu, ok);
        // lanes per token: a power of two, 4..32, whose chunks of 4 tile the
        // n_pad columns exactly
        int T = 32;
        while (T > 4 && (p.n_pad % (4 * T) != 0 || T * rows_own > R_EPI_THREADS)) T >>= 1;
        const int et = tid - 64;
        const int g = et / T;                                 // owned token
        const int j = et & (T - 1);                           // lane within the token
        if (ok && (et & ~31) / T < own_n) {                   // warp-uniform: the warp has a live token
            const bool live = g < own_n;
            const int64_t t = static_cast<int64_t>(row0) + static_cast<int>(rank) * rows_own + g;
            const int nq = p.n_pad / (4 * T);                 // float4 chunks per lane
            int m = 1;                                        // group maxima per lane
            while (m < R_MMAX && T * m < 2 * p.top_k && nq % (2 * m) == 0) m <<= 1;
            const int qpg = nq / m;                           // chunks per group
            const int ng = T * m;                             // group maxima per token
            const float* row_s0 = reinterpret_cast<const float*>(smem + p.off_slots) + g * RS;
            const int sstride = rows_own * RS;                // floats between two source ranks' rows
            // chunk q of this lane: experts 4(j + qT) .. +3, the S partial rows summed in rank order
            auto chunk = [&](int q) {
                const int c = 4 * (j + q * T);
                float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    const float4 b = *reinterpret_cast<const float4*>(row_s0 + s * sstride + c);
                    a.x += b.x;
                    a.y += b.y;
                    a.z += b.z;
                    a.w += b.w;
                }
                return a;
            };
            auto logit = [&](int32_t e) {
                float l = 0.0f;
#pragma unroll
                for (int s = 0; s < S; ++s) l += row_s0[s * sstride + e];
                return l;
            };
            float* list = reinterpret_cast<float*>(smem + p.off_cand) + g * R_CSTRIDE;   // (logit, expert) pairs
            const int n_e = p.n_experts;
            // A lane whose logits fit one list (at most KMAX) in a token of at
            // most 8 lanes (three merge rounds) takes the list path directly;
            // every other token selects through theta first.
            const bool direct = 4 * nq <= KMAX && T <= 8;
            float mx = -INFINITY, sum = 0.0f;                 // the token's max logit and sum of exp(l - mx)
            bool general = true;
            if (!direct) {
                // (a) group maxima (padding experts count as -inf; NaN never wins
                // a max), kept in registers and in the list for the token's lanes
                float gm[R_MMAX];
#pragma unroll
                for (int a = 0; a < R_MMAX; ++a) gm[a] = -INFINITY;
                if (live) {
#pragma unroll
                    for (int a = 0; a < R_MMAX; ++a) {
                        if (a >= m) break;
                        for (int qq = 0; qq < qpg; ++qq) {
                            const int q = a * qpg + qq;
                            const float4 v = chunk(q);
                            const int e0 = 4 * (j + q * T);
                            gm[a] = fmaxf(gm[a], e0 < n_e ? v.x : -INFINITY);
                            gm[a] = fmaxf(gm[a], e0 + 1 < n_e ? v.y : -INFINITY);
                            gm[a] = fmaxf(gm[a], e0 + 2 < n_e ? v.z : -INFINITY);
                            gm[a] = fmaxf(gm[a], e0 + 3 < n_e ? v.w : -INFINITY);
                        }
                        list[j * m + a] = gm[a];
                    }
                }
                float th = INFINITY;
#pragma unroll
                for (int a = 0; a < R_MMAX; ++a) mx = fmaxf(mx, gm[a]);
                __syncwarp();
                // theta: the k-th largest of the token's ng <= 32 group maxima
                // (the smallest of them with fewer than k others above it)
                if (live) {
                    float4 all[8];
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4)
                        all[i4] = 4 * i4 < ng ? reinterpret_cast<const float4*>(list)[i4]
                                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
                    for (int a = 0; a < R_MMAX; ++a) {
                        if (a >= m) break;
                        int above = 0;
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4)
                            above += (all[i4].x > gm[a] ? 1 : 0) + (all[i4].y > gm[a] ? 1 : 0) +
                                     (all[i4].z > gm[a] ? 1 : 0) + (all[i4].w > gm[a] ? 1 : 0);
                        if (above < p.top_k) th = fminf(th, gm[a]);
                    }
                }
                for (int d = 1; d < T; d <<= 1) {
                    th = fminf(th, __shfl_xor_sync(0xffffffffu, th, d));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
                }
                __syncwarp();                                     // the maxima are read: the list is free
                // (b) candidates (logit >= theta): a bit per value of this lane,
                // then one prefix sum over the token's lanes places them in the
                // list; the same pass sums exp(l - max)
                uint64_t cbits = 0;                               // bit 4q + i: value i of chunk q (V <= 64)
                if (live) {
                    for (int q = 0; q < nq; ++q) {
                        const float4 v4 = chunk(q);
                        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (4 * (j + q * T) + i >= n_e) continue;
                            sum += __expf(vv[i] - mx);
                            if (vv[i] >= th) cbits |= 1ull << (4 * q + i);
                        }
                    }
                }
                const int mine = __popcll(cbits);
                int incl = mine;                                  // inclusive prefix over the token's lanes
                for (int d = 1; d < T; d <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, d);
                    if (j >= d) incl += o;
                    sum += __shfl_xor_sync(0xffffffffu, sum, d);
                }
                const int c = __shfl_sync(0xffffffffu, incl, (lane & ~(T - 1)) + T - 1);   // the token's candidates
                for (int pos = incl - mine; cbits != 0 && pos < R_CMAX; ++pos) {
                    const int li = __ffsll(static_cast<long long>(cbits)) - 1;
                    cbits &= cbits - 1;
                    const int e = 4 * (j + (li >> 2) * T) + (li & 3);
                    reinterpret_cast<float2*>(list)[pos] = make_float2(logit(e), __int_as_float(e));
                }
                __syncwarp();
                general = __any_sync(0xffffffffu, live && (c > R_CMAX || ng < p.top_k));
                if (!general) {
                    // (c) rank the candidates: the k best are exactly those of rank < k
                    if (live) {
                        const float2* cl = reinterpret_cast<const float2*>(list);
                        const float inv = 1.0f / sum;
                        for (int i = j; i < c; i += T) {
                            const float2 me = cl[i];
                            const int32_t ei = __float_as_int(me.y);
                            int r = 0;
#pragma unroll 4
                            for (int i2 = 0; i2 < c; ++i2) {
                                const float2 o = cl[i2];
                                r += ranks_above(o.x, __float_as_int(o.y), me.x, ei) ? 1 : 0;
                            }
                            if (r < p.top_k) {
                                MOE_DCHECK(ei >= 0 && ei < n_e, p.status);
                                p.topk_ids[t * p.top_k + r] = ei;
                                p.topk_weights[t * p.top_k + r] = __expf(me.x - mx) * inv;
                            }
                        }
                        // fewer candidates than k (NaN logits never rank): empty outputs
                        for (int r = c + j; r < p.top_k; r += T) {
                            p.topk_ids[t * p.top_k + r] = -1;
                            p.topk_weights[t * p.top_k + r] = 0.0f;
                        }
                    }
                }
            }
            if (general) {
                // general path: lane j keeps a sorted list of its best KMAX of
                // experts j, j + T, ..., built KMAX at a time with bitonic
                // sorts; the token's lanes merge their lists in butterfly rounds
                float bv[KMAX];
                int32_t bi[KMAX];
#pragma unroll
                for (int q = 0; q < KMAX; ++q) {
                    bv[q] = -INFINITY;
                    bi[q] = 0x7fffffff;
                }
                for (int32_t e0 = j; live && e0 < n_e; e0 += KMAX * T) {
                    float cv[KMAX];
                    int32_t ci[KMAX];
#pragma unroll
                    for (int q = 0; q < KMAX; ++q) {
                        const int32_t e = e0 + q * T;
                        cv[q] = e < n_e ? logit(e) : -INFINITY;
                        ci[q] = e < n_e ? e : 0x7fffffff;
                    }
                    bitonic_sort_desc<KMAX>(cv, ci);
                    merge_topk<KMAX>(bv, bi, cv, ci);
                }
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
                if (direct) {
                    // the merged list is the same in all of the token's lanes
                    mx = bv[0];
                    for (int32_t e = j; live && e < n_e; e += T) sum += __expf(logit(e) - mx);
                    for (int d = 1; d < T; d <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
                }
                if (live && j == 0) {
#pragma unroll
                    for (int q = 0; q < KMAX; ++q) {
                        if (q < p.top_k) {
                            // an id in range: a finite logit ranked q-th (NaN logits never rank)
                            MOE_DCHECK(bi[q] >= 0 && bi[q] < n_e, p.status);
                            p.topk_ids[t * p.top_k + q] = bi[q] < n_e ? bi[q] : -1;
                            p.topk_weights[t * p.top_k + q] = bi[q] < n_e ? __expf(bv[q] - mx) / sum : 0.0f;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (S > 1) cluster_wait_acquire();
    // a pair: neither CTA frees the pair's TMEM or leaves while the other may
    // still use it or its shared memory
    if (PAIR) cluster_sync_all();
    if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after_sync();
        if (PAIR) tmem_dealloc_pair(tmem_base, static_cast<uint32_t>(p.tmem_cols));
        else tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
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
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return cudaErrorNoDevice;
    const int smem_max = optin < R_SMEM_MAX ? optin : R_SMEM_MAX;
    auto layout_for = [&](int64_t sp, bool pair, RouterLayout* L) {
        const int kb = static_cast<int>((p.k_blocks + sp - 1) / sp);
        return router_layout(p.n_pad, static_cast<int>(sp), pair, kb, smem_max, L);
    };
    // K split: the largest power of two S <= R_MAX_SPLIT with tiles x S
    // within the SM count, at most one CTA per 64-wide K block, and a
    // shared-memory layout that fits
    RouterLayout L{};
    int64_t split = 1;
    while (split * 2 <= R_MAX_SPLIT && tiles * split * 2 <= device_sm_count() && split * 2 <= p.k_blocks &&
           layout_for(split * 2, false, &L))
        split *= 2;
    const int kmax = top_k <= 4 ? 4 : top_k <= 8 ? 8 : 16;
    auto kernel_for = [kmax](int64_t sp, bool pair) {
        if (pair) return kmax == 4 ? router_kernel<1, 4, true> : kmax == 8 ? router_kernel<1, 8, true>
                                                                             : router_kernel<1, 16, true>;
        if (kmax == 4)
            return sp >= 8 ? router_kernel<8, 4, false> : sp == 4 ? router_kernel<4, 4, false>
                 : sp == 2 ? router_kernel<2, 4, false> : router_kernel<1, 4, false>;
        if (kmax == 8)
            return sp >= 8 ? router_kernel<8, 8, false> : sp == 4 ? router_kernel<4, 8, false>
                 : sp == 2 ? router_kernel<2, 8, false> : router_kernel<1, 8, false>;
        return sp >= 8 ? router_kernel<8, 16, false> : sp == 4 ? router_kernel<4, 16, false>
             : sp == 2 ? router_kernel<2, 16, false> : router_kernel<1, 16, false>;
    };
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(R_THREADS);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a cluster shape the device can place (clusters live inside one GPC);
    // the answer is cached per device, kernel and shared-memory size
    static std::mutex mu;
    static std::map<std::tuple<int, int, int64_t, bool, size_t>, bool> placeable;
    auto placeable_for = [&](int64_t sp, bool pair) -> int {   // 1 yes, 0 no, -1 error
        const int64_t cl = pair ? 2 : sp;
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_tuple(dev, kmax, sp, pair, L.smem);
        auto it = placeable.find(key);
        if (it == placeable.end()) {
            if (cudaFuncSetAttribute(kernel_for(sp, pair), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
                cudaSuccess)
                return -1;
            attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
            cfg.gridDim = dim3(static_cast<unsigned>(cl));
            cfg.dynamicSmemBytes = L.smem;
            int n = 0;
            const bool ok = cl == 1 || (cudaOccupancyMaxActiveClusters(&n, kernel_for(sp, pair), &cfg) == cudaSuccess &&
                                        n > 0);
            if (!ok) cudaGetLastError();
            it = placeable.emplace(key, ok).first;
        }
        return it->second ? 1 : 0;
    };
    // Without a K split (as many tiles as SMs, or more), tiles pair up on
    // 2-SM MMAs that split W_g's rows when that moves fewer bytes per SM
    // (at least 64 experts' rows)
    bool pair = false;
    for (; split >= 1; split /= 2) {
        if (!layout_for(split, false, &L)) {
            if (split == 1) return cudaErrorInvalidConfiguration;
            continue;
        }
        const int r = placeable_for(split, false);
        if (r < 0) return cudaErrorInvalidConfiguration;
        if (r == 1) break;
    }
    if (split == 1 && tiles >= 2 && p.n_pad >= 64) {
        RouterLayout L1 = L;
        if (layout_for(1, true, &L)) {
            const int r = placeable_for(1, true);
            if (r < 0) return cudaErrorInvalidConfiguration;
            pair = r == 1;
        }
        if (!pair) L = L1;
    }
    if (pair && !router_map(&map_w, router_w, static_cast<uint64_t>(n_experts), static_cast<uint64_t>(hidden),
                            static_cast<uint32_t>(p.n_pad / 2)))
        return cudaErrorInvalidValue;
    p.stages = L.stages;
    p.stage_bytes = L.stage_bytes;
    p.rs = L.rs;
    p.off_slots = L.off_slots;
    p.off_cand = L.off_cand;
    p.off_bars = L.off_bars;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pair ? 2 : split);
    cfg.gridDim = dim3(static_cast<unsigned>(pair ? (tiles + 1) / 2 * 2 : tiles * split));
    cfg.dynamicSmemBytes = L.smem;
    return cudaLaunchKernelEx(&cfg, kernel_for(split, pair), map_x, map_w, p);
}

}  // namespace moe
