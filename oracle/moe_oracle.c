/*
 * CPU oracle for the routed fused-MoE expert GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, __graft_entry__.smoke() and the cpu_baseline /
 * reference legs of bench.py use it.  It shares no code, header, table or
 * constant with the CUDA library; it is a plain, slow restatement of what the
 * pages define, written so that it can be checked against them by eye.
 *
 * Sources (page title, then section):
 *   [P1] "Fused MoE GEMM 提交说明" — §算子来源 (the expert MLP semantics),
 *        §实现要点 (padded vs compact indexing, padding rows neither computed nor
 *        written), §完整算子代码 (block_token = 128, fp16 data, fp32 accumulation,
 *        SiLU·up stored to the fp16 up_logits workspace, routed weight applied to
 *        the fp32 accumulator before the fp16 store of out).
 *   [P2] "moe_dispatch_contract.py" (TileLang tutorial, ch. 18) — the module
 *        docstring (meaning of the four tables) and build_contract (flatten,
 *        stable sort by expert, histogram, offsets, ceil((c+1)/padding_M)
 *        padded offsets, m_blocks, block -> expert map), and its three checks.
 *   [P3] "MetaX-TileLang工具链" — §1.9 (the two launches and their arguments),
 *        §1.12.1 and §2.4 (gate = SiLU(x W_gate), up = x W_up, mid = gate*up,
 *        out = mid W_down; the router: logits = W_g(x), softmax, top-k).
 *
 * Readings where the pages are silent:
 *   - fp32 -> fp16 conversion is IEEE-754 round-to-nearest-even, overflow to inf.
 *   - group_offsets and group_padded_offsets hold E+1 entries; entry E is the
 *     total number of pairs / padded rows.
 *   - within one expert, pairs keep their flat (token-major) order: the sort in
 *     [P2] build_contract is Python's stable sort.
 *   - SiLU is g / (1 + e^-g) in fp32; the page's exp2 form with log2(e) is the
 *     same function.
 *
 * Parity pins: every function here is pinned by a -m "not gpu" test (fp16
 * conversion against numpy over all bit patterns, tables against [P2]'s
 * invariants and hand-derived examples, the forward against closed forms and a
 * tables-free brute force, the router against one-hot weights whose logits
 * are the token's own values and a float64 brute force).  No function is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16, from the format's definition                            */
/* ------------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN;
 * otherwise value = (1024 + fraction) * 2^(exponent - 25). */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Round to nearest integer, ties to even.  q >= 0 and q < 2^52, so floor()
 * and the subtraction are exact. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double rem = q - fl;
    if (rem > 0.5) return fl + 1.0;
    if (rem < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Nearest binary16 to v (round half to even).  Every float is a double, so
 * this also serves fp32 values without a double rounding. */
uint16_t oracle_half_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    /* 65504 is the largest finite half; the next step would be 65536, so the
     * rounding boundary is their midpoint 65520 (a tie there rounds to the even
     * significand, i.e. up to 65536 = overflow). */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; a carry to 1024 lands exactly on
         * the smallest normal's encoding (exponent 1, fraction 0). */
        double q = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int ex;
    double m = frexp(a, &ex);          /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                    /* a = s * 2^e, s in [1, 2)   */
    double q = round_half_even(ldexp(m, 11)); /* s * 2^10 rounded, in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* Bulk helpers used by the pins and the Python wrapper. */
void oracle_halves_to_doubles(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}

void oracle_doubles_to_halves(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_from_double(v[i]);
}

static float h2f(uint16_t h) { return (float)oracle_half_to_double(h); }

/* ------------------------------------------------------------------------- */
/* Dispatch tables — [P2] build_contract, step by step                        */
/* ------------------------------------------------------------------------- */

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* m_blocks = ceil(pairs / block_token) + n_experts   ([P2] build_contract
 * step 4; restated in [P3] §1.9 as M = ceil(group_sum/block_token) + group_count). */
int64_t oracle_num_blocks(int64_t pairs, int32_t n_experts, int32_t block_token)
{
    return ceil_div64(pairs, block_token) + n_experts;
}

/* Tables from topk_ids [n_tokens, top_k] (row-major; flat pair index t*k + j).
 *   group_sizes[e]           histogram of the flattened expert ids
 *   group_offsets[e]         exclusive prefix sum of group_sizes; [E] = pairs
 *   group_padded_offsets[e]  exclusive prefix sum of ceil((c+1)/padding_m)*padding_m;
 *                            [E] = total padded rows
 *   group_idx_for_bx[bx]     the last e whose padded start is <= bx*block_token,
 *                            found by the page's linear scan over all experts
 * Returns 0, or -1 if an expert id is out of range / a size is inconsistent. */
int oracle_build_dispatch(const int32_t* topk_ids, int64_t n_tokens, int32_t top_k,
                          int32_t n_experts, int32_t padding_m, int32_t block_token,
                          int32_t* group_sizes, int32_t* group_offsets,
                          int32_t* group_padded_offsets, int32_t* group_idx_for_bx,
                          int64_t num_blocks_m)
{
    int64_t pairs = n_tokens * (int64_t)top_k;
    if (num_blocks_m != oracle_num_blocks(pairs, n_experts, block_token)) return -1;

    /* 1) flatten token-major; 2) count per expert */
    for (int32_t e = 0; e < n_experts; ++e) group_sizes[e] = 0;
    for (int64_t f = 0; f < pairs; ++f) {
        int32_t e = topk_ids[f];
        if (e < 0 || e >= n_experts) return -1;
        group_sizes[e] += 1;
    }
    /* compact offsets */
    int64_t acc = 0;
    for (int32_t e = 0; e < n_experts; ++e) {
        group_offsets[e] = (int32_t)acc;
        acc += group_sizes[e];
    }
    group_offsets[n_experts] = (int32_t)acc;
    /* 3) padded offsets with the "+1" rule */
    group_padded_offsets[0] = 0;
    for (int32_t e = 1; e <= n_experts; ++e) {
        int64_t prev = ceil_div64((int64_t)group_sizes[e - 1] + 1, padding_m) * padding_m;
        group_padded_offsets[e] = (int32_t)(group_padded_offsets[e - 1] + prev);
    }
    /* 4) block -> expert, linear scan as on the page */
    for (int64_t bx = 0; bx < num_blocks_m; ++bx) {
        int64_t start = bx * (int64_t)block_token;
        int32_t g = 0;
        for (int32_t e = 0; e < n_experts; ++e)
            if (start >= group_padded_offsets[e]) g = e;
        group_idx_for_bx[bx] = g;
    }
    return 0;
}

/* Padded row of every pair under the stable sort by expert ([P2] build_contract
 * step 2: sorted(range(pairs), key=expert) keeps equal keys in flat order).
 * The pair of rank r within expert e sits at padded row padded[e] + r and at
 * compact index offsets[e] + r.  Written as the page's sort would place them:
 * walk the experts in order and, for each, the pairs in flat order. */
int oracle_pair_padded_rows(const int32_t* topk_ids, int64_t pairs, int32_t n_experts,
                            const int32_t* group_padded_offsets, int32_t* pair_rows)
{
    for (int32_t e = 0; e < n_experts; ++e) {
        int64_t rank = 0;
        for (int64_t f = 0; f < pairs; ++f) {
            if (topk_ids[f] == e) {
                pair_rows[f] = (int32_t)(group_padded_offsets[e] + rank);
                rank += 1;
            }
        }
    }
    for (int64_t f = 0; f < pairs; ++f)
        if (topk_ids[f] < 0 || topk_ids[f] >= n_experts) return -1;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Fused forward — [P1] §算子来源 and §完整算子代码, [P3] §2.4                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* x;        /* [rows_total, H] fp16, padded rows       */
    const uint16_t* gate_w;   /* [E, I, H] fp16                          */
    const uint16_t* up_w;     /* [E, I, H] fp16                          */
    const uint16_t* down_w;   /* [E, H, I] fp16                          */
    const float* rw;          /* [valid] fp32, compact (sorted) order     */
    const int32_t* sizes;
    const int32_t* offsets;
    const int32_t* padded;
    const int32_t* gidx;
    int64_t rows_total;
    int64_t num_blocks_m;
    int32_t H, I, E, block_token;
    int32_t acc_f64;          /* 0: fp32 accumulation (the pages'); 1: fp64 (error bound) */
} fwd_args;

/* Which expert / compact index a padded row belongs to, by the page's per-block
 * arithmetic: e = group_idx_for_bx[bx], token_offset = bx*block_token -
 * padded[e], actual_rows = max(0, min(block_token, sizes[e] - token_offset)).
 * Returns 1 for a valid row (i < actual_rows), 0 for a padding row. */
static int row_route(const fwd_args* a, int64_t row, int32_t* e_out, int64_t* compact_out)
{
    int64_t bx = row / a->block_token;
    int64_t i = row % a->block_token;
    if (bx < 0 || bx >= a->num_blocks_m) return 0;
    int32_t e = a->gidx[bx];
    int64_t block_start = bx * a->block_token;
    int64_t token_offset = block_start - a->padded[e];
    int64_t actual = (int64_t)a->sizes[e] - token_offset;
    if (actual > a->block_token) actual = a->block_token;
    if (actual < 0) actual = 0;
    if (i >= actual) return 0;
    *e_out = e;
    *compact_out = (int64_t)a->offsets[e] + token_offset + i;
    return 1;
}

/* One valid row, fp32 accumulation in natural k order.  Products of two fp16
 * values are exact in fp32 (11 x 11 significand bits). */
static void forward_row_f32(const fwd_args* a, int64_t row, int32_t e, int64_t compact,
                            uint16_t* up_row, uint16_t* out_row)
{
    const int32_t H = a->H, I = a->I;
    const uint16_t* xr = a->x + row * (int64_t)H;
    const uint16_t* gw = a->gate_w + (int64_t)e * I * H;
    const uint16_t* uw = a->up_w + (int64_t)e * I * H;
    const uint16_t* dw = a->down_w + (int64_t)e * H * I;
    /* phase 1: gate and up logits, SiLU(gate) * up in fp32, one rounding */
    for (int32_t j = 0; j < I; ++j) {
        float g = 0.0f, u = 0.0f;
        for (int32_t h = 0; h < H; ++h) {
            float xv = h2f(xr[h]);
            g += xv * h2f(gw[(int64_t)j * H + h]);
            u += xv * h2f(uw[(int64_t)j * H + h]);
        }
        float s = g / (1.0f + expf(-g));
        up_row[j] = oracle_half_from_double((double)(s * u));
    }
    /* phase 2: down projection of the fp16 workspace row, then the routed
     * weight on the fp32 accumulator, one rounding */
    float w = a->rw[compact];
    for (int32_t c = 0; c < H; ++c) {
        float acc = 0.0f;
        for (int32_t j = 0; j < I; ++j)
            acc += h2f(up_row[j]) * h2f(dw[(int64_t)c * I + j]);
        out_row[c] = oracle_half_from_double((double)(acc * w));
    }
}

/* The same row with every step in fp64 (rounding to fp16 at the same two
 * places).  Used only to bound the fp32 oracle's own rounding error. */
static void forward_row_f64(const fwd_args* a, int64_t row, int32_t e, int64_t compact,
                            uint16_t* up_row, uint16_t* out_row)
{
    const int32_t H = a->H, I = a->I;
    const uint16_t* xr = a->x + row * (int64_t)H;
    const uint16_t* gw = a->gate_w + (int64_t)e * I * H;
    const uint16_t* uw = a->up_w + (int64_t)e * I * H;
    const uint16_t* dw = a->down_w + (int64_t)e * H * I;
    for (int32_t j = 0; j < I; ++j) {
        double g = 0.0, u = 0.0;
        for (int32_t h = 0; h < H; ++h) {
            double xv = oracle_half_to_double(xr[h]);
            g += xv * oracle_half_to_double(gw[(int64_t)j * H + h]);
            u += xv * oracle_half_to_double(uw[(int64_t)j * H + h]);
        }
        double s = g / (1.0 + exp(-g));
        up_row[j] = oracle_half_from_double(s * u);
    }
    double w = (double)a->rw[compact];
    for (int32_t c = 0; c < H; ++c) {
        double acc = 0.0;
        for (int32_t j = 0; j < I; ++j)
            acc += oracle_half_to_double(up_row[j]) * oracle_half_to_double(dw[(int64_t)c * I + j]);
        out_row[c] = oracle_half_from_double(acc * w);
    }
}

static int check_args(const fwd_args* a)
{
    if (!a->x || !a->gate_w || !a->up_w || !a->down_w || !a->rw || !a->sizes ||
        !a->offsets || !a->padded || !a->gidx) return -1;
    if (a->H <= 0 || a->I <= 0 || a->E <= 0 || a->block_token <= 0) return -1;
    for (int64_t bx = 0; bx < a->num_blocks_m; ++bx)
        if (a->gidx[bx] < 0 || a->gidx[bx] >= a->E) return -1;
    return 0;
}

/* Full forward over every block of the padded array: the valid rows of
 * up_logits [rows_total, I] and out [rows_total, H] are written; padding rows
 * are left exactly as the caller filled them.  n_threads <= 0 uses the default
 * OpenMP thread count.  Returns 0 or -1. */
int oracle_fused_forward(const uint16_t* x, int64_t rows_total, int32_t H,
                         const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
                         int32_t E, int32_t I, const float* rw,
                         const int32_t* sizes, const int32_t* offsets, const int32_t* padded,
                         const int32_t* gidx, int64_t num_blocks_m, int32_t block_token,
                         uint16_t* up_logits, uint16_t* out, int32_t acc_f64, int32_t n_threads)
{
    fwd_args a = {x, gate_w, up_w, down_w, rw, sizes, offsets, padded, gidx,
                  rows_total, num_blocks_m, H, I, E, block_token, acc_f64};
    if (check_args(&a)) return -1;
    int64_t rows = num_blocks_m * (int64_t)block_token;
    if (rows > rows_total) rows = rows_total;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int64_t r;
#pragma omp parallel for schedule(dynamic, 4)
    for (r = 0; r < rows; ++r) {
        int32_t e;
        int64_t compact;
        if (!row_route(&a, r, &e, &compact)) continue;
        if (acc_f64)
            forward_row_f64(&a, r, e, compact, up_logits + r * (int64_t)I, out + r * (int64_t)H);
        else
            forward_row_f32(&a, r, e, compact, up_logits + r * (int64_t)I, out + r * (int64_t)H);
    }
    return 0;
}

/* The same computation for a chosen list of padded rows (for sampled checks of
 * full-size runs).  Row n of the results goes to up_rows[n, :] and
 * out_rows[n, :]; valid[n] is 1 for a valid row, 0 for a padding row (whose
 * result rows are left untouched). */
int oracle_forward_rows(const uint16_t* x, int64_t rows_total, int32_t H,
                        const uint16_t* gate_w, const uint16_t* up_w, const uint16_t* down_w,
                        int32_t E, int32_t I, const float* rw,
                        const int32_t* sizes, const int32_t* offsets, const int32_t* padded,
                        const int32_t* gidx, int64_t num_blocks_m, int32_t block_token,
                        const int64_t* row_list, int64_t n_rows,
                        uint16_t* up_rows, uint16_t* out_rows, int32_t* valid,
                        int32_t acc_f64, int32_t n_threads)
{
    fwd_args a = {x, gate_w, up_w, down_w, rw, sizes, offsets, padded, gidx,
                  rows_total, num_blocks_m, H, I, E, block_token, acc_f64};
    if (check_args(&a)) return -1;
    for (int64_t n = 0; n < n_rows; ++n)
        if (row_list[n] < 0 || row_list[n] >= rows_total) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int64_t n;
#pragma omp parallel for schedule(dynamic, 1)
    for (n = 0; n < n_rows; ++n) {
        int32_t e;
        int64_t compact;
        valid[n] = row_route(&a, row_list[n], &e, &compact);
        if (!valid[n]) continue;
        if (acc_f64)
            forward_row_f64(&a, row_list[n], e, compact, up_rows + n * (int64_t)I, out_rows + n * (int64_t)H);
        else
            forward_row_f32(&a, row_list[n], e, compact, up_rows + n * (int64_t)I, out_rows + n * (int64_t)H);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Steps on either side of the path (test harness): pack and combine          */
/* ------------------------------------------------------------------------- */

/* Gather token rows into the grouped, padded layout and put the routed weights
 * in compact order ([P1] §实现要点: x / up_logits / out use padded rows, the
 * routed weights use compact rows offsets[e] + token_offset).  Padding rows of
 * x_packed are not touched (the caller fills them).  pair_rows from
 * oracle_pair_padded_rows. */
int oracle_pack(const uint16_t* x_tokens, int64_t n_tokens, int32_t top_k, int32_t H,
                const int32_t* topk_ids, const float* topk_weights,
                const int32_t* pair_rows, const int32_t* offsets, const int32_t* padded,
                uint16_t* x_packed, int64_t rows_total, float* rw_compact)
{
    int64_t pairs = n_tokens * (int64_t)top_k;
    for (int64_t f = 0; f < pairs; ++f) {
        int64_t row = pair_rows[f];
        int32_t e = topk_ids[f];
        if (row < 0 || row >= rows_total) return -1;
        memcpy(x_packed + row * (int64_t)H, x_tokens + (f / top_k) * (int64_t)H,
               (size_t)H * sizeof(uint16_t));
        rw_compact[offsets[e] + (row - padded[e])] = topk_weights[f];
    }
    return 0;
}

/* Sum each token's k expert outputs back into token order: y[t, c] =
 * fp16( sum_j out[row(t, j), c] ), summed in fp32 in j order.  The pages do
 * this with a PyTorch scatter_reduce ([P3] §2.7); the fp32 sum with one
 * rounding is this library's reading of it. */
int oracle_combine(const uint16_t* out, int64_t rows_total, int32_t H,
                   const int32_t* pair_rows, int64_t n_tokens, int32_t top_k, uint16_t* y)
{
    for (int64_t t = 0; t < n_tokens; ++t) {
        for (int32_t c = 0; c < H; ++c) {
            float s = 0.0f;
            for (int32_t j = 0; j < top_k; ++j) {
                int64_t row = pair_rows[t * top_k + j];
                if (row < 0 || row >= rows_total) return -1;
                s += h2f(out[row * (int64_t)H + c]);
            }
            y[t * (int64_t)H + c] = oracle_half_from_double((double)s);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Router — "MetaX-TileLang工具链" §2.4: logits = W_g(x), scores =            */
/* softmax(logits), (topk_scores, topk_indices) = topk(scores)                */
/* ------------------------------------------------------------------------- */

/* For every token t: logits[e] = sum_h x[t,h] * wg[e,h] in fp32 (natural h
 * order); softmax over all E experts in fp32 (max subtracted, expf, sum in e
 * order); the k largest logits (equal logits: the lower expert index first),
 * in descending order; their probabilities are the routed weights.  The
 * top-k is decided on the logits, which orders the experts exactly as the
 * probabilities do.  Returns 0, or -1 for bad arguments. */
int oracle_router(const uint16_t* x, int64_t n_tokens, int32_t H, const uint16_t* wg, int32_t E,
                  int32_t top_k, int32_t* topk_ids, float* topk_weights, int32_t n_threads)
{
    if (!x || !wg || !topk_ids || !topk_weights || H <= 0 || E <= 0 || top_k <= 0 || top_k > E)
        return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int64_t t;
#pragma omp parallel for schedule(dynamic, 16)
    for (t = 0; t < n_tokens; ++t) {
        float* logit = (float*)malloc(sizeof(float) * (size_t)E);
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        const uint16_t* xr = x + t * (int64_t)H;
        for (int32_t e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int32_t h = 0; h < H; ++h)
                acc += h2f(xr[h]) * h2f(wg[(int64_t)e * H + h]);
            logit[e] = acc;
        }
        float mx = logit[0];
        for (int32_t e = 1; e < E; ++e)
            if (logit[e] > mx) mx = logit[e];
        float sum = 0.0f;
        for (int32_t e = 0; e < E; ++e) sum += expf(logit[e] - mx);
        for (int32_t j = 0; j < top_k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || logit[e] > logit[best])) best = e;
            taken[best] = 1;
            topk_ids[t * top_k + j] = best;
            topk_weights[t * top_k + j] = expf(logit[best] - mx) / sum;
        }
        free(logit);
        free(taken);
    }
    return 0;
}
