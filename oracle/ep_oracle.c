/*
 * ep_oracle.c — plain, slow, obviously-correct CPU oracle for the MoE
 * expert-parallel routing plan, the dispatch row scatter (BF16 and FP8 E4M3)
 * and the weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library; it is compiled with plain gcc.
 *
 * Every function follows the definition as the source pages state it, in
 * nested loops and in the pages' order, with no blocking, fusion or prefix
 * tricks.  Sources (page title, then section):
 *   [DO]  "Ascend DeepEP MoE Dispatch Optimization" (blog post)
 *         - "从 Python 接口进入真实调用链": the six-tensor dispatch handle table
 *         - "Host 侧先造一张通信地图" / "Notify 先交换数量和前缀": counts -> prefix
 *         - "Device 侧如何把 channel 变成远端 Put": per-channel cursor bases
 *         - "P 维路由为什么值得单独优化": the [S,P] routing matrix
 *   [TT]  TileLang tutorial, chapter 38 "DeepEP-Ascend"
 *         - §1.2 byte ledger, §1.3 per-destination dedup
 *         - §2.2 expanded layout and expert padding
 *         - §2.3 combine is the inverse of dispatch
 *         - §3.5 deterministic layout (stable sort by expert, then source token)
 *         - §3.6 FP8 dispatch scales (one fp32 scale per 128 hidden elements)
 *         - §4.5 combine reduction: widen to fp32, accumulate, round once to bf16
 *
 * Readings where the pages are silent or garbled (each listed in the design
 * notes of the repository):
 *   - expert -> rank map: contiguous blocks, rank = e / (E/P)
 *   - topk_idx == -1 marks an unused slot: no row, slot = -1, no contribution
 *   - duplicate expert ids inside one token row are invalid
 *   - rank_prefix_matrix and channel_prefix_matrix are INCLUSIVE cumulative sums
 *   - recv_channel_prefix_matrix[d][s][c] is the start offset of segment (s,c)
 *     inside destination d's compact window
 *   - send_head[g][d] is the row index inside d's compact window, else -1
 *   - compact windows and expert segments are ordered by increasing global token
 *   - channel c of a source rank covers tokens [c*ceil(S/C), min(S,(c+1)*ceil(S/C)))
 *   - FP8: scale = amax/448 (fp32 IEEE division), q = E4M3_RNE_satfinite(x/scale);
 *     amax == 0 gives scale = 0 and all-zero codes
 *   - FP8 on non-finite x: NaN elements are left out of amax, an infinite
 *     element makes the scale +inf, and every NaN quotient encodes as 0x7f
 *   - combine: acc = 0.0f, then for k = 0..K-1 with slot >= 0:
 *     acc = fmaf(w[g,k], float(y[slot]), acc); out = bf16_RNE(acc)
 *
 * Compile: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 * The same source built with -fopenmp is the multi-core variant: the
 * "omp parallel for" lines below split the per-row loops of the scatter, the
 * combine and the synthetic experts over threads.  Every output element is
 * still computed by the same sequential code in the same order; only which
 * thread computes which rows changes, so both builds give identical bits.
 * Without -fopenmp the pragmas are ignored.  The plan stays sequential.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID 1
#define ORACLE_ERR_CAPACITY 2

/* Threads the row loops use: 1 for the plain build. */
int ep_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
float ep_oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round binary32 to bf16, round-to-nearest-even on the 16 dropped bits.
 * A NaN stays a (quiet) NaN. */
uint16_t ep_oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t dropped = u & 0xffffu;
    uint32_t kept = u >> 16;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u; /* carry may move into the exponent: that is correct rounding */
    return (uint16_t)kept;
}

/* OCP 8-bit floating point, E4M3 ("fn") variant: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest
 * finite magnitude 1.75 * 2^8 = 448, smallest normal 2^-6, subnormal spacing
 * 2^-9.  Decoding follows that definition field by field. */
float ep_oracle_e4m3_to_f32(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int exp_field = (b >> 3) & 0xf;
    int mant = b & 7;
    double v;
    if (exp_field == 0xf && mant == 7)
        return sign ? -NAN : NAN;
    if (exp_field == 0)
        v = ldexp((double)mant, -9); /* subnormal: mant/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + mant / 8.0, exp_field - 7);
    return (float)(sign ? -v : v);
}

/* Encode a binary32 value as E4M3 with round-to-nearest-even and saturation
 * of finite overflow to +-448.  Written from the format definition: find the
 * spacing of representable values in the binade of |v|, round |v|/spacing to
 * the nearest integer (ties to even), then lay the result out in fields.
 * Every NaN encodes as 0x7f (S.1111.111 with the sign bit clear): IEEE
 * arithmetic leaves the sign of a NaN result unspecified (x86 and Arm hosts
 * differ on inf/inf), so the reading fixes it, and the result does not
 * depend on the CPU that computes the quotient. */
uint8_t ep_oracle_f32_to_e4m3(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)0x7f;
    if (isinf(v))
        return (uint8_t)(sign | 0x7e); /* satfinite: +-448 */
    double a = fabs((double)v);
    double min_normal = ldexp(1.0, -6);
    double spacing;
    if (a < min_normal) {
        spacing = ldexp(1.0, -9);
    } else {
        int e2;
        frexp(a, &e2); /* a = m * 2^e2 with m in [0.5, 1): binade starts at 2^(e2-1) */
        spacing = ldexp(1.0, (e2 - 1) - 3);
    }
    double n = a / spacing; /* exact: spacing is a power of two */
    double r = nearbyint(n); /* default rounding mode: nearest, ties to even */
    double val = r * spacing;
    if (val > 448.0)
        val = 448.0; /* satfinite */
    if (val == 0.0)
        return sign;
    if (val < min_normal)
        return (uint8_t)(sign | (int)(val / ldexp(1.0, -9)));
    int e2;
    double m = frexp(val, &e2); /* val = m * 2^e2, m in [0.5, 1) */
    int exp_field = (e2 - 1) + 7;
    int mant = (int)((2.0 * m - 1.0) * 8.0); /* exact: three fraction bits */
    return (uint8_t)(sign | (exp_field << 3) | mant);
}

/* ------------------------------------------------------------------------ */
/* Routing plan                                                              */
/* ------------------------------------------------------------------------ */

/* Validation of the routing inputs, mirroring the required-argument checks of
 * the dispatch entry ([DO] "从 Python 接口进入真实调用链") and the readings above. */
int ep_oracle_validate(const int64_t *topk_idx, int64_t S, int P, int K, int E,
                       int A, int C)
{
    if (P < 1 || E < 1 || K < 1 || S < 0 || A < 1 || C < 1)
        return ORACLE_ERR_INVALID;
    if (E % P != 0 || K > E || (S > 0 && C > S))
        return ORACLE_ERR_INVALID;
    int64_t T = (int64_t)P * S;
    for (int64_t g = 0; g < T; ++g) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[g * K + k];
            if (e < -1 || e >= E)
                return ORACLE_ERR_INVALID;
            if (e < 0)
                continue;
            for (int k2 = 0; k2 < k; ++k2)
                if (topk_idx[g * K + k2] == e)
                    return ORACLE_ERR_INVALID;
        }
    }
    return ORACLE_OK;
}

/* Worst-case sizes a caller must provide for the variable-length outputs. */
int64_t ep_oracle_max_recv_rows(int64_t S, int P, int K)
{
    return (int64_t)P * S * (K < P ? K : P);
}

int64_t ep_oracle_max_expanded_rows(int64_t S, int P, int K, int E, int A)
{
    return (int64_t)P * S * K + (int64_t)E * (A - 1);
}

/*
 * The routing plan, by direct definition.
 *
 * Inputs:  topk_idx [T,K] int64 with T = P*S; global token g = s*S + t.
 * Outputs (caller-allocated, sizes in brackets):
 *   is_token_in_rank      [T,P]   u8   1 if some expert of g lives on rank d
 *   num_tokens_per_rank   [P,P]   i32  [s][d]: tokens of source s that go to d
 *   num_tokens_per_expert [P,E]   i32  [s][e]: (token,slot) pairs of s that pick e
 *   expert_counts         [E]     i32  n_e = sum over s
 *   num_recv              [P]     i32  distinct tokens received by d
 *   rank_prefix           [P,P]   i32  [s][d] inclusive sum over sources <= s
 *   channel_prefix        [P,P,C] i32  [s][d][c] inclusive sum over channels <= c
 *   recv_channel_prefix   [P,P,C] i32  [d][s][c] start of segment (s,c) in d's window
 *   send_head             [T,P]   i32  row of g inside d's window, else -1
 *   recv_offsets          [P+1]   i32  start of d's window in the flat recv_src_idx
 *   recv_src_idx          [N_recv]i32  source-local token index t of each window row
 *   expert_offsets        [E+1]   i32  padded start of expert e's segment
 *   slot                  [T,K]   i32  expanded row of (g,k), -1 for an unused slot
 *   exp_src               [N_exp] i32  global source token of each expanded row,
 *                                      -1 on padding rows
 *   sizes                 [2]     i64  {N_recv, N_exp}
 * Returns ORACLE_OK, ORACLE_ERR_INVALID, or ORACLE_ERR_CAPACITY when a
 * variable-length output does not fit the given capacity.
 */
int ep_oracle_plan(const int64_t *topk_idx, int64_t S, int P, int K, int E, int A,
                   int C, uint8_t *is_token_in_rank, int32_t *num_tokens_per_rank,
                   int32_t *num_tokens_per_expert, int32_t *expert_counts,
                   int32_t *num_recv, int32_t *rank_prefix, int32_t *channel_prefix,
                   int32_t *recv_channel_prefix, int32_t *send_head,
                   int32_t *recv_offsets, int32_t *recv_src_idx, int64_t recv_src_cap,
                   int32_t *expert_offsets, int32_t *slot, int32_t *exp_src,
                   int64_t exp_src_cap, int64_t *sizes)
{
    int rc = ep_oracle_validate(topk_idx, S, P, K, E, A, C);
    if (rc != ORACLE_OK)
        return rc;
    const int64_t T = (int64_t)P * S;
    const int E_l = E / P;                /* local experts per rank */
    const int64_t chunk = S > 0 ? (S + C - 1) / C : 0; /* tokens per channel */

    /* Step 1. Destination set of each token, deduplicated: rank d is in
     * dests(g) when some valid idx[g,k] has idx/E_l == d ([TT] §1.3 item 1). */
    for (int64_t g = 0; g < T; ++g)
        for (int d = 0; d < P; ++d) {
            uint8_t hit = 0;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[g * K + k];
                if (e >= 0 && e / E_l == d)
                    hit = 1;
            }
            is_token_in_rank[g * P + d] = hit;
        }

    /* Step 2. Counts by direct summation. */
    for (int s = 0; s < P; ++s) {
        for (int d = 0; d < P; ++d) {
            int32_t n = 0;
            for (int64_t t = 0; t < S; ++t)
                n += is_token_in_rank[((int64_t)s * S + t) * P + d];
            num_tokens_per_rank[s * P + d] = n;
        }
        for (int e = 0; e < E; ++e) {
            int32_t n = 0;
            for (int64_t t = 0; t < S; ++t)
                for (int k = 0; k < K; ++k)
                    n += topk_idx[((int64_t)s * S + t) * K + k] == e;
            num_tokens_per_expert[(int64_t)s * E + e] = n;
        }
    }
    for (int e = 0; e < E; ++e) {
        int32_t n = 0;
        for (int s = 0; s < P; ++s)
            n += num_tokens_per_expert[(int64_t)s * E + e];
        expert_counts[e] = n;
    }
    for (int d = 0; d < P; ++d) {
        int32_t n = 0;
        for (int s = 0; s < P; ++s)
            n += num_tokens_per_rank[s * P + d];
        num_recv[d] = n;
    }

    /* Step 3. Prefix matrices ([DO] handle table; the cursor bases of the
     * per-channel payload loop in "Device 侧如何把 channel 变成远端 Put"). */
    for (int s = 0; s < P; ++s)
        for (int d = 0; d < P; ++d) {
            int32_t acc = 0;
            for (int s2 = 0; s2 <= s; ++s2)
                acc += num_tokens_per_rank[s2 * P + d];
            rank_prefix[s * P + d] = acc;
        }
    for (int s = 0; s < P; ++s)
        for (int d = 0; d < P; ++d) {
            int32_t acc = 0;
            for (int c = 0; c < C; ++c) {
                int64_t lo = (int64_t)c * chunk, hi = (int64_t)(c + 1) * chunk;
                if (lo > S) lo = S;
                if (hi > S) hi = S;
                for (int64_t t = lo; t < hi; ++t)
                    acc += is_token_in_rank[((int64_t)s * S + t) * P + d];
                channel_prefix[((int64_t)s * P + d) * C + c] = acc;
            }
        }
    for (int d = 0; d < P; ++d)
        for (int s = 0; s < P; ++s)
            for (int c = 0; c < C; ++c) {
                int32_t base = s > 0 ? rank_prefix[(s - 1) * P + d] : 0;
                int32_t in_src = c > 0 ? channel_prefix[((int64_t)s * P + d) * C + c - 1] : 0;
                recv_channel_prefix[((int64_t)d * P + s) * C + c] = base + in_src;
            }

    /* Step 4. Compact receive windows: walk tokens in increasing g and append
     * each token that goes to d. */
    recv_offsets[0] = 0;
    for (int d = 0; d < P; ++d)
        recv_offsets[d + 1] = recv_offsets[d] + num_recv[d];
    if (recv_offsets[P] > recv_src_cap)
        return ORACLE_ERR_CAPACITY;
    for (int d = 0; d < P; ++d) {
        int32_t pos = 0;
        for (int64_t g = 0; g < T; ++g) {
            if (is_token_in_rank[g * P + d]) {
                send_head[g * P + d] = pos;
                recv_src_idx[recv_offsets[d] + pos] = (int32_t)(g % S);
                ++pos;
            } else {
                send_head[g * P + d] = -1;
            }
        }
    }

    /* Step 5. Expanded layout: expert segments in expert order, each padded
     * to ceil(n_e/A)*A rows ([TT] §2.2), rows inside a segment in increasing
     * source token ([TT] §3.5). */
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t padded = ((int64_t)expert_counts[e] + A - 1) / A * A;
        expert_offsets[e + 1] = (int32_t)(expert_offsets[e] + padded);
    }
    if (expert_offsets[E] > exp_src_cap)
        return ORACLE_ERR_CAPACITY;
    for (int64_t i = 0; i < T * K; ++i)
        slot[i] = -1;
    for (int e = 0; e < E; ++e) {
        int32_t row = expert_offsets[e];
        for (int64_t g = 0; g < T; ++g)
            for (int k = 0; k < K; ++k)
                if (topk_idx[g * K + k] == e) {
                    slot[g * K + k] = row;
                    exp_src[row] = (int32_t)g;
                    ++row;
                }
        for (; row < expert_offsets[e + 1]; ++row)
            exp_src[row] = -1;
    }
    sizes[0] = recv_offsets[P];
    sizes[1] = expert_offsets[E];
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch                                                                  */
/* ------------------------------------------------------------------------ */

/* BF16 dispatch: expanded row r holds a bit copy of x[exp_src[r]]; padding
 * rows are zero when zero_pad is set and left untouched otherwise
 * ([TT] §2.2 item 2). */
void ep_oracle_dispatch_bf16(const uint16_t *x, int64_t H, const int32_t *exp_src,
                             int64_t n_rows, int zero_pad, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int32_t g = exp_src[r];
        for (int64_t h = 0; h < H; ++h) {
            if (g >= 0)
                out[r * H + h] = x[(int64_t)g * H + h];
            else if (zero_pad)
                out[r * H + h] = 0;
        }
    }
}

/* FP8 dispatch: for each expanded row and each group of 128 hidden elements,
 * amax = max |x| (exact in fp32), scale = amax / 448 (IEEE fp32 division),
 * q = E4M3(x / scale) with RNE and saturation; scales are row-major
 * [rows, H/128] fp32 ([TT] §3.6).  amax == 0 gives scale 0 and zero codes.
 * Non-finite x (the pages define none): NaN elements do not take part in
 * amax (the comparison below is false for them); an infinite element makes
 * amax and the scale +inf, so finite elements of its group give signed zero
 * codes and the infinite one inf/inf = NaN; every NaN quotient is code 0x7f. */
void ep_oracle_dispatch_fp8(const uint16_t *x, int64_t H, const int32_t *exp_src,
                            int64_t n_rows, int zero_pad, uint8_t *out_q,
                            float *out_scales)
{
    const int64_t G = H / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int32_t g = exp_src[r];
        if (g < 0) {
            if (zero_pad) {
                for (int64_t h = 0; h < H; ++h)
                    out_q[r * H + h] = 0;
                for (int64_t j = 0; j < G; ++j)
                    out_scales[r * G + j] = 0.0f;
            }
            continue;
        }
        for (int64_t j = 0; j < G; ++j) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float v = fabsf(ep_oracle_bf16_to_f32(x[(int64_t)g * H + j * 128 + i]));
                if (v > amax)
                    amax = v;
            }
            float scale = amax / 448.0f;
            out_scales[r * G + j] = scale;
            for (int64_t i = 0; i < 128; ++i) {
                uint8_t q = 0;
                if (amax != 0.0f) {
                    float v = ep_oracle_bf16_to_f32(x[(int64_t)g * H + j * 128 + i]);
                    q = ep_oracle_f32_to_e4m3(v / scale);
                }
                out_q[r * H + j * 128 + i] = q;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Combine                                                                   */
/* ------------------------------------------------------------------------ */

/* Weighted k-way reduction back to token order ([TT] §4.5): widen each bf16
 * expert output to fp32, accumulate in fixed slot order k = 0..K-1 with a
 * fused multiply-add, then add the optional bias row ([TT] §3.3, the fused
 * residual / shared-expert output) in fp32, round once to bf16.  A token
 * without a valid slot gives its bias (zeros without bias). */
void ep_oracle_combine_bias(const uint16_t *y, int64_t H, const int32_t *slot,
                            const float *topk_weights, const uint16_t *bias, int64_t T, int K,
                            uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < T; ++g)
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = slot[g * K + k];
                if (r < 0)
                    continue;
                acc = fmaf(topk_weights[g * K + k], ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]), acc);
            }
            if (bias)
                acc = acc + ep_oracle_bf16_to_f32(bias[g * H + h]);
            out[g * H + h] = ep_oracle_f32_to_bf16(acc);
        }
}

void ep_oracle_combine(const uint16_t *y, int64_t H, const int32_t *slot,
                       const float *topk_weights, int64_t T, int K, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < T; ++g)
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = slot[g * K + k];
                if (r < 0)
                    continue;
                acc = fmaf(topk_weights[g * K + k], ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]), acc);
            }
            out[g * H + h] = ep_oracle_f32_to_bf16(acc);
        }
}

/* ------------------------------------------------------------------------ */
/* Synthetic experts used between dispatch and combine in the parity tests   */
/* ------------------------------------------------------------------------ */

/* Per-expert scaling expert: y[r] = bf16_RNE(float(x[r]) * (1 + e/E)) for a
 * row r in expert e's segment; padding rows give zeros. */
void ep_oracle_expert_scale(const uint16_t *x_exp, int64_t H, const int32_t *exp_src,
                            const int32_t *expert_offsets, int E, uint16_t *y)
{
    for (int e = 0; e < E; ++e) {
        float f = 1.0f + (float)e / (float)E;
#pragma omp parallel for schedule(static)
        for (int64_t r = expert_offsets[e]; r < expert_offsets[e + 1]; ++r)
            for (int64_t h = 0; h < H; ++h)
                y[r * H + h] = exp_src[r] >= 0
                    ? ep_oracle_f32_to_bf16(ep_oracle_bf16_to_f32(x_exp[r * H + h]) * f)
                    : 0;
    }
}

/* Dequantising identity expert for FP8 rows: y = bf16_RNE(float(q) * scale). */
void ep_oracle_expert_dequant(const uint8_t *q, const float *scales, int64_t H,
                              int64_t n_rows, uint16_t *y)
{
    const int64_t G = H / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t h = 0; h < H; ++h)
            y[r * H + h] = ep_oracle_f32_to_bf16(ep_oracle_e4m3_to_f32(q[r * H + h]) * scales[r * G + h / 128]);
}

/* The same scaling expert on a list of rows whose experts are given
 * explicitly (row_expert[i] < 0 marks a padding row). */
void ep_oracle_expert_scale_rows(const uint16_t *x_rows, int64_t H, const int32_t *row_expert,
                                 int64_t n_rows, int E, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int e = row_expert[r];
        float f = e >= 0 ? 1.0f + (float)e / (float)E : 0.0f;
        for (int64_t h = 0; h < H; ++h)
            y[r * H + h] = e >= 0
                ? ep_oracle_f32_to_bf16(ep_oracle_bf16_to_f32(x_rows[r * H + h]) * f)
                : 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Backward on the same handle ([TT] §2.3: the backward of dispatch is a     */
/* combine, the backward of combine is a dispatch, both on the forward plan) */
/* ------------------------------------------------------------------------ */

/* Dispatch backward: recv[slot[g,k]] = x[g] for every valid k, so
 * grad_x[g] = sum over k = 0..K-1 with slot >= 0 of grad_recv[slot[g,k]],
 * accumulated in fp32 in slot order and rounded once to bf16 (the combine
 * with unit weights). */
void ep_oracle_dispatch_backward(const uint16_t *grad_recv, int64_t H, const int32_t *slot,
                                 int64_t T, int K, uint16_t *grad_x)
{
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < T; ++g)
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = slot[g * K + k];
                if (r >= 0)
                    acc = acc + ep_oracle_bf16_to_f32(grad_recv[(int64_t)r * H + h]);
            }
            grad_x[g * H + h] = ep_oracle_f32_to_bf16(acc);
        }
}

/* Combine backward: out[g] = sum_k w[g,k] * y[slot[g,k]], so
 *   grad_y[slot[g,k]] = bf16_RNE(w[g,k] * float(grad_out[g]))  (fp32 product),
 *   grad_w[g,k]       = sum_h grad_out[g,h] * y[slot[g,k],h]    (fp64 here),
 * with grad_w = 0 for an unused slot.  Padding rows of grad_y are zeroed
 * when zero_pad is set (they receive no gradient), left untouched otherwise. */
void ep_oracle_combine_backward(const uint16_t *grad_out, const uint16_t *y, int64_t H,
                                const int32_t *slot, const int32_t *exp_src, int64_t n_rows,
                                const float *topk_weights, int64_t T, int K, int zero_pad,
                                uint16_t *grad_y, double *grad_w)
{
    if (zero_pad)
        for (int64_t r = 0; r < n_rows; ++r)
            if (exp_src[r] < 0)
                for (int64_t h = 0; h < H; ++h)
                    grad_y[r * H + h] = 0;
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < T; ++g)
        for (int k = 0; k < K; ++k) {
            int32_t r = slot[g * K + k];
            double dot = 0.0;
            if (r >= 0) {
                float wk = topk_weights[g * K + k];
                for (int64_t h = 0; h < H; ++h) {
                    float go = ep_oracle_bf16_to_f32(grad_out[g * H + h]);
                    grad_y[(int64_t)r * H + h] = ep_oracle_f32_to_bf16(wk * go);
                    dot += (double)go * (double)ep_oracle_bf16_to_f32(y[(int64_t)r * H + h]);
                }
            }
            grad_w[g * K + k] = dot;
        }
}

/* ------------------------------------------------------------------------ */
/* Metadata-carrying dispatch and pre-quantised FP8 input                    */
/* ------------------------------------------------------------------------ */

/* Per expanded row, the metadata the pages carry next to the hidden bytes
 * ([TT] §2.1, §4.2: routing weight and source token): recv_weights[r] =
 * w[g,k] and recv_meta[r] = {g, k} for r = slot[g,k]; padding rows get
 * weight 0 and {-1, -1}. */
void ep_oracle_dispatch_metadata(const int32_t *slot, const float *topk_weights, int64_t T, int K,
                                 int64_t n_rows, float *recv_weights, int32_t *recv_meta)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        recv_weights[r] = 0.0f;
        recv_meta[2 * r] = -1;
        recv_meta[2 * r + 1] = -1;
    }
    for (int64_t g = 0; g < T; ++g)
        for (int k = 0; k < K; ++k) {
            int32_t r = slot[g * K + k];
            if (r < 0)
                continue;
            recv_weights[r] = topk_weights[g * K + k];
            recv_meta[2 * r] = (int32_t)g;
            recv_meta[2 * r + 1] = k;
        }
}

/* Dispatch of input that is already FP8 ([TT] §3.6: x arrives as (codes,
 * scales)): expanded row r holds the codes and the H/128 fp32 scales of
 * token exp_src[r]; padding rows are zero when zero_pad is set. */
void ep_oracle_dispatch_fp8_input(const uint8_t *xq, const float *xs, int64_t H, const int32_t *exp_src,
                                  int64_t n_rows, int zero_pad, uint8_t *out_q, float *out_scales)
{
    const int64_t G = H / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        int32_t g = exp_src[r];
        if (g < 0 && !zero_pad)
            continue;
        for (int64_t h = 0; h < H; ++h)
            out_q[r * H + h] = g >= 0 ? xq[(int64_t)g * H + h] : 0;
        for (int64_t j = 0; j < G; ++j)
            out_scales[r * G + j] = g >= 0 ? xs[(int64_t)g * G + j] : 0.0f;
    }
}
