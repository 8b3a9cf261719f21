/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for MoE token
 * layout -> dispatch -> combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library; it is written from the definitions alone, one obvious loop per
 * step, with no blocking, fusion or reordering.
 *
 * Sources (page title, then section or code fragment):
 *  [P1] "DeepEP Symmetric Memory" architecture analysis,
 *       section 6.1 (the dispatch launch: per-rank / per-expert prefix sums,
 *       destination slot index, expert alignment), section 7.3 (receive
 *       counts read back per rank and per local expert), section 9.2
 *       (dispatch returns recv_x, recv_topk_idx, recv_topk_weights; combine
 *       takes topk_weights and returns the combined rows).
 *  [P2] "DeepEP V2 ElasticBuffer architecture", the TokenLayout fragment
 *       (each received token carries its hidden row, scale factors, top-k
 *       indices, top-k weights and source token index) and the limits
 *       fragment (kNumMaxRanks, kNumMaxExperts, kNumMaxExpertsPerRank).
 *
 * Readings where the pages are silent (each repeated at its use):
 *  - T is the total token count; receive order inside a rank is ascending
 *    global token index (source rank s owns tokens [s*T/R, (s+1)*T/R)).
 *  - Expert e lives on rank e / (E/R) (contiguous blocks of local experts).
 *  - topk_idx is int64 with -1 = masked; received indices are int32 local
 *    expert ids, -1 where the expert is not on the receiving rank, with
 *    weight 0.0f.
 *  - FP8: per 128-channel block, amax = max|x|, sf = amax/448,
 *    q = e4m3_rne_satfinite(x * (448/amax)) in fp32; an all-zero block has
 *    sf = 1 and multiplier 0.
 *  - Combine: out[t] = sum over ranks r holding t of c(t,r) * y[dst_row[t,r]],
 *    c = 1 unweighted, else the sum of t's weights whose expert is on r.
 *    The oracle accumulates in fp64 and returns fp64 (the exact sum up to
 *    fp64 rounding); the parity test applies the fp32/bf16 tolerance.
 *
 * Parity pins for every function live in the CPU test suite (brute force,
 * closed forms, invariants, the OCP FP8 definition, a library cast).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (see build.py).
 * -ffp-contract=off keeps every multiply and add separately rounded on both
 * x86-64 and aarch64.  A second build with -fopenmp splits the token loops
 * of dispatch (non-compact form) and combine over host threads, for the
 * benchmark's all-cores CPU baseline; the arithmetic is the same code.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK            0
#define OR_INVALID_INDEX 4
#define OR_CAPACITY      8

/* Threads the dispatch and combine loops may use: 1, or OpenMP's count in  */
/* a build with -fopenmp (the benchmark's all-cores CPU baseline).          */
int ep_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> float.  A bf16 is the upper 16 bits of an IEEE binary32.        */
/* ------------------------------------------------------------------------ */

float ep_oracle_bf16_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even (finite inputs). */
uint16_t ep_oracle_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {           /* inf / nan */
        if (u & 0x007fffffu) return (uint16_t)((u >> 16) | 0x40u);
        return (uint16_t)(u >> 16);
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (OCP 8-bit floating point, E4M3 variant):                       */
/*   1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;                 */
/*   exponent field 0 = subnormal, value (m/8) * 2^-6;                      */
/*   S.1111.111 is NaN; no infinities; largest finite 1.75 * 2^8 = 448.     */
/* ------------------------------------------------------------------------ */

float ep_oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int ex = (code >> 3) & 0xf;
    int man = code & 7;
    double v;
    if (ex == 0xf && man == 7) return NAN;
    if (ex == 0) v = ldexp((double)man / 8.0, -6);
    else v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return (float)(sign ? -v : v);
}

/* Round half to even of a non-negative double that is a multiple of 2^-k
 * for small k (exact in double).  Returns an integer-valued double. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double frac = q - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary32 -> e4m3, round to nearest even, saturating to +-448 (satfinite).
 * NaN -> 0x7f (with sign). */
uint8_t ep_oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v)) return (uint8_t)(sign | 0x7f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; a result of 8 steps is the smallest
         * normal, whose code is also 8 (exponent field 1, mantissa 0). */
        double m = round_half_even(a / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e;
    frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                     /* a in [2^e, 2^(e+1)) */
    double m = round_half_even(a / ldexp(1.0, e - 3));  /* in [8, 16] */
    if (m == 16.0) { m = 8.0; e += 1; }
    int field = e + 7;
    int code = (field << 3) | ((int)m - 8);
    if (code > 0x7e) code = 0x7e;  /* 480 is not finite in E4M3 -> 448 */
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------ */
/* Layout: routing counts, membership and prefix offsets.                   */
/* [P1 section 6.1] psum_num_recv_tokens_per_scaleup_rank,                 */
/* psum_num_recv_tokens_per_expert, dst_buffer_slot_idx, expert_alignment;  */
/* [P1 section 7.3] per-rank and per-local-expert receive counts.           */
/*                                                                          */
/* Per token t in ascending order and per k: skip -1; flag and skip ids     */
/* outside [0,E); count the expert; mark its rank and node.  Then each      */
/* marked rank gives t the next local slot of that rank.  Offsets are the   */
/* exclusive prefix sums; dst_row = rank_offset[r] + local slot, else -1.   */
/* ------------------------------------------------------------------------ */

int ep_oracle_layout(const int64_t* topk_idx, int T, int K, int E, int R,
                     int ranks_per_node, int expert_alignment,
                     int32_t* num_tokens_per_rank,     /* [R]            */
                     int32_t* num_tokens_per_node,     /* [R/rpn] or NULL */
                     int32_t* num_tokens_per_expert,   /* [E]            */
                     uint8_t* is_token_in_rank,        /* [T,R]          */
                     int32_t* rank_offset,             /* [R+1]          */
                     int32_t* expert_offset,           /* [E+1]          */
                     int32_t* dst_row,                 /* [T,R]          */
                     int32_t* src_dst_count,           /* [R,R] or NULL  */
                     int32_t* token_offset,            /* [T+1] or NULL  */
                     int32_t* scratch_local,           /* [T,R] scratch  */
                     uint8_t* scratch_mark)            /* [R + nodes]    */
{
    int status = OR_OK;
    int experts_per_rank = E / R;
    int num_nodes = (ranks_per_node > 0) ? R / ranks_per_node : 0;
    int align = expert_alignment > 0 ? expert_alignment : 1;

    for (int r = 0; r < R; ++r) num_tokens_per_rank[r] = 0;
    for (int e = 0; e < E; ++e) num_tokens_per_expert[e] = 0;
    if (num_tokens_per_node)
        for (int n = 0; n < num_nodes; ++n) num_tokens_per_node[n] = 0;

    uint8_t* mark = scratch_mark;
    uint8_t* node_mark = scratch_mark + R;

    for (int t = 0; t < T; ++t) {
        for (int r = 0; r < R; ++r) mark[r] = 0;
        for (int n = 0; n < num_nodes; ++n) node_mark[n] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) { status |= OR_INVALID_INDEX; continue; }
            num_tokens_per_expert[e] += 1;
            int r = (int)(e / experts_per_rank);
            mark[r] = 1;
            if (num_nodes > 0) node_mark[r / ranks_per_node] = 1;
        }
        for (int r = 0; r < R; ++r) {
            is_token_in_rank[(int64_t)t * R + r] = mark[r];
            if (mark[r]) {
                scratch_local[(int64_t)t * R + r] = num_tokens_per_rank[r];
                num_tokens_per_rank[r] += 1;
            } else {
                scratch_local[(int64_t)t * R + r] = -1;
            }
        }
        if (num_tokens_per_node)
            for (int n = 0; n < num_nodes; ++n)
                num_tokens_per_node[n] += node_mark[n];
    }

    rank_offset[0] = 0;
    for (int r = 0; r < R; ++r)
        rank_offset[r + 1] = rank_offset[r] + num_tokens_per_rank[r];

    expert_offset[0] = 0;
    for (int e = 0; e < E; ++e) {
        int c = num_tokens_per_expert[e];
        int padded = ((c + align - 1) / align) * align;
        expert_offset[e + 1] = expert_offset[e] + padded;
    }

    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r) {
            int32_t l = scratch_local[(int64_t)t * R + r];
            dst_row[(int64_t)t * R + r] = (l >= 0) ? rank_offset[r] + l : -1;
        }

    /* Rows numbered token by token: token_offset[t] = sum over t' < t of
     * the number of ranks that receive t'. */
    if (token_offset) {
        token_offset[0] = 0;
        for (int t = 0; t < T; ++t) {
            int n = 0;
            for (int r = 0; r < R; ++r) n += is_token_in_rank[(int64_t)t * R + r];
            token_offset[t + 1] = token_offset[t] + n;
        }
    }

    /* Source rank s owns tokens [s*T/R, (s+1)*T/R) (needs R | T). */
    if (src_dst_count) {
        for (int i = 0; i < R * R; ++i) src_dst_count[i] = 0;
        int per_src = T / R;
        for (int t = 0; t < T && per_src > 0; ++t) {
            int s = t / per_src;
            for (int r = 0; r < R; ++r)
                if (is_token_in_rank[(int64_t)t * R + r])
                    src_dst_count[s * R + r] += 1;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* FP8 cast of one row: [P1 section 6.1] / [P1 section 9.1]                 */
/* use_fp8_dispatch with per-block scale factors (sf_ptr, num_sf_packs).    */
/* ------------------------------------------------------------------------ */

void ep_oracle_fp8_cast_row(const uint16_t* x_row, int H, uint8_t* q_row, float* sf_row)
{
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(ep_oracle_bf16_to_float(x_row[b * 128 + i]));
            if (v > amax) amax = v;
        }
        float sf, mult;
        if (amax > 0.0f) {
            volatile float a = amax;        /* two separate fp32 divides */
            sf = a / 448.0f;
            mult = 448.0f / a;
        } else {
            sf = 1.0f;
            mult = 0.0f;
        }
        sf_row[b] = sf;
        for (int i = 0; i < 128; ++i) {
            volatile float p = ep_oracle_bf16_to_float(x_row[b * 128 + i]) * mult;
            q_row[b * 128 + i] = ep_oracle_e4m3_encode(p);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dispatch: [P1 section 9.2] recv_x, recv_topk_idx, recv_topk_weights;     */
/* [P2 TokenLayout fragment] each received row carries hidden, sf,          */
/* topk_idx, topk_weights and the source token index.                       */
/*                                                                          */
/* tokens: list of source tokens to dispatch (NULL = all T in order).       */
/* compact = 0: output row = dst_row[t,r] (arrays sized by capacity).        */
/* compact = 1: output rows are numbered 0,1,2,... in (listed token, rank)  */
/*              order and out_rows[j] receives dst_row[t,r].               */
/* fp8 = 0: recv_x rows are H bf16 (2H bytes); fp8 = 1: H e4m3 bytes and    */
/* recv_sf rows of H/128 floats (row-major) or, when sf_col_major, element  */
/* (j, b) at recv_sf[b * sf_stride + j].                                    */
/* Returns status bits (invalid index, capacity).                           */
/* ------------------------------------------------------------------------ */

int ep_oracle_dispatch(const uint16_t* x, const int64_t* topk_idx, const float* topk_weights,
                       int T, int H, int K, int E, int R, const int32_t* dst_row,
                       const int32_t* tokens, int num_listed, int compact, int64_t capacity,
                       int fp8, int sf_col_major, int64_t sf_stride,
                       uint8_t* recv_x, float* recv_sf, int32_t* recv_topk_idx,
                       float* recv_topk_weights, int32_t* recv_src_idx, int32_t* out_rows)
{
    int status = OR_OK;
    int experts_per_rank = E / R;
    int n_list = tokens ? num_listed : T;
    int64_t j = 0;
    size_t row_bytes = fp8 ? (size_t)H : (size_t)H * 2;
    int nb = H / 128;

    /* Tokens write disjoint rows when not compact, so a build with OpenMP
     * (the all-cores timing of the benchmark) may split this loop over
     * threads; without OpenMP the pragma is ignored.  Same work either way. */
#pragma omp parallel for schedule(static) reduction(|:status) if(!compact)
    for (int i = 0; i < n_list; ++i) {
        int t = tokens ? tokens[i] : i;
        uint8_t q_tmp[65536];
        float sf_tmp[512];
        for (int r = 0; r < R; ++r) {
            int32_t d = dst_row[(int64_t)t * R + r];
            if (d < 0) continue;
            int64_t row;
            if (compact) { row = j; out_rows[j] = d; j += 1; }
            else {
                if ((int64_t)d >= capacity) { status |= OR_CAPACITY; continue; }
                row = d;
            }
            const uint16_t* src = x + (int64_t)t * H;
            if (fp8) {
                ep_oracle_fp8_cast_row(src, H, q_tmp, sf_tmp);
                memcpy(recv_x + row * (int64_t)row_bytes, q_tmp, row_bytes);
                if (recv_sf)
                    for (int b = 0; b < nb; ++b) {
                        if (sf_col_major) recv_sf[(int64_t)b * sf_stride + row] = sf_tmp[b];
                        else recv_sf[row * nb + b] = sf_tmp[b];
                    }
            } else {
                memcpy(recv_x + row * (int64_t)row_bytes, src, row_bytes);
            }
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[(int64_t)t * K + k];
                int on_r = (e >= 0 && e < E && (int)(e / experts_per_rank) == r);
                if (recv_topk_idx)
                    recv_topk_idx[row * K + k] = on_r ? (int32_t)(e - (int64_t)r * experts_per_rank) : -1;
                if (recv_topk_weights)
                    recv_topk_weights[row * K + k] = on_r ? topk_weights[(int64_t)t * K + k] : 0.0f;
                if (e < -1 || e >= E) status |= OR_INVALID_INDEX;
            }
            if (recv_src_idx) recv_src_idx[row] = t;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Combine: [P1 section 9.2] combine(x, handle, topk_weights) -> combined_x. */
/* For each listed token t: out[t] = sum over r ascending with              */
/* dst_row[t,r] >= 0 of c(t,r) * y[dst_row[t,r]], with c = 1 (weighted = 0) */
/* or c = sum over k of topk_weights[t,k] whose expert is on r.             */
/* fp64 accumulation; out row i belongs to the i-th listed token.           */
/* Rows at or beyond num_y_rows are skipped and flagged.                    */
/* ------------------------------------------------------------------------ */

int ep_oracle_combine(const uint16_t* y, int64_t num_y_rows,
                      const int64_t* topk_idx, const float* topk_weights, int weighted,
                      int T, int H, int K, int E, int R, const int32_t* dst_row,
                      const int32_t* tokens, int num_listed, double* out)
{
    int status = OR_OK;
    int experts_per_rank = E / R;
    int n_list = tokens ? num_listed : T;
    /* one output row per listed token: threads may share the tokens (OpenMP build) */
#pragma omp parallel for schedule(static) reduction(|:status)
    for (int i = 0; i < n_list; ++i) {
        int t = tokens ? tokens[i] : i;
        double* o = out + (int64_t)i * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int r = 0; r < R; ++r) {
            int32_t d = dst_row[(int64_t)t * R + r];
            if (d < 0) continue;
            if ((int64_t)d >= num_y_rows) { status |= OR_CAPACITY; continue; }
            double c = 1.0;
            if (weighted) {
                c = 0.0;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[(int64_t)t * K + k];
                    if (e >= 0 && e < E && (int)(e / experts_per_rank) == r)
                        c += (double)topk_weights[(int64_t)t * K + k];
                }
            }
            const uint16_t* yr = y + (int64_t)d * H;
            for (int h = 0; h < H; ++h)
                o[h] += c * (double)ep_oracle_bf16_to_float(yr[h]);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Array forms of the element conversions above (test convenience).         */
/* ------------------------------------------------------------------------ */

void ep_oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_e4m3_encode(v[i]);
}

void ep_oracle_e4m3_decode_array(const uint8_t* c, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_e4m3_decode(c[i]);
}

void ep_oracle_float_to_bf16_array(const float* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_float_to_bf16(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Expanded (per-expert) receive layout: [P2] dispatch_copy_epilogue and     */
/* combine_reduce_epilogue, [P2 TokenLayout fragment] linked_list_idx,      */
/* [P1 section 6.1] expert_alignment.  Every valid (t, k) gets its own row: */
/* expert e's rows are expert_offset[e] + 0, 1, ... in (token, k) order,    */
/* so rows are grouped by expert (ranks' experts in order) and each         */
/* expert's block starts at its aligned offset.  Masked or invalid -> -1.   */
/* ------------------------------------------------------------------------ */

int ep_oracle_expanded_rows(const int64_t* topk_idx, int T, int K, int E,
                            const int32_t* expert_offset, int32_t* expanded_row,
                            int32_t* scratch_count /* [E] */)
{
    int status = OR_OK;
    for (int e = 0; e < E; ++e) scratch_count[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            int64_t i = (int64_t)t * K + k;
            if (e < 0 || e >= E) {
                expanded_row[i] = -1;
                if (e < -1 || e >= E) status |= OR_INVALID_INDEX;
                continue;
            }
            expanded_row[i] = expert_offset[e] + scratch_count[e];
            scratch_count[e] += 1;
        }
    return status;
}

/* Expanded dispatch: row expanded_row[t,k] receives x[t] (bf16 copy or the  */
/* FP8 cast), its source token t and its weight topk_weights[t,k].         */
/* FP8 scales: row-major [row][block], or with sf_col_major the TMA-aligned  */
/* column-major form of [P2 SF-layout fragment] / [P1 section 6.1]          */
/* (sf_token_stride = 1, sf_hidden_stride = sf_stride): scale (row, b) at   */
/* b * sf_stride + row.  Padding rows of an expert block are not written.   */
int ep_oracle_dispatch_expanded(const uint16_t* x, const float* topk_weights, int T, int H, int K,
                                const int32_t* expanded_row, int64_t capacity, int fp8,
                                int sf_col_major, int64_t sf_stride,
                                uint8_t* recv_x, float* recv_sf, int32_t* recv_src_idx,
                                float* recv_weight)
{
    int status = OR_OK;
    size_t row_bytes = fp8 ? (size_t)H : (size_t)H * 2;
    int nb = H / 128;
    uint8_t q_tmp[65536];
    float sf_tmp[512];
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t d = expanded_row[(int64_t)t * K + k];
            if (d < 0) continue;
            if ((int64_t)d >= capacity) { status |= OR_CAPACITY; continue; }
            const uint16_t* src = x + (int64_t)t * H;
            if (fp8) {
                ep_oracle_fp8_cast_row(src, H, q_tmp, sf_tmp);
                memcpy(recv_x + (int64_t)d * (int64_t)row_bytes, q_tmp, row_bytes);
                if (recv_sf)
                    for (int b = 0; b < nb; ++b) {
                        if (sf_col_major) recv_sf[(int64_t)b * sf_stride + d] = sf_tmp[b];
                        else recv_sf[(int64_t)d * nb + b] = sf_tmp[b];
                    }
            } else {
                memcpy(recv_x + (int64_t)d * (int64_t)row_bytes, src, row_bytes);
            }
            if (recv_src_idx) recv_src_idx[d] = t;
            if (recv_weight) recv_weight[d] = topk_weights[(int64_t)t * K + k];
        }
    return status;
}

/* Expanded combine: out[t] = sum over valid k (ascending) of c * y[expanded_row[t,k]], */
/* c = topk_weights[t,k] (weighted) or 1; fp64 accumulation.                         */
int ep_oracle_combine_expanded(const uint16_t* y, int64_t num_y_rows, const float* topk_weights,
                               int weighted, int T, int H, int K, const int32_t* expanded_row,
                               double* out)
{
    int status = OR_OK;
    for (int t = 0; t < T; ++t) {
        double* o = out + (int64_t)t * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int k = 0; k < K; ++k) {
            int32_t d = expanded_row[(int64_t)t * K + k];
            if (d < 0) continue;
            if ((int64_t)d >= num_y_rows) { status |= OR_CAPACITY; continue; }
            double c = weighted ? (double)topk_weights[(int64_t)t * K + k] : 1.0;
            const uint16_t* yr = y + (int64_t)d * H;
            for (int h = 0; h < H; ++h) o[h] += c * (double)ep_oracle_bf16_to_float(yr[h]);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Combined top-k weights: [P1 section 9.2] combine returns                 */
/* combined_topk_weights.  For every token t and slot k: the fp32 sum over  */
/* the ranks r holding t (ascending) of the received row's weight in slot k. */
/* Rows at or beyond num_rows are skipped and flagged.                      */
/* ------------------------------------------------------------------------ */

int ep_oracle_combine_topk_weights(const float* recv_topk_weights, int64_t num_rows, int T, int K,
                                   int R, const int32_t* dst_row, float* combined)
{
    int status = OR_OK;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            float acc = 0.0f;
            for (int r = 0; r < R; ++r) {
                int32_t d = dst_row[(int64_t)t * R + r];
                if (d < 0) continue;
                if ((int64_t)d >= num_rows) { status |= OR_CAPACITY; continue; }
                acc += recv_topk_weights[(int64_t)d * K + k];
            }
            combined[(int64_t)t * K + k] = acc;
        }
    return status;
}

/* Cumulative receive statistics: [P1 section 6.1]                          */
/* cumulative_local_expert_recv_stats -- stats[e] += tokens routed to e.    */
void ep_oracle_accumulate_expert_stats(const int32_t* num_tokens_per_expert, int E, int64_t* stats)
{
    for (int e = 0; e < E; ++e) stats[e] += num_tokens_per_expert[e];
}

/* ------------------------------------------------------------------------ */
/* Hierarchical (two-stage) path: [P2] hybrid_dispatch / hybrid_combine,    */
/* chosen when there is more than one scale-out domain, and the             */
/* WorkspaceLayout fragment (scale-out rank counts kept beside the          */
/* scale-up ones); [P3 section 3.2] node = rank / ranks_per_node.           */
/* Readings: node n holds ranks [n*rpn, (n+1)*rpn); a token crosses the     */
/* scale-out link once per node that holds any of its experts (node-level   */
/* deduplication) and is then copied inside the node to each rank that      */
/* needs it.  Node n's scale-out buffer holds its tokens in ascending t.    */
/* Combine runs the other way: a scale-up reduce per (token, node) stored   */
/* as bf16 (the data type on the link), then a scale-out reduce of the      */
/* token's node partials.                                                   */
/* ------------------------------------------------------------------------ */

/* fp64 -> nearest bf16, ties to even, in one rounding (finite inputs inside */
/* bf16's range).  |v| = m * 2^e with m in [0.5, 1): the bf16 quantum is    */
/* 2^(e-8), and below the smallest normal (e < -125) the fixed subnormal    */
/* quantum 2^-133.  nearbyint rounds ties to even in the default mode.      */
uint16_t ep_oracle_double_to_bf16(double v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint16_t b = 0;
    if (a != 0.0) {
        int e;
        (void)frexp(a, &e);
        if (e < -125) e = -125;
        double q = nearbyint(ldexp(a, 8 - e));      /* integer, at most 2^8 */
        float f = (float)ldexp(q, e - 8);           /* exact: <= 8 significant bits */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        b = (uint16_t)(u >> 16);
    }
    return neg ? (uint16_t)(b | 0x8000u) : b;
}

void ep_oracle_double_to_bf16_array(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_double_to_bf16(v[i]);
}

/* Node rows: node_row[t, n] = row of token t in node n's scale-out buffer   */
/* (node_offset[n] + number of earlier tokens reaching n) or -1;             */
/* node_offset is the exclusive prefix of the per-node token counts.        */
int ep_oracle_node_rows(const int64_t* topk_idx, int T, int K, int E, int R, int rpn,
                        int32_t* node_offset, int32_t* node_row)
{
    int status = OR_OK;
    int nodes = R / rpn;
    int experts_per_rank = E / R;
    node_offset[0] = 0;
    for (int n = 0; n < nodes; ++n) {
        int32_t count = 0;
        for (int t = 0; t < T; ++t) {
            int hit = 0;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[(int64_t)t * K + k];
                if (e < -1 || e >= E) { status |= OR_INVALID_INDEX; continue; }
                if (e >= 0 && (int)(e / experts_per_rank) / rpn == n) hit = 1;
            }
            node_row[(int64_t)t * nodes + n] = hit ? node_offset[n] + count : -1;
            count += hit;
        }
        node_offset[n + 1] = node_offset[n] + count;
    }
    return status;
}

/* Hierarchical dispatch.  Stage 1 (scale-out): node_x[node_row[t,n]] = x[t]  */
/* (bf16 copy, or the FP8 cast with row-major node_sf), node_src_idx = t.   */
/* Stage 2 (scale-up): every node row j of node n is forwarded to each rank */
/* r of n with dst_row[t,r] >= 0 (t = node_src_idx[j]): recv_x / recv_sf   */
/* copied from the node row, metadata as in ep_oracle_dispatch.             */
int ep_oracle_dispatch_hierarchical(const uint16_t* x, const int64_t* topk_idx,
                                    const float* topk_weights, int T, int H, int K, int E, int R,
                                    int rpn, const int32_t* node_row, const int32_t* dst_row, int fp8,
                                    int64_t node_capacity, uint8_t* node_x, float* node_sf,
                                    int32_t* node_src_idx, int64_t recv_capacity, int sf_col_major,
                                    int64_t sf_stride, uint8_t* recv_x, float* recv_sf,
                                    int32_t* recv_topk_idx, float* recv_topk_weights,
                                    int32_t* recv_src_idx)
{
    int status = OR_OK;
    int nodes = R / rpn;
    int experts_per_rank = E / R;
    size_t row_bytes = fp8 ? (size_t)H : (size_t)H * 2;
    int nb = H / 128;
    uint8_t q_tmp[65536];
    float sf_tmp[512];

    /* stage 1: one copy of each token per node it reaches */
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < nodes; ++n) {
            int32_t j = node_row[(int64_t)t * nodes + n];
            if (j < 0) continue;
            if ((int64_t)j >= node_capacity) { status |= OR_CAPACITY; continue; }
            const uint16_t* src = x + (int64_t)t * H;
            if (fp8) {
                ep_oracle_fp8_cast_row(src, H, q_tmp, sf_tmp);
                memcpy(node_x + (int64_t)j * (int64_t)row_bytes, q_tmp, row_bytes);
                for (int b = 0; b < nb; ++b) node_sf[(int64_t)j * nb + b] = sf_tmp[b];
            } else {
                memcpy(node_x + (int64_t)j * (int64_t)row_bytes, src, row_bytes);
            }
            node_src_idx[j] = t;
        }

    /* stage 2: each node row to the ranks of its node that need the token */
    for (int n = 0; n < nodes; ++n)
        for (int t0 = 0; t0 < T; ++t0) {
            int32_t j = node_row[(int64_t)t0 * nodes + n];
            if (j < 0 || (int64_t)j >= node_capacity) continue;
            int t = node_src_idx[j];
            for (int r = n * rpn; r < (n + 1) * rpn; ++r) {
                int32_t d = dst_row[(int64_t)t * R + r];
                if (d < 0) continue;
                if ((int64_t)d >= recv_capacity) { status |= OR_CAPACITY; continue; }
                memcpy(recv_x + (int64_t)d * (int64_t)row_bytes, node_x + (int64_t)j * (int64_t)row_bytes,
                       row_bytes);
                if (fp8 && recv_sf)
                    for (int b = 0; b < nb; ++b) {
                        float s = node_sf[(int64_t)j * nb + b];
                        if (sf_col_major) recv_sf[(int64_t)b * sf_stride + d] = s;
                        else recv_sf[(int64_t)d * nb + b] = s;
                    }
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[(int64_t)t * K + k];
                    int on_r = (e >= 0 && e < E && (int)(e / experts_per_rank) == r);
                    if (recv_topk_idx)
                        recv_topk_idx[(int64_t)d * K + k] = on_r ? (int32_t)(e - (int64_t)r * experts_per_rank) : -1;
                    if (recv_topk_weights)
                        recv_topk_weights[(int64_t)d * K + k] = on_r ? topk_weights[(int64_t)t * K + k] : 0.0f;
                }
                if (recv_src_idx) recv_src_idx[d] = t;
            }
        }
    return status;
}

/* Hierarchical combine.  Stage 1 (scale-up reduce): for every (t, n) with   */
/* j = node_row[t,n] >= 0, node_y[j] = bf16( sum over ranks r of n,         */
/* ascending, with dst_row[t,r] >= 0 of c(t,r) * y[dst_row[t,r]] ) (fp64    */
/* sum, one rounding; c as in ep_oracle_combine).  Stage 2 (scale-out       */
/* reduce): out[t] = sum over nodes n ascending with j >= 0 of node_y[j]    */
/* (fp64, returned unrounded).                                               */
int ep_oracle_combine_hierarchical(const uint16_t* y, int64_t num_y_rows, const int64_t* topk_idx,
                                   const float* topk_weights, int weighted, int T, int H, int K, int E,
                                   int R, int rpn, const int32_t* node_row, const int32_t* dst_row,
                                   int64_t node_capacity, uint16_t* node_y, double* out,
                                   double* scratch /* [H] */)
{
    int status = OR_OK;
    int nodes = R / rpn;
    int experts_per_rank = E / R;

    /* stage 1 */
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < nodes; ++n) {
            int32_t j = node_row[(int64_t)t * nodes + n];
            if (j < 0) continue;
            if ((int64_t)j >= node_capacity) { status |= OR_CAPACITY; continue; }
            for (int h = 0; h < H; ++h) scratch[h] = 0.0;
            for (int r = n * rpn; r < (n + 1) * rpn; ++r) {
                int32_t d = dst_row[(int64_t)t * R + r];
                if (d < 0) continue;
                if ((int64_t)d >= num_y_rows) { status |= OR_CAPACITY; continue; }
                double c = 1.0;
                if (weighted) {
                    c = 0.0;
                    for (int k = 0; k < K; ++k) {
                        int64_t e = topk_idx[(int64_t)t * K + k];
                        if (e >= 0 && e < E && (int)(e / experts_per_rank) == r)
                            c += (double)topk_weights[(int64_t)t * K + k];
                    }
                }
                const uint16_t* yr = y + (int64_t)d * H;
                for (int h = 0; h < H; ++h) scratch[h] += c * (double)ep_oracle_bf16_to_float(yr[h]);
            }
            for (int h = 0; h < H; ++h) node_y[(int64_t)j * H + h] = ep_oracle_double_to_bf16(scratch[h]);
        }

    /* stage 2 */
    for (int t = 0; t < T; ++t) {
        double* o = out + (int64_t)t * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int n = 0; n < nodes; ++n) {
            int32_t j = node_row[(int64_t)t * nodes + n];
            if (j < 0 || (int64_t)j >= node_capacity) continue;
            for (int h = 0; h < H; ++h) o[h] += (double)ep_oracle_bf16_to_float(node_y[(int64_t)j * H + h]);
        }
    }
    return status;
}
