/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-parallel route -> dispatch -> expert stand-in -> combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * import this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; every step is written out as the plain definition, in
 * nested loops, so it can be checked against the sources by eye.
 *
 * Sources (web pages; cited by title and section):
 *   [DSD] Perplexity, "Lower latency and higher throughput with multi-node
 *         DeepSeek deployment" -- sections "Expert parallelism",
 *         "Quantization", "MoE router".
 *   [EFA] Perplexity, "Enabling trillion-parameter models on AWS EFA" --
 *         sections "Send and receive buffers", "Dispatch and combine".
 *   [EPK] lehuy.net, "Giai ma nhan EP hieu suat cao" (Decoding
 *         high-performance EP kernels) -- sections "Our task",
 *         "Optimising for throughput: ask first, send later" > "Dispatch",
 *         > "Combine", and "Optimising for latency: send without asking".
 *
 * Notation: R ranks, E experts, K experts per token, H hidden size,
 * L = E/R local experts per rank (expert e lives on rank e / L), B[s] tokens
 * on rank s, T = sum B[s]; global token g is rank-major, g = rank_off[s] + t.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -lm.
 * -ffp-contract=off is required: every fp32 multiply and add below must be
 * rounded on its own, exactly as written (the only fused multiply-add is the
 * explicit fmaf() in the combine accumulation).
 *
 * Parity status per function (what pins each one is in the test suite):
 *   oracle_bf16_from_f32 / oracle_f32_from_bf16   pinned (library cast, IEEE cases)
 *   oracle_e4m3_decode / oracle_e4m3_encode       pinned (library cast, OCP table)
 *   oracle_route_topk                             pinned (argmax, full sort, brute force, softmax)
 *   oracle_route_topk_grouped                     pinned (one group / all groups = plain route, library sort)
 *   oracle_dispatch                               pinned (library stable sort, brute force, invariants)
 *   oracle_dispatch_ll / oracle_combine_ll_push   pinned (same slots and payload as the ragged layout)
 *   oracle_expert_scale                           pinned (library arithmetic)
 *   oracle_combine / oracle_combine_f64           pinned (identity experts, one-hot, error bound)
 *   oracle_combine_partial                        pinned (R = 1 gives the receive-side result, slots, bound)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the top 16 bits of an IEEE binary32.  Round to nearest, ties to
 * even on the 16 dropped bits; NaN keeps its sign and becomes a quiet NaN. */
uint16_t oracle_bf16_from_f32(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)            /* NaN */
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                                 /* may carry into inf: correct */
    return (uint16_t)upper;
}

float oracle_f32_from_bf16(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits.  No infinities; S.1111.111 is NaN; largest finite value is
 * S.1111.110 = 1.75 * 2^8 = 448.  Exponent field 0 encodes subnormals
 * m/8 * 2^-6. */
float oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int ex = (c >> 3) & 15;
    int man = c & 7;
    float v;
    if (ex == 15 && man == 7) return sign ? -NAN : NAN;
    if (ex == 0) v = ldexpf((float)man, -9);              /* man/8 * 2^-6 */
    else v = ldexpf((float)(8 + man), ex - 7 - 3);        /* (1+man/8) * 2^(ex-7) */
    return sign ? -v : v;
}

/* Round a non-negative value that is already scaled so that one unit in the
 * last place is 1.0 to the nearest integer, ties to even.  f < 2^24, so the
 * truncation and the subtraction below are exact. */
static uint32_t round_half_even(float f)
{
    uint32_t i = (uint32_t)f;
    float frac = f - (float)i;
    if (frac > 0.5f || (frac == 0.5f && (i & 1u))) i += 1u;
    return i;
}

/* fp32 -> E4M3, round to nearest even, saturating: any finite or infinite
 * magnitude that would round past 448 becomes 448 (same sign); NaN -> NaN. */
uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign = (f32_bits(x) >> 31) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7f);
    float a = fabsf(x);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7e);
    if (a < 0x1p-6f) {
        /* subnormal range: spacing 2^-9; a * 2^9 is exact */
        uint32_t m = round_half_even(a * 512.0f);      /* 0..8; 8 == smallest normal */
        return (uint8_t)(sign | m);
    }
    int e2;
    frexpf(a, &e2);                                    /* a = f * 2^e2, f in [0.5,1) */
    int E = e2 - 1;                                    /* a in [2^E, 2^(E+1)), E in -6..8 */
    uint32_t q = round_half_even(ldexpf(a, 3 - E));    /* in 8..16, exact scaling */
    if (q == 16u) { q = 8u; E += 1; }
    if (E > 8 || (E == 8 && q > 14u)) return (uint8_t)(sign | 0x7e);  /* past 448 */
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | (int)(q - 8u)));
}

/* ------------------------------------------------------------------------ */
/* Route: [DSD] "MoE router" (top-K scores with their expert indices) and     */
/* "Expert parallelism" (each token goes to K routed experts whose outputs are */
/* summed with weights).  Reading: ties between equal logits go to the smaller */
/* expert id; output order is by descending logit; the K weights are the       */
/* softmax of the K selected logits (= full softmax renormalised over the      */
/* top-K).  Weights are evaluated in fp64 and rounded once to fp32.            */
/* ------------------------------------------------------------------------ */
void oracle_route_topk(const float *logits, int T, int E, int K,
                       int32_t *topk_idx, float *topk_w)
{
    unsigned char *chosen = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    double *ex = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int g = 0; g < T; ++g) {
        const float *l = logits + (size_t)g * E;
        memset(chosen, 0, (size_t)E);
        for (int j = 0; j < K; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: lower id wins ties */
            }
            chosen[best] = 1;
            topk_idx[(size_t)g * K + j] = best;
        }
        double m = (double)l[topk_idx[(size_t)g * K]];
        double sum = 0.0;
        for (int j = 0; j < K; ++j) {
            ex[j] = exp((double)l[topk_idx[(size_t)g * K + j]] - m);
            sum += ex[j];
        }
        for (int j = 0; j < K; ++j)
            topk_w[(size_t)g * K + j] = (float)(ex[j] / sum);
    }
    free(chosen);
    free(ex);
}

/* ------------------------------------------------------------------------ */
/* Group-limited route: [DSD] "MoE router" (DeepSeek's routing takes a group  */
/* top-K first; Mixtral's routing is the special case where the group top-K  */
/* is the group of all experts).  Reading (the page gives no formula): the E  */
/* experts form n_groups contiguous groups of E/n_groups; a group's score is  */
/* its largest logit; the topk_groups best groups are kept (equal scores ->   */
/* smaller group id); then the K largest logits among the kept groups' experts */
/* are chosen exactly as in oracle_route_topk, and weighted the same way.     */
/* ------------------------------------------------------------------------ */
void oracle_route_topk_grouped(const float *logits, int T, int E, int K, int n_groups, int topk_groups,
                               int32_t *topk_idx, float *topk_w)
{
    int gs = E / n_groups;
    unsigned char *allowed = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    unsigned char *chosen = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    unsigned char *gkept = (unsigned char *)malloc((size_t)(n_groups > 0 ? n_groups : 1));
    float *gscore = (float *)malloc(sizeof(float) * (size_t)(n_groups > 0 ? n_groups : 1));
    double *ex = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int g = 0; g < T; ++g) {
        const float *l = logits + (size_t)g * E;
        /* 1. group scores */
        for (int q = 0; q < n_groups; ++q) {
            float m = l[q * gs];
            for (int e = q * gs + 1; e < (q + 1) * gs; ++e)
                if (l[e] > m) m = l[e];
            gscore[q] = m;
            gkept[q] = 0;
        }
        /* 2. keep the topk_groups best groups */
        for (int r = 0; r < topk_groups; ++r) {
            int best = -1;
            for (int q = 0; q < n_groups; ++q) {
                if (gkept[q]) continue;
                if (best < 0 || gscore[q] > gscore[best]) best = q;
            }
            gkept[best] = 1;
        }
        for (int e = 0; e < E; ++e) {
            allowed[e] = gkept[e / gs];
            chosen[e] = 0;
        }
        /* 3. top-K among the allowed experts */
        for (int j = 0; j < K; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (!allowed[e] || chosen[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            chosen[best] = 1;
            topk_idx[(size_t)g * K + j] = best;
        }
        /* 4. softmax over the chosen logits (fp64, rounded once) */
        double m = (double)l[topk_idx[(size_t)g * K]];
        double sum = 0.0;
        for (int j = 0; j < K; ++j) {
            ex[j] = exp((double)l[topk_idx[(size_t)g * K + j]] - m);
            sum += ex[j];
        }
        for (int j = 0; j < K; ++j)
            topk_w[(size_t)g * K + j] = (float)(ex[j] / sum);
    }
    free(allowed);
    free(chosen);
    free(gkept);
    free(gscore);
    free(ex);
}

/* ------------------------------------------------------------------------ */
/* FP8 block quantisation of one token row: [DSD] "Quantization" (activation  */
/* scales over 128-element vectors, computed on the fly) and [EPK] "Optimising */
/* for latency" (FP8 payload for dispatch).  Reading: per block of 128        */
/* channels, amax = max |x|, raised to at least 2^-119; scale = amax / 448 and */
/* inv = 448 / amax, each one IEEE fp32 division (subnormal results kept);    */
/* q = e4m3(x * inv) with one fp32 multiply and a saturating round-to-nearest- */
/* even encode.  Dequantised value: e4m3_decode(q) * scale.                    */
/* The pages say nothing of zero or tiny blocks.  2^-119 is the smallest power */
/* of two for which 448 / amax is finite in fp32 (448 * 2^119 = 1.75 * 2^127); */
/* below it the division would overflow and a zero element would give 0 * inf. */
/* With this floor no nonzero bf16 value encodes to a zero code because of the */
/* floor: the smallest, 2^-133, scales to 448 * 2^-14, above e4m3's 2^-6.      */
/* ------------------------------------------------------------------------ */
static void quantize_row_e4m3(const uint16_t *xrow, int H, uint8_t *q, float *scale)
{
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(oracle_f32_from_bf16(xrow[b * 128 + i]));
            if (v > amax) amax = v;
        }
        if (amax < 0x1p-119f) amax = 0x1p-119f;
        float s = amax / 448.0f;
        float inv = 448.0f / amax;
        scale[b] = s;
        for (int i = 0; i < 128; ++i) {
            float v = oracle_f32_from_bf16(xrow[b * 128 + i]);
            float p = v * inv;
            q[b * 128 + i] = oracle_e4m3_encode(p);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dispatch: [EPK] "Optimising for throughput" > "Dispatch" (count, exchange   */
/* counts, prefix sum gives the write layout, copy each token to its slot) and */
/* [EFA] "Dispatch and combine" (per-expert counts, prefix sum -> offsets,     */
/* pack; the receiver reorganises rows into the grouped-GEMM input).           */
/*                                                                            */
/* counts[e*R + s]  = number of tokens of rank s whose top-K contains e.       */
/* offsets          = exclusive prefix sum of counts in (e, s) order, E*R+1.   */
/* expert_offsets[e]= offsets[e*R] (E+1 entries).                              */
/* Rows inside one (e, s) segment follow the source token order t (reading:   */
/* the pages leave this open; ascending source is the plain choice).          */
/* tok2row[g*K + j] = row that holds the j-th copy of token g;                */
/* row2src[row]     = g*K + j (the inverse map).                               */
/* recv_fp8 == 0: recv is bf16 [T*K, H] (uint16 bit patterns), scale unused.  */
/* recv_fp8 != 0: recv is e4m3 [T*K, H], recv_scale fp32 [T*K, H/128].        */
/* Returns 0, or -1 if an index is outside [0, E).                            */
/* ------------------------------------------------------------------------ */
int oracle_dispatch(const uint16_t *x, const int32_t *topk_idx,
                    int R, const int32_t *B, int E, int K, int H, int recv_fp8,
                    void *recv, float *recv_scale,
                    int32_t *counts, int32_t *offsets, int32_t *expert_offsets,
                    int32_t *tok2row, int32_t *row2src)
{
    int64_t T = 0;
    for (int s = 0; s < R; ++s) T += B[s];
    for (int64_t i = 0; i < T * K; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;

    /* 1. count (the coordination pass's payload) */
    for (int i = 0; i < E * R; ++i) counts[i] = 0;
    int64_t g = 0;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < B[s]; ++t, ++g)
            for (int j = 0; j < K; ++j)
                counts[topk_idx[g * K + j] * R + s] += 1;

    /* 2. exclusive prefix sum over (e, s) */
    offsets[0] = 0;
    for (int i = 0; i < E * R; ++i) offsets[i + 1] = offsets[i] + counts[i];
    for (int e = 0; e <= E; ++e) expert_offsets[e] = offsets[e * R];

    /* 3. scatter with one write cursor per (e, s) */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E * R > 0 ? E * R : 1));
    for (int i = 0; i < E * R; ++i) cursor[i] = offsets[i];
    uint8_t *qrow = NULL;
    float *srow = NULL;
    if (recv_fp8) {
        qrow = (uint8_t *)malloc((size_t)H);
        srow = (float *)malloc(sizeof(float) * (size_t)(H / 128 > 0 ? H / 128 : 1));
    }
    g = 0;
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < B[s]; ++t, ++g) {
            const uint16_t *xrow = x + g * (int64_t)H;
            if (recv_fp8) quantize_row_e4m3(xrow, H, qrow, srow);   /* once per token */
            for (int j = 0; j < K; ++j) {
                int e = topk_idx[g * K + j];
                int32_t row = cursor[e * R + s]++;
                tok2row[g * K + j] = row;
                row2src[row] = (int32_t)(g * K + j);
                if (recv_fp8) {
                    memcpy((uint8_t *)recv + (int64_t)row * H, qrow, (size_t)H);
                    memcpy(recv_scale + (int64_t)row * (H / 128), srow,
                           sizeof(float) * (size_t)(H / 128));
                } else {
                    memcpy((uint16_t *)recv + (int64_t)row * H, xrow, sizeof(uint16_t) * (size_t)H);
                }
            }
        }
    }
    free(cursor);
    free(qrow);
    free(srow);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Low-latency dispatch: [EPK] "Optimising for latency: send without asking"  */
/* (a fixed private region per (source rank, expert) pair, sized for the     */
/* worst case, so the write address is a static formula -- no prefix sum over */
/* actual counts -- with the tokens a rank may dispatch per call capped at a  */
/* fixed chunk size C).                                                       */
/* Row of copy j of token g = (e*R + s)*C + slot, where s is g's rank and     */
/* slot counts the earlier tokens of rank s routed to e (ascending t, as in   */
/* the throughput layout).  recv has E*R*C rows; rows past counts[e*R+s] in a */
/* region are left untouched.  Requires B[s] <= C.  Returns 0, -1 for an      */
/* expert index out of range, -2 for B[s] > C.                                */
/* ------------------------------------------------------------------------ */
int oracle_dispatch_ll(const uint16_t *x, const int32_t *topk_idx,
                       int R, const int32_t *B, int E, int K, int H, int C, int recv_fp8,
                       void *recv, float *recv_scale, int32_t *counts,
                       int32_t *tok2row, int32_t *row2src)
{
    int64_t T = 0;
    for (int s = 0; s < R; ++s) {
        if (B[s] > C) return -2;
        T += B[s];
    }
    for (int64_t i = 0; i < T * K; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;
    for (int i = 0; i < E * R; ++i) counts[i] = 0;   /* doubles as the per-region cursor */
    uint8_t *qrow = NULL;
    float *srow = NULL;
    if (recv_fp8) {
        qrow = (uint8_t *)malloc((size_t)H);
        srow = (float *)malloc(sizeof(float) * (size_t)(H / 128 > 0 ? H / 128 : 1));
    }
    int64_t g = 0;
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < B[s]; ++t, ++g) {
            const uint16_t *xrow = x + g * (int64_t)H;
            if (recv_fp8) quantize_row_e4m3(xrow, H, qrow, srow);
            for (int j = 0; j < K; ++j) {
                int e = topk_idx[g * K + j];
                int32_t slot = counts[e * R + s]++;
                int64_t row = ((int64_t)e * R + s) * C + slot;
                tok2row[g * K + j] = (int32_t)row;
                row2src[row] = (int32_t)(g * K + j);
                if (recv_fp8) {
                    memcpy((uint8_t *)recv + row * H, qrow, (size_t)H);
                    memcpy(recv_scale + row * (H / 128), srow, sizeof(float) * (size_t)(H / 128));
                } else {
                    memcpy((uint16_t *)recv + row * H, xrow, sizeof(uint16_t) * (size_t)H);
                }
            }
        }
    }
    free(qrow);
    free(srow);
    return 0;
}

/* Push-style return of the low-latency layout ([EPK] "Optimising for        */
/* latency": dispatch tagged every token with where it came from, so the     */
/* expert's host writes each output straight to a private slot on the token's */
/* origin rank, indexed by the token's position there and by which of its K   */
/* experts this is).  ret[g*K + j] = y[row] for every filled row of the       */
/* rectangle (row2src[row] = g*K + j).  The origin then forms                 */
/* out[g] = sum_j w[g,j] * ret[g*K + j] (oracle_combine with tok2row = id).   */
void oracle_combine_ll_push(const uint16_t *y, const int32_t *row2src, const int32_t *counts,
                            int R, int E, int C, int H, uint16_t *ret)
{
    for (int e = 0; e < E; ++e)
        for (int s = 0; s < R; ++s)
            for (int slot = 0; slot < counts[e * R + s]; ++slot) {
                int64_t row = ((int64_t)e * R + s) * C + slot;
                memcpy(ret + (int64_t)row2src[row] * H, y + row * H, sizeof(uint16_t) * (size_t)H);
            }
}

/* ------------------------------------------------------------------------ */
/* Expert stand-in (replaces the grouped GEMM, which is not on this path):    */
/* y[row] = bf16( xhat * s_e ), s_e = 1 + e/256 (identity != 0: s_e = 1),      */
/* e = the expert whose segment [expert_offsets[e], expert_offsets[e+1])      */
/* holds the row; xhat = the bf16 value, or e4m3_decode(q) * scale (one fp32  */
/* multiply) for an FP8 receive buffer.                                       */
/* ------------------------------------------------------------------------ */
void oracle_expert_scale(const void *recv, const float *recv_scale, int recv_fp8,
                         const int32_t *expert_offsets, int E, int H, int identity,
                         uint16_t *y)
{
    for (int e = 0; e < E; ++e) {
        float se = identity ? 1.0f : 1.0f + (float)e / 256.0f;
        for (int32_t row = expert_offsets[e]; row < expert_offsets[e + 1]; ++row) {
            for (int h = 0; h < H; ++h) {
                float xhat;
                if (recv_fp8) {
                    uint8_t q = ((const uint8_t *)recv)[(int64_t)row * H + h];
                    xhat = oracle_e4m3_decode(q) * recv_scale[(int64_t)row * (H / 128) + h / 128];
                } else {
                    xhat = oracle_f32_from_bf16(((const uint16_t *)recv)[(int64_t)row * H + h]);
                }
                float v = xhat * se;
                y[(int64_t)row * H + h] = oracle_bf16_from_f32(v);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Combine: [EPK] "Optimising for throughput" > "Combine" (undo the dispatch  */
/* permutation and add up each token's contributions, reusing dispatch's      */
/* routing, no coordination) and [EFA] "Dispatch and combine" (the receiver   */
/* accumulates the returned tokens into the output as a weighted sum).        */
/* out[g] = sum_j w[g,j] * y[tok2row[g*K+j]], accumulated in fp32 by explicit */
/* fused multiply-add in fixed order j = 0..K-1 starting from +0, then kept   */
/* as fp32 (out_f32) or rounded to bf16 (out_bf16).  Either output may be     */
/* NULL.                                                                       */
/* ------------------------------------------------------------------------ */
void oracle_combine(const uint16_t *y, const int32_t *tok2row, const float *topk_w,
                    int T, int K, int H, uint16_t *out_bf16, float *out_f32)
{
    for (int64_t g = 0; g < T; ++g) {
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < K; ++j) {
                int32_t row = tok2row[g * K + j];
                float v = oracle_f32_from_bf16(y[(int64_t)row * H + h]);
                acc = fmaf(topk_w[g * K + j], v, acc);
            }
            if (out_f32) out_f32[g * H + h] = acc;
            if (out_bf16) out_bf16[g * H + h] = oracle_bf16_from_f32(acc);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Sender-side partial accumulation: [EFA] "Evaluation" (DeepEP accumulates  */
/* on the sending side of combine to cut the bytes returned; doing so may    */
/* affect precision; pplx accumulates on the receiving side).  Reading (no   */
/* formula on the page): rank r hosts the experts e with e / (E/R) == r; for */
/* each token g and each rank r hosting at least one of g's experts,         */
/*   p[g,r] = bf16( fp32 fma chain over those copies j, ascending j, from +0 ) */
/* is the one row returned, stored in slot g*K + j0 with j0 the first such j. */
/* The origin then adds its partials in ascending r, in fp32 from +0, and     */
/* rounds to bf16 (out_bf16) or keeps fp32 (out_f32).  `partial` may be NULL. */
/* ------------------------------------------------------------------------ */
void oracle_combine_partial(const uint16_t *y, const int32_t *tok2row, const int32_t *topk_idx,
                            const float *topk_w, int T, int K, int H, int E, int R,
                            uint16_t *partial, uint16_t *out_bf16, float *out_f32)
{
    int L = E / R;
    for (int64_t g = 0; g < T; ++g) {
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int r = 0; r < R; ++r) {
                int j0 = -1;
                float part = 0.0f;
                for (int j = 0; j < K; ++j) {
                    if (topk_idx[g * K + j] / L != r) continue;
                    if (j0 < 0) j0 = j;
                    int32_t row = tok2row[g * K + j];
                    part = fmaf(topk_w[g * K + j], oracle_f32_from_bf16(y[(int64_t)row * H + h]), part);
                }
                if (j0 < 0) continue;                       /* no expert of g on rank r */
                uint16_t wire = oracle_bf16_from_f32(part);  /* the row that would travel back */
                if (partial) partial[(g * K + j0) * (int64_t)H + h] = wire;
                acc = acc + oracle_f32_from_bf16(wire);
            }
            if (out_f32) out_f32[g * H + h] = acc;
            if (out_bf16) out_bf16[g * H + h] = oracle_bf16_from_f32(acc);
        }
    }
}

/* The same weighted sum in fp64 (for error-bound checks of the fp32 one). */
void oracle_combine_f64(const uint16_t *y, const int32_t *tok2row, const float *topk_w,
                        int T, int K, int H, double *out)
{
    for (int64_t g = 0; g < T; ++g) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < K; ++j) {
                int32_t row = tok2row[g * K + j];
                acc += (double)topk_w[g * K + j] * (double)oracle_f32_from_bf16(y[(int64_t)row * H + h]);
            }
            out[g * H + h] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the format conversions (so the tests can sweep millions of */
/* values without one foreign call per value).                               */
/* ------------------------------------------------------------------------ */
void oracle_bf16_from_f32_array(const float *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f32(in[i]);
}

void oracle_e4m3_encode_array(const float *in, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(in[i]);
}

void oracle_e4m3_decode_array(const uint8_t *in, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(in[i]);
}

/* Quantise rows of bf16 values on their own (the FP8 step of dispatch,     */
/* exposed for the codec tests): q [n, H], scale [n, H/128].                 */
void oracle_quantize_rows_e4m3(const uint16_t *x, int64_t n, int H, uint8_t *q, float *scale)
{
    for (int64_t r = 0; r < n; ++r)
        quantize_row_e4m3(x + r * H, H, q + r * H, scale + r * (H / 128));
}
