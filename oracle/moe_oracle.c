/*
 * moe_oracle.c -- plain, slow CPU oracle of the single-GPU MoE layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library; it is written from the definitions on the
 * pages it cites, step by step, in the order the pages give them.
 *
 * Precision: the pages fix it.  Rows are bf16, counts are integers, the
 * expert GEMMs are int8 x int8 with integer accumulation, the dequant scales
 * are fp32, and the combine casts bf16 rows to fp32, multiplies and adds in
 * fp32 and rounds back to bf16 with round-to-nearest-even.  This file must
 * be compiled with -ffp-contract=off and without fast-math so that every
 * fp32 multiply and add is a separately rounded IEEE operation.
 *
 * Pages cited:
 *   [P1] "dispatch_combine_shmem.py" (TileLang-Ascend dispatch/combine example)
 *   [P2] "aclnnMoeDistributeCombineV4" (CANN operator documentation)
 *   [P3] "PTO MegaMoE Dispatch + Combine Fusion Example"
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   - SwiGLU halves: columns [0, N/2) of GMM1 go through SiLU and multiply
 *     columns [N/2, N) (P3 names them "up" and "gate" without a layout).
 *   - dynamic quantisation is symmetric per row: s = max|v| / 127,
 *     q = clamp(rint(v / s), -127, 127), s = 0 and q = 0 for an all-zero row.
 *   - dequant multiplies by the per-channel scale first, then the per-row one.
 *   - FFN intermediates stay fp32 (P3 stores them in half); y is bf16.
 *   - the shared-expert term is added once, unscaled, after the routed sum.
 *   - an inactive token's output is bf16(shared) if present, else +0.
 *   - triplets are (source partition, token within partition, topK slot).
 *
 * Parity pins: every function below is checked by the CPU test suite against
 * something other than itself (library restatements, closed forms,
 * brute force, invariants, and small fixtures worked by hand from the cited
 * definitions).  Where the pages leave a convention open (the readings
 * above), the pins check the oracle against that reading; the pages print no
 * value of the FFN's output to compare with.
 *
 * The threaded drivers at the end of the file add no arithmetic: they split
 * tokens or rows into contiguous slices over pthreads and call the functions
 * above on each slice.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32.  bf16 is the upper half of an IEEE binary32.          */
/* ------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even narrowing ("CAST_RINT" in P1's combine).  NaN keeps
 * its sign and becomes a quiet NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* Array forms of the two conversions, element by element (the values
 * travel as raw 32-bit words, so a signalling NaN reaches the narrowing
 * unchanged). */
void oracle_f32_to_bf16_n(int64_t n, const float *v, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(v[i]);
}

void oracle_bf16_to_f32_n(int64_t n, const uint16_t *b, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(b[i]);
}

/* ------------------------------------------------------------------ */
/* Routing: active routes, counts, prefix offsets, stable expert-major   */
/* row order, triplets and the inverse index.                            */
/* ------------------------------------------------------------------ */

/* A route (t, k) takes part when the mask lets it and its expert id names
 * an expert.  P2 (xActiveMask parameter): a 1-D mask [BS] switches a whole
 * token, a 2-D mask [BS, K] switches single routes.  Expert ids
 * ("aclnnMoeDistributeCombineV4", zeroExpertNum / copyExpertNum):
 *   [0, E)           MoE experts, each with its own FFN and rows
 *   [E, E+Z)         zero experts: their output is zero
 *   [E+Z, E+Z+C)     copy experts: their output is the unprocessed token (oriX)
 * anything else is not an expert; such routes are inactive and counted as
 * invalid. */
enum { ROUTE_OFF = 0, ROUTE_EXPERT = 1, ROUTE_ZERO = 2, ROUTE_COPY = 3, ROUTE_INVALID = 4 };

static int route_class(int64_t t, int64_t k, int64_t K, int64_t E, int64_t Z, int64_t C,
                       const int32_t *ids, int mask_kind, const uint8_t *mask)
{
    if (mask_kind == 1 && mask[t] == 0) return ROUTE_OFF;
    if (mask_kind == 2 && mask[t * K + k] == 0) return ROUTE_OFF;
    int64_t e = ids[t * K + k];
    if (e >= 0 && e < E) return ROUTE_EXPERT;
    if (e >= E && e < E + Z) return ROUTE_ZERO;
    if (e >= E + Z && e < E + Z + C) return ROUTE_COPY;
    return ROUTE_INVALID;
}

static int route_active(int64_t t, int64_t k, int64_t K, int64_t E,
                        const int32_t *ids, int mask_kind, const uint8_t *mask)
{
    return route_class(t, k, K, E, 0, 0, ids, mask_kind, mask) == ROUTE_EXPERT;
}

/*
 * oracle_route -- the dispatch bookkeeping.
 *
 * counts_pe[e][p] = number of active routes of partition p to expert e
 *   (P1 main_dispatch, "SetStatus": the per-(expert, source rank) count;
 *    P3 FrontReorder Stage: tokenPerExpert[srcRank, globalExpert]).
 * counts[e] = sum_p counts_pe[e][p], int64 (P1 "UpdateTokenNumsOut":
 *   expert_token_nums_out).
 * offsets = exclusive prefix sum of counts, offsets[E] = R.
 * recv_cum = inclusive running sum of counts_pe in (expert, partition)
 *   order, expert-major (P1 "Obtain ep_receive_count").
 * Row order: expert, then source partition, then token, then topK slot
 *   (P1 "Local data copy" walks status index local_expert*W + src_rank in
 *    increasing order and copies each source's rows in arrival order; the
 *    arrival order inside one source is the route order of the send loop).
 * route_row[t*K+k] = row of route (t, k) (P3 Memory Layout: expandedRowIdx,
 *   route -> expert-major row); -1 if inactive, -2 for a zero expert and -3
 *   for a copy expert (special experts have no rows).
 * assist[3r..3r+2] = (p, t - p*M, k) for row r (P1 send loop triplet:
 *   rank, token index local to the rank, slot k).
 * row_token[r] = t (the global token of row r).
 *
 * Returns R, the number of routed rows.  *num_invalid receives the number
 * of routes whose id names no expert (outside [0, E+Z+C)) and whose mask (if
 * any) was set.  Z zero experts and C copy experts follow the E MoE experts.
 */
int64_t oracle_route(int64_t T, int64_t P, int64_t K, int64_t E, int64_t Z, int64_t C,
                     const int32_t *ids, int mask_kind, const uint8_t *mask,
                     int64_t *counts, int32_t *offsets, int32_t *recv_cum,
                     int32_t *route_row, int32_t *assist, int32_t *row_token,
                     int64_t *num_invalid)
{
    int64_t M = T / P;
    int64_t invalid = 0;
    int64_t *counts_pe = (int64_t *)calloc((size_t)(E * P), sizeof(int64_t));

    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < K; ++k) {
            int cls = route_class(t, k, K, E, Z, C, ids, mask_kind, mask);
            if (cls == ROUTE_INVALID) invalid++;
            if (cls != ROUTE_EXPERT) continue;
            int64_t p = t / M;
            counts_pe[(int64_t)ids[t * K + k] * P + p] += 1;
        }
    }

    int64_t running = 0;
    for (int64_t e = 0; e < E; ++e) {
        int64_t c = 0;
        for (int64_t p = 0; p < P; ++p) {
            c += counts_pe[e * P + p];
            running += counts_pe[e * P + p];
            recv_cum[e * P + p] = (int32_t)running;
        }
        counts[e] = c;
    }
    int64_t acc = 0;
    for (int64_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)acc;
        acc += counts[e];
    }
    offsets[E] = (int32_t)acc;

    /* route_row codes for routes without a row: -1 inactive, -2 zero expert,
     * -3 copy expert */
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            int cls = route_class(t, k, K, E, Z, C, ids, mask_kind, mask);
            route_row[t * K + k] = cls == ROUTE_ZERO ? -2 : cls == ROUTE_COPY ? -3 : -1;
        }

    /* Emit rows in (expert, partition, token, slot) order. */
    int64_t r = 0;
    for (int64_t e = 0; e < E; ++e) {
        for (int64_t p = 0; p < P; ++p) {
            for (int64_t tl = 0; tl < M; ++tl) {
                int64_t t = p * M + tl;
                for (int64_t k = 0; k < K; ++k) {
                    if (ids[t * K + k] != e) continue;
                    if (!route_active(t, k, K, E, ids, mask_kind, mask)) continue;
                    route_row[t * K + k] = (int32_t)r;
                    assist[3 * r + 0] = (int32_t)p;
                    assist[3 * r + 1] = (int32_t)tl;
                    assist[3 * r + 2] = (int32_t)k;
                    row_token[r] = (int32_t)t;
                    r++;
                }
            }
        }
    }
    free(counts_pe);
    if (num_invalid) *num_invalid = invalid;
    return r;
}

/* expand_x[r] = x[token of row r], a bit copy of the bf16 row (P1 send loop
 * copies x[token] into the outgoing row; "Local data copy" copies it into
 * expand_x_out). */
void oracle_gather(int64_t T, int64_t H, int64_t K, const uint16_t *x,
                   const int32_t *route_row, uint16_t *expand_x)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            int32_t r = route_row[t * K + k];
            if (r < 0) continue;
            memcpy(expand_x + (int64_t)r * H, x + t * H, (size_t)H * sizeof(uint16_t));
        }
}

/* ------------------------------------------------------------------ */
/* Quantised dispatch: int8 rows with one dynamic scale per row.         */
/* ------------------------------------------------------------------ */

void oracle_quant_row(int64_t n, const float *v, int8_t *q, float *s_out);

/* The dispatch of P2's sample run with a quantisation mode ("aclnnMoe-
 * DistributeCombineV4", Example: DispatchV4 takes smooth scales [experts, H]
 * when quantMode > 0 and returns int8 expandX with dynamicScales [A]): row r
 * of token t routed to expert e holds the dynamic int8 quantisation of
 * v = float(x[t]) * smooth[e] (or of float(x[t]) when smooth is NULL), and
 * scales[r] its scale.  route_row comes from oracle_route.
 * q: int8 [rows, H]; scales: fp32 [rows]. */
void oracle_dispatch_quant(int64_t T, int64_t H, int64_t K, const uint16_t *x,
                           const int32_t *ids, const int32_t *route_row,
                           const float *smooth, int8_t *q, float *scales)
{
    float *v = (float *)malloc((size_t)H * sizeof(float));
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            int32_t r = route_row[t * K + k];
            if (r < 0) continue;
            int64_t e = ids[t * K + k];
            for (int64_t h = 0; h < H; ++h) {
                float xv = oracle_bf16_to_f32(x[t * H + h]);
                v[h] = smooth ? xv * smooth[e * H + h] : xv;
            }
            oracle_quant_row(H, v, q + (int64_t)r * H, &scales[r]);
        }
    free(v);
}

/* ------------------------------------------------------------------ */
/* Dynamic per-row int8 quantisation (P3 FrontReorder Stage writes       */
/* quantised rows with a per-row scale; SwiGLU: "dynamic quantization" */
/* -> int8 + perTokenScale).                                             */
/* ------------------------------------------------------------------ */

void oracle_quant_row(int64_t n, const float *v, int8_t *q, float *s_out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *s_out = s;
    for (int64_t i = 0; i < n; ++i) {
        if (s == 0.0f) { q[i] = 0; continue; }
        float r = rintf(v[i] / s);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

/* ------------------------------------------------------------------ */
/* One expert's FFN on one routed row (P3 "GMM1 / SwiGLU / GMM2 Stages" */
/* and the dequant of "Combine / Unpermute Stages").                     */
/* ------------------------------------------------------------------ */

float oracle_silu(float v)
{
    return v / (1.0f + expf(-v));
}

/*
 * x_row: bf16 [H]; w1: int8 [N, H] (row n = output channel n, reduction dim
 * contiguous); scale1: fp32 [N]; w2: int8 [H, N/2]; scale2: fp32 [H].
 * Any of the intermediate outputs may be NULL.  y: bf16 [H].
 *
 *   q1, s1   = quant(x_row)                       (P3 FrontReorder, offsetA)
 *   acc1[n]  = sum_h q1[h] * w1[n, h]              (GMM1, int32 accumulator)
 *   h[n]     = (float(acc1[n]) * scale1[n]) * s1   (fixpipe scale1, perTokenScale1)
 *   g[j]     = silu(h[j]) * h[j + N/2]             (SwiGLU)
 *   q2, s2   = quant(g)                            (dynamic quantization)
 *   acc2[c]  = sum_j q2[j] * w2[c, j]              (GMM2, int32 accumulator)
 *   y[c]     = bf16((float(acc2[c]) * scale2[c]) * s2)   (fixpipe scale2, perTokenScale2)
 *
 * Returns 0, or 1 if an accumulator left the int32 range.
 */
int oracle_ffn_row(int64_t H, int64_t N, const uint16_t *x_row,
                   const int8_t *w1, const float *scale1,
                   const int8_t *w2, const float *scale2,
                   int8_t *q1_out, float *s1_out, int32_t *acc1_out,
                   float *g_out, int8_t *q2_out, float *s2_out,
                   int32_t *acc2_out, uint16_t *y)
{
    int64_t Nh = N / 2;
    int overflow = 0;
    float *xf = (float *)malloc((size_t)H * sizeof(float));
    int8_t *q1 = (int8_t *)malloc((size_t)H);
    float *hbuf = (float *)malloc((size_t)N * sizeof(float));
    float *g = (float *)malloc((size_t)Nh * sizeof(float));
    int8_t *q2 = (int8_t *)malloc((size_t)Nh);
    float s1, s2;

    for (int64_t i = 0; i < H; ++i) xf[i] = oracle_bf16_to_f32(x_row[i]);
    oracle_quant_row(H, xf, q1, &s1);

    for (int64_t n = 0; n < N; ++n) {
        int64_t acc = 0;
        for (int64_t i = 0; i < H; ++i)
            acc += (int64_t)q1[i] * (int64_t)w1[n * H + i];
        if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
        if (acc1_out) acc1_out[n] = (int32_t)acc;
        float deq = (float)(int32_t)acc * scale1[n];
        hbuf[n] = deq * s1;
    }
    for (int64_t j = 0; j < Nh; ++j) {
        float a = oracle_silu(hbuf[j]);
        g[j] = a * hbuf[j + Nh];
    }
    oracle_quant_row(Nh, g, q2, &s2);
    for (int64_t c = 0; c < H; ++c) {
        int64_t acc = 0;
        for (int64_t j = 0; j < Nh; ++j)
            acc += (int64_t)q2[j] * (int64_t)w2[c * Nh + j];
        if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
        if (acc2_out) acc2_out[c] = (int32_t)acc;
        float deq = (float)(int32_t)acc * scale2[c];
        y[c] = oracle_f32_to_bf16(deq * s2);
    }
    if (q1_out) memcpy(q1_out, q1, (size_t)H);
    if (s1_out) *s1_out = s1;
    if (g_out) memcpy(g_out, g, (size_t)Nh * sizeof(float));
    if (q2_out) memcpy(q2_out, q2, (size_t)Nh);
    if (s2_out) *s2_out = s2;
    free(xf); free(q1); free(hbuf); free(g); free(q2);
    return overflow;
}

/*
 * Grouped int8 GEMM with int32 result: rows [offsets[e], offsets[e+1]) of A
 * are multiplied by expert e's weight W[e] ([N, Kd], reduction contiguous).
 * C[r, n] = sum_i A[r, i] * W[e, n, i].  Returns 1 if a sum left int32.
 * (P3 GMM1/GMM2: int8 x int8 -> int32 accumulator, per local expert.)
 */
int oracle_grouped_gemm_s32(int64_t E, int64_t N, int64_t Kd,
                            const int32_t *offsets, const int8_t *A,
                            const int8_t *W, int32_t *C)
{
    int overflow = 0;
    for (int64_t e = 0; e < E; ++e) {
        const int8_t *We = W + e * N * Kd;
        for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) {
            for (int64_t n = 0; n < N; ++n) {
                int64_t acc = 0;
                for (int64_t i = 0; i < Kd; ++i)
                    acc += (int64_t)A[r * Kd + i] * (int64_t)We[n * Kd + i];
                if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
                C[r * N + n] = (int32_t)acc;
            }
        }
    }
    return overflow;
}

/* ------------------------------------------------------------------ */
/* Combine / unpermute.                                                  */
/* ------------------------------------------------------------------ */

/*
 * out[t] = bf16_rne( sum_{k active, ascending} probs[t,k] * float(y[route_row[t,k]])
 *                    + float(shared[t]) )
 * P1 "Implement the Combine operator": for each slot k in order the bf16 row
 * is cast to fp32, multiplied by expert_scales[t, k] and added to an fp32
 * accumulator that starts at zero; the result is cast with CAST_RINT.
 * P2 Function/Formula: xOut = Sum(expertScales * ataOut) plus the shared
 * expert term, read here as added once, unscaled, after the routed sum.
 * P3 Unpermute: topK weighted accumulation back into the original order.
 * A zero-expert slot (route_row -2) contributes probs * 0 and a copy-expert
 * slot (-3) probs * oriX[t] ("aclnnMoeDistributeCombineV4", zeroExpertNum,
 * copyExpertNum, oriXOptional), in their slot position.
 * y: bf16 [rows, H]; route_row: [T*K]; probs fp32 [T, K]; shared: bf16
 * [T, H] or NULL; ori_x: bf16 [T, H] or NULL (needed if a slot is -3);
 * out: bf16 [T, H].
 */
void oracle_combine(int64_t T, int64_t H, int64_t K, const uint16_t *y,
                    const int32_t *route_row, const float *probs,
                    const uint16_t *shared, const uint16_t *ori_x, uint16_t *out)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                int32_t r = route_row[t * K + k];
                float v;
                if (r >= 0) v = oracle_bf16_to_f32(y[(int64_t)r * H + h]);
                else if (r == -2) v = 0.0f;                                  /* zero expert */
                else if (r == -3) v = oracle_bf16_to_f32(ori_x[t * H + h]);  /* copy expert */
                else continue;
                float prod = probs[t * K + k] * v;
                acc = acc + prod;
            }
            if (shared) acc = acc + oracle_bf16_to_f32(shared[t * H + h]);
            out[t * H + h] = oracle_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Whole layer, token by token (P3 Functionality:                       */
/*   out[token] = sum_topK probs[token, route] * FFN_expert(x[token])).  */
/* ------------------------------------------------------------------ */

/*
 * Computes out[t] for the listed tokens only, so a sample of a large
 * workload can be checked.  The routed sum for token t runs over its active
 * slots in k order, each expert's FFN applied to x[t]; combine rounding as
 * in oracle_combine.  w1: int8 [E, N, H]; scale1 [E, N]; w2: int8 [E, H, N/2];
 * scale2 [E, H].  out_rows: bf16 [n_tokens, H].  Returns 1 on an int32
 * overflow in any accumulator.
 */
int oracle_layer_tokens(int64_t T, int64_t H, int64_t E, int64_t Z, int64_t C,
                        int64_t K, int64_t N,
                        const uint16_t *x, const int32_t *ids, int mask_kind,
                        const uint8_t *mask, const float *probs,
                        const uint16_t *shared,
                        const int8_t *w1, const float *scale1,
                        const int8_t *w2, const float *scale2,
                        int64_t n_tokens, const int64_t *tokens,
                        uint16_t *out_rows)
{
    int overflow = 0;
    int64_t Nh = N / 2;
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    uint16_t *y = (uint16_t *)malloc((size_t)H * sizeof(uint16_t));
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens[i];
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            int cls = route_class(t, k, K, E, Z, C, ids, mask_kind, mask);
            if (cls == ROUTE_OFF || cls == ROUTE_INVALID) continue;
            if (cls == ROUTE_EXPERT) {
                int64_t e = ids[t * K + k];
                overflow |= oracle_ffn_row(H, N, x + t * H,
                                           w1 + e * N * H, scale1 + e * N,
                                           w2 + e * H * Nh, scale2 + e * H,
                                           NULL, NULL, NULL, NULL, NULL, NULL, NULL, y);
            }
            for (int64_t h = 0; h < H; ++h) {
                float v = cls == ROUTE_EXPERT ? oracle_bf16_to_f32(y[h])
                        : cls == ROUTE_COPY ? oracle_bf16_to_f32(x[t * H + h]) : 0.0f;
                float prod = probs[t * K + k] * v;
                acc[h] = acc[h] + prod;
            }
        }
        for (int64_t h = 0; h < H; ++h) {
            float a = acc[h];
            if (shared) a = a + oracle_bf16_to_f32(shared[t * H + h]);
            out_rows[i * H + h] = oracle_f32_to_bf16(a);
        }
    }
    free(acc);
    free(y);
    return overflow;
}

/* ------------------------------------------------------------------ */
/* Threaded drivers.  They add no arithmetic: each worker calls one of   */
/* the functions above, unchanged, on its own contiguous slice of tokens */
/* or rows.  Those functions treat every token and every row on its own, */
/* so the slices together give exactly the result of one call over the   */
/* whole range, whatever the number of threads.                          */
/* ------------------------------------------------------------------ */

typedef struct {
    void (*fn)(void *arg, int64_t lo, int64_t hi, int *flag);
    void *arg;
    int64_t lo, hi;
    int flag;
} oracle_slice;

static void *oracle_slice_run(void *p)
{
    oracle_slice *j = (oracle_slice *)p;
    j->fn(j->arg, j->lo, j->hi, &j->flag);
    return NULL;
}

/* Runs fn on [0, n) cut into nthreads contiguous slices; returns the OR of
 * the slices' flags.  A thread that cannot be started runs its slice here. */
static int oracle_parallel(int64_t n, int nthreads,
                           void (*fn)(void *, int64_t, int64_t, int *), void *arg)
{
    enum { MAX_THREADS = 512 };
    pthread_t tid[MAX_THREADS];
    int started[MAX_THREADS];
    oracle_slice job[MAX_THREADS];
    if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
    if (nthreads > n) nthreads = (int)n;
    if (nthreads < 1) nthreads = 1;
    for (int i = 0; i < nthreads; ++i) {
        job[i].fn = fn;
        job[i].arg = arg;
        job[i].lo = n * i / nthreads;
        job[i].hi = n * (i + 1) / nthreads;
        job[i].flag = 0;
    }
    for (int i = 1; i < nthreads; ++i)
        started[i] = pthread_create(&tid[i], NULL, oracle_slice_run, &job[i]) == 0;
    oracle_slice_run(&job[0]);
    int flag = job[0].flag;
    for (int i = 1; i < nthreads; ++i) {
        if (started[i]) pthread_join(tid[i], NULL);
        else oracle_slice_run(&job[i]);
        flag |= job[i].flag;
    }
    return flag;
}

typedef struct {
    int64_t H, K;
    const uint16_t *x;
    const int32_t *route_row;
    uint16_t *out;
} gather_args;

static void gather_slice(void *p, int64_t lo, int64_t hi, int *flag)
{
    const gather_args *a = (const gather_args *)p;
    (void)flag;
    oracle_gather(hi - lo, a->H, a->K, a->x + lo * a->H, a->route_row + lo * a->K, a->out);
}

/* oracle_gather with its tokens split over nthreads threads. */
void oracle_gather_mt(int64_t T, int64_t H, int64_t K, const uint16_t *x,
                      const int32_t *route_row, uint16_t *out, int nthreads)
{
    gather_args a = {H, K, x, route_row, out};
    oracle_parallel(T, nthreads, gather_slice, &a);
}

typedef struct {
    int64_t H, K;
    const uint16_t *y;
    const int32_t *route_row;
    const float *probs;
    const uint16_t *shared, *ori_x;
    uint16_t *out;
} combine_args;

static void combine_slice(void *p, int64_t lo, int64_t hi, int *flag)
{
    const combine_args *a = (const combine_args *)p;
    (void)flag;
    oracle_combine(hi - lo, a->H, a->K, a->y, a->route_row + lo * a->K, a->probs + lo * a->K,
                   a->shared ? a->shared + lo * a->H : NULL,
                   a->ori_x ? a->ori_x + lo * a->H : NULL, a->out + lo * a->H);
}

/* oracle_combine with its tokens split over nthreads threads. */
void oracle_combine_mt(int64_t T, int64_t H, int64_t K, const uint16_t *y,
                       const int32_t *route_row, const float *probs,
                       const uint16_t *shared, const uint16_t *ori_x, uint16_t *out,
                       int nthreads)
{
    combine_args a = {H, K, y, route_row, probs, shared, ori_x, out};
    oracle_parallel(T, nthreads, combine_slice, &a);
}

typedef struct {
    int64_t T, H, E, Z, C, K, N;
    const uint16_t *x;
    const int32_t *ids;
    int mask_kind;
    const uint8_t *mask;
    const float *probs;
    const uint16_t *shared;
    const int8_t *w1;
    const float *scale1;
    const int8_t *w2;
    const float *scale2;
    const int64_t *tokens;
    uint16_t *out_rows;
} layer_args;

static void layer_slice(void *p, int64_t lo, int64_t hi, int *flag)
{
    const layer_args *a = (const layer_args *)p;
    *flag |= oracle_layer_tokens(a->T, a->H, a->E, a->Z, a->C, a->K, a->N, a->x, a->ids,
                                 a->mask_kind, a->mask, a->probs, a->shared, a->w1, a->scale1,
                                 a->w2, a->scale2, hi - lo, a->tokens + lo,
                                 a->out_rows + lo * a->H);
}

/* oracle_layer_tokens with the token list split over nthreads threads.
 * Returns 1 on an int32 overflow in any accumulator. */
int oracle_layer_tokens_mt(int64_t T, int64_t H, int64_t E, int64_t Z, int64_t C,
                           int64_t K, int64_t N,
                           const uint16_t *x, const int32_t *ids, int mask_kind,
                           const uint8_t *mask, const float *probs,
                           const uint16_t *shared,
                           const int8_t *w1, const float *scale1,
                           const int8_t *w2, const float *scale2,
                           int64_t n_tokens, const int64_t *tokens,
                           uint16_t *out_rows, int nthreads)
{
    layer_args a = {T, H, E, Z, C, K, N, x, ids, mask_kind, mask, probs, shared,
                    w1, scale1, w2, scale2, tokens, out_rows};
    return oracle_parallel(n_tokens, nthreads, layer_slice, &a);
}

typedef struct {
    int64_t H, N;
    const uint16_t *x;
    const int64_t *token, *expert;
    const int8_t *w1;
    const float *scale1;
    const int8_t *w2;
    const float *scale2;
    int8_t *q1;
    float *s1, *g;
    int8_t *q2;
    float *s2;
    uint16_t *y;
} ffn_rows_args;

static void ffn_rows_slice(void *p, int64_t lo, int64_t hi, int *flag)
{
    const ffn_rows_args *a = (const ffn_rows_args *)p;
    const int64_t H = a->H, N = a->N, Nh = N / 2;
    for (int64_t i = lo; i < hi; ++i) {
        const int64_t t = a->token[i], e = a->expert[i];
        *flag |= oracle_ffn_row(H, N, a->x + t * H, a->w1 + e * N * H, a->scale1 + e * N,
                                a->w2 + e * H * Nh, a->scale2 + e * H,
                                a->q1 + i * H, a->s1 + i, NULL, a->g + i * Nh,
                                a->q2 + i * Nh, a->s2 + i, NULL, a->y + i * H);
    }
}

/* Every stage of the FFN for n dispatched rows: row i holds token token[i]
 * of x and runs expert expert[i]'s FFN (oracle_ffn_row).  Outputs per row:
 * q1 int8 [n, H], s1 [n], g [n, N/2], q2 int8 [n, N/2], s2 [n], y bf16
 * [n, H].  Rows are split over nthreads threads.  Returns 1 on an int32
 * overflow in any accumulator. */
int oracle_ffn_rows_mt(int64_t n, int64_t H, int64_t N, const uint16_t *x,
                       const int64_t *token, const int64_t *expert,
                       const int8_t *w1, const float *scale1,
                       const int8_t *w2, const float *scale2,
                       int8_t *q1, float *s1, float *g, int8_t *q2, float *s2,
                       uint16_t *y, int nthreads)
{
    ffn_rows_args a = {H, N, x, token, expert, w1, scale1, w2, scale2, q1, s1, g, q2, s2, y};
    return oracle_parallel(n, nthreads, ffn_rows_slice, &a);
}
