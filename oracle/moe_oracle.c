/*
 * moe_oracle.c -- CPU oracle for the W4A16 group-32 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; it is a plain, slow, obviously correct restatement
 * of what the layer computes, in IEEE double precision, single-threaded.
 *
 * What the layer is.  "[Perf][SM70] Narrow Qwen3.8 AWQ active grouped decode",
 * section Purpose, names the geometry (512 experts, top-k 10, hidden 2560,
 * AWQ W4A16 with groups of 32, local intermediate 160 under TP4) and the
 * structure of the hot path (multi-row active-expert segments scheduled by
 * offsets).  "[Model][SM70] Adapt Qwen3.8 Flash Next NVFP4", section
 * Implemented route, gives the full geometry (2560, 640, 512, top-10).  The
 * pages never write the arithmetic down; every function below states the
 * standard definition it follows, and where a choice had to be made (packing
 * order, tie rule, renormalisation) the reading is stated at that function.
 *
 * Layouts (all row-major, little-endian words):
 *   logits  f32 [T][E]
 *   x       binary16 [T][H]
 *   W13     qweight u32 [E][2I][H/8]  -- rows [0,I) gate, rows [I,2I) up
 *           scales  binary16 [E][2I][H/32]
 *           qzeros  u32 [E][2I/8][H/32]
 *   W2      qweight u32 [E][H][I/8], scales binary16 [E][H][I/32],
 *           qzeros u32 [E][H/8][I/32]
 *   For a weight matrix W[N][K] of one expert: element (n, kk) has
 *     q = bits [4*(kk%8), 4*(kk%8)+4) of qweight[n][kk/8]
 *     z = bits [4*(n%8),  4*(n%8)+4)  of qzeros[n/8][kk/32]
 *     s = scales[n][kk/32]
 *     w = (q - z) * s
 *   A pair is p = t*k + j: token t's j-th selected expert.
 *
 * Second weight format (NVFP4 weights, fp16 activations).  "[Model][SM70]
 * Adapt Qwen3.8 Flash Next NVFP4", section Implemented route, runs the
 * checkpoint's ModelOpt NVFP4 routed experts through the W4A16 kernel with
 * fp16 activations; the page does not restate the format, so the functions
 * *_nvfp4 below follow its public definition: 4-bit E2M1 values, one FP8
 * E4M3 scale per 16 consecutive elements along K, one fp32 scale per
 * expert matrix.  Layout for one expert's W[N][K]:
 *     codes  u32 [E][N][K/8]   value of (n, kk) = E2M1 nibble 4*(kk%8) of word [n][kk/8]
 *     bscale u8  [E][N][K/16]  E4M3 scale of (n, kk) = bscale[n][kk/16]
 *     gscale f32 [E]           per-expert scale
 *     w = e2m1(code) * e4m3(bscale) * gscale
 *
 * Parity status: every function here is pinned by the CPU test suite against
 * brute force, closed forms and invariants (see tests/test_oracle_pins.py
 * and tests/test_oracle_nvfp4.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

ORACLE_API int oracle_abi_version(void) { return 1; }

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is subnormal
 * (fraction * 2^-24), exponent 31 is inf/NaN. */
ORACLE_API double oracle_half_to_double(uint16_t h)
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

/* Dequantised weight w = (q - z) * s of element (n, kk) of expert e's
 * matrix W[N][K], per the AWQ-style group-32 scheme ("effective g32",
 * Purpose section of the grouped-decode page). */
ORACLE_API double oracle_dequant(const uint32_t *qweight, const uint16_t *scales,
                                 const uint32_t *qzeros, int N, int K,
                                 int e, int n, int kk)
{
    size_t G = (size_t)K / 32;
    size_t qword = ((size_t)e * N + n) * (K / 8) + kk / 8;
    int q = (int)((qweight[qword] >> (4 * (kk % 8))) & 0xfu);
    size_t zword = ((size_t)e * (N / 8) + n / 8) * G + kk / 32;
    int z = (int)((qzeros[zword] >> (4 * (n % 8))) & 0xfu);
    double s = oracle_half_to_double(scales[((size_t)e * N + n) * G + kk / 32]);
    return (double)(q - z) * s;
}

/* "a is ranked before b": larger logit first; equal logits go to the lower
 * expert index.  The decision is taken on the fp32 logits as given, the
 * same values the device compares. */
static int ranks_before(float la, int a, float lb, int b)
{
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b;
}

/* Router: softmax over all E logits, the k most probable experts, and their
 * probabilities renormalised to sum to one.  Softmax is strictly increasing
 * in the logit, so ranking by probability is ranking by logit; the ranking
 * uses the logits.  Output order within a token is the ranking order.
 * topk_ids [T][k], topk_w [T][k]. */
ORACLE_API void oracle_route(const float *logits, int T, int E, int k,
                             int32_t *topk_ids, double *topk_w)
{
    double *prob = (double *)malloc(sizeof(double) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        /* full softmax, max-subtracted for range safety */
        double m = -INFINITY;
        for (int e = 0; e < E; ++e)
            if ((double)l[e] > m) m = (double)l[e];
        double denom = 0.0;
        for (int e = 0; e < E; ++e) {
            prob[e] = exp((double)l[e] - m);
            denom += prob[e];
        }
        for (int e = 0; e < E; ++e) prob[e] /= denom;
        /* k rounds of "best not yet taken" */
        memset(taken, 0, (size_t)E);
        double selected_mass = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            topk_ids[(size_t)t * k + j] = best;
            selected_mass += prob[best];
        }
        for (int j = 0; j < k; ++j) {
            int e = topk_ids[(size_t)t * k + j];
            topk_w[(size_t)t * k + j] = prob[e] / selected_mass;
        }
    }
    free(prob);
    free(taken);
}

/* Active-expert segments ("multi-row active-expert segments and
 * offsets-based scheduling", Purpose section of the grouped-decode page).
 * Pairs are grouped by expert, experts in ascending id, pairs in ascending
 * pair id inside a segment, with no padding.
 *   expert_offsets [E+1]: segment of expert e is [offsets[e], offsets[e+1])
 *   sorted_pair    [T*k]: pair ids in segment order
 *   active_experts [E]  : experts with a non-empty segment, ascending;
 *                         entries past num_active are -1
 *   num_active     [1]  */
ORACLE_API void oracle_align(const int32_t *topk_ids, int T, int E, int k,
                             int32_t *expert_offsets, int32_t *sorted_pair,
                             int32_t *active_experts, int32_t *num_active)
{
    int P = T * k;
    int pos = 0, na = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = pos;
        for (int p = 0; p < P; ++p)
            if (topk_ids[p] == e) sorted_pair[pos++] = p;
        if (pos > expert_offsets[e]) active_experts[na++] = e;
    }
    expert_offsets[E] = pos;
    for (int a = na; a < E; ++a) active_experts[a] = -1;
    num_active[0] = na;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* Gate/up projection of one token row through expert e, fused with SiLU*up:
 * g_i = sum_K x[K] * W13[i][K], u_i = sum_K x[K] * W13[I+i][K],
 * h_i = silu(g_i) * u_i, for i in [0, I).  Sums run in K order. */
static void expert_gate_up(const uint16_t *xrow, int H, int I,
                           const uint32_t *w13q, const uint16_t *w13s,
                           const uint32_t *w13z, int e, double *hrow)
{
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int kk = 0; kk < H; ++kk) {
            double xv = oracle_half_to_double(xrow[kk]);
            g += xv * oracle_dequant(w13q, w13s, w13z, 2 * I, H, e, i, kk);
            u += xv * oracle_dequant(w13q, w13s, w13z, 2 * I, H, e, I + i, kk);
        }
        hrow[i] = silu(g) * u;
    }
}

/* Down projection of one intermediate row through expert e:
 * y_n = sum_i h[i] * W2[n][i], for n in [0, H).  Sums run in i order. */
static void expert_down(const double *hrow, int H, int I,
                        const uint32_t *w2q, const uint16_t *w2s,
                        const uint32_t *w2z, int e, double *yrow)
{
    for (int n = 0; n < H; ++n) {
        double y = 0.0;
        for (int i = 0; i < I; ++i)
            y += hrow[i] * oracle_dequant(w2q, w2s, w2z, H, I, e, n, i);
        yrow[n] = y;
    }
}

/* Step 3 over the grouped layout: for every active expert and every pair of
 * its segment, h[r] = silu(x_t W_gate^T) * (x_t W_up^T), where r is the
 * pair's position in sorted order and t = pair / k.  h is [T*k][I]. */
ORACLE_API void oracle_gate_up_silu(const uint16_t *x, int T, int H, int I, int k,
                                    const uint32_t *w13q, const uint16_t *w13s,
                                    const uint32_t *w13z,
                                    const int32_t *expert_offsets,
                                    const int32_t *sorted_pair,
                                    const int32_t *active_experts,
                                    const int32_t *num_active, double *h)
{
    (void)T;
    for (int a = 0; a < num_active[0]; ++a) {
        int e = active_experts[a];
        for (int r = expert_offsets[e]; r < expert_offsets[e + 1]; ++r) {
            int t = sorted_pair[r] / k;
            expert_gate_up(x + (size_t)t * H, H, I, w13q, w13s, w13z, e,
                           h + (size_t)r * I);
        }
    }
}

/* Step 4 over the grouped layout: y[r] = h[r] W_down^T for every sorted row
 * r, then out[t] = sum_j topk_w[t][j] * y[row of pair t*k+j], summed in j
 * order.  out is [T][H]. */
ORACLE_API void oracle_down_combine(const double *h, int T, int H, int I, int k,
                                    const uint32_t *w2q, const uint16_t *w2s,
                                    const uint32_t *w2z,
                                    const int32_t *expert_offsets,
                                    const int32_t *sorted_pair,
                                    const int32_t *active_experts,
                                    const int32_t *num_active,
                                    const double *topk_w, double *out)
{
    int P = T * k;
    double *y = (double *)malloc(sizeof(double) * (size_t)P * H);
    int *row_of_pair = (int *)malloc(sizeof(int) * (size_t)P);
    for (int a = 0; a < num_active[0]; ++a) {
        int e = active_experts[a];
        for (int r = expert_offsets[e]; r < expert_offsets[e + 1]; ++r) {
            expert_down(h + (size_t)r * I, H, I, w2q, w2s, w2z, e, y + (size_t)r * H);
            row_of_pair[sorted_pair[r]] = r;
        }
    }
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int r = row_of_pair[t * k + j];
                acc += topk_w[(size_t)t * k + j] * y[(size_t)r * H + n];
            }
            out[(size_t)t * H + n] = acc;
        }
    free(y);
    free(row_of_pair);
}

/* The whole layer for a single token, straight from the definition of a
 * routed MoE layer: out_t = sum_j w_j * FFN_{e_j}(x_t), with FFN_e(x) =
 * W_down,e (silu(W_gate,e x) * (W_up,e x)).  No grouping, no offsets: it is
 * what the grouped steps must add up to, and it lets large workloads be
 * checked on sampled tokens.  out_row is [H]. */
ORACLE_API void oracle_moe_token(int t, const float *logits, const uint16_t *x,
                                 int E, int k, int H, int I,
                                 const uint32_t *w13q, const uint16_t *w13s,
                                 const uint32_t *w13z,
                                 const uint32_t *w2q, const uint16_t *w2s,
                                 const uint32_t *w2z, double *out_row)
{
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    double *w = (double *)malloc(sizeof(double) * (size_t)k);
    double *hrow = (double *)malloc(sizeof(double) * (size_t)I);
    double *yrow = (double *)malloc(sizeof(double) * (size_t)H);
    oracle_route(logits + (size_t)t * E, 1, E, k, ids, w);
    for (int n = 0; n < H; ++n) out_row[n] = 0.0;
    for (int j = 0; j < k; ++j) {
        expert_gate_up(x + (size_t)t * H, H, I, w13q, w13s, w13z, ids[j], hrow);
        expert_down(hrow, H, I, w2q, w2s, w2z, ids[j], yrow);
        for (int n = 0; n < H; ++n) out_row[n] += w[j] * yrow[n];
    }
    free(ids);
    free(w);
    free(hrow);
    free(yrow);
}

/* The four steps in order over a whole batch.  Every output buffer is
 * caller-owned: topk_ids/topk_w [T][k], expert_offsets [E+1],
 * sorted_pair [T*k], active_experts [E], num_active [1], h [T*k][I],
 * out [T][H]. */
ORACLE_API void oracle_moe_forward(const float *logits, const uint16_t *x,
                                   int T, int E, int k, int H, int I,
                                   const uint32_t *w13q, const uint16_t *w13s,
                                   const uint32_t *w13z,
                                   const uint32_t *w2q, const uint16_t *w2s,
                                   const uint32_t *w2z,
                                   int32_t *topk_ids, double *topk_w,
                                   int32_t *expert_offsets, int32_t *sorted_pair,
                                   int32_t *active_experts, int32_t *num_active,
                                   double *h, double *out)
{
    oracle_route(logits, T, E, k, topk_ids, topk_w);
    oracle_align(topk_ids, T, E, k, expert_offsets, sorted_pair, active_experts,
                 num_active);
    oracle_gate_up_silu(x, T, H, I, k, w13q, w13s, w13z, expert_offsets,
                        sorted_pair, active_experts, num_active, h);
    oracle_down_combine(h, T, H, I, k, w2q, w2s, w2z, expert_offsets,
                        sorted_pair, active_experts, num_active, topk_w, out);
}


/* ---------------------------------------------------------------- NVFP4 */

/* E2M1 (4 bits: sign, 2 exponent bits with bias 1, 1 mantissa bit) ->
 * double, from the format's definition: exponent 0 is subnormal
 * (mantissa * 2^-1 * 2^(1-1)); otherwise 2^(exp-1) * (1 + mantissa/2).  No
 * infinities or NaN. */
ORACLE_API double oracle_e2m1_to_double(uint8_t nib)
{
    int sign = (nib >> 3) & 1;
    int expo = (nib >> 1) & 3;
    int mant = nib & 1;
    double v = expo == 0 ? 0.5 * mant : ldexp(1.0 + 0.5 * mant, expo - 1);
    return sign ? -v : v;
}

/* FP8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits, the
 * variant without infinities) -> double: exponent 0 is subnormal
 * (mantissa/8 * 2^-6); the all-ones exponent with all-ones mantissa is NaN;
 * otherwise 2^(exp-7) * (1 + mantissa/8). */
ORACLE_API double oracle_e4m3_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 15;
    int mant = b & 7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant / 8.0, -6);
    else
        v = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -v : v;
}

/* Dequantised NVFP4 weight of element (n, kk) of expert e's W[N][K]. */
ORACLE_API double oracle_dequant_nvfp4(const uint32_t *codes, const uint8_t *bscale,
                                       const float *gscale, int N, int K,
                                       int e, int n, int kk)
{
    size_t word = ((size_t)e * N + n) * (K / 8) + kk / 8;
    uint8_t nib = (uint8_t)((codes[word] >> (4 * (kk % 8))) & 0xfu);
    double bs = oracle_e4m3_to_double(bscale[((size_t)e * N + n) * (K / 16) + kk / 16]);
    return oracle_e2m1_to_double(nib) * bs * (double)gscale[e];
}

static void expert_gate_up_nvfp4(const uint16_t *xrow, int H, int I,
                                 const uint32_t *c13, const uint8_t *b13,
                                 const float *g13, int e, double *hrow)
{
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            double xv = oracle_half_to_double(xrow[c]);
            g += xv * oracle_dequant_nvfp4(c13, b13, g13, 2 * I, H, e, i, c);
            u += xv * oracle_dequant_nvfp4(c13, b13, g13, 2 * I, H, e, I + i, c);
        }
        hrow[i] = u * silu(g);
    }
}

static void expert_down_nvfp4(const double *hrow, int H, int I,
                              const uint32_t *c2, const uint8_t *b2,
                              const float *g2, int e, double *yrow)
{
    for (int n = 0; n < H; ++n) {
        double y = 0.0;
        for (int i = 0; i < I; ++i)
            y += hrow[i] * oracle_dequant_nvfp4(c2, b2, g2, H, I, e, n, i);
        yrow[n] = y;
    }
}

/* Step 3 with NVFP4 weights (as oracle_gate_up_silu). */
ORACLE_API void oracle_gate_up_silu_nvfp4(const uint16_t *x, int T, int H, int I, int k,
                                          const uint32_t *c13, const uint8_t *b13,
                                          const float *g13,
                                          const int32_t *expert_offsets,
                                          const int32_t *sorted_pair,
                                          const int32_t *active_experts,
                                          const int32_t *num_active, double *h)
{
    (void)T;
    for (int a = 0; a < num_active[0]; ++a) {
        int e = active_experts[a];
        for (int r = expert_offsets[e]; r < expert_offsets[e + 1]; ++r) {
            int t = sorted_pair[r] / k;
            expert_gate_up_nvfp4(x + (size_t)t * H, H, I, c13, b13, g13, e,
                                 h + (size_t)r * I);
        }
    }
}

/* The layer for a single token with NVFP4 weights (as oracle_moe_token). */
ORACLE_API void oracle_moe_token_nvfp4(int t, const float *logits, const uint16_t *x,
                                       int E, int k, int H, int I,
                                       const uint32_t *c13, const uint8_t *b13,
                                       const float *g13,
                                       const uint32_t *c2, const uint8_t *b2,
                                       const float *g2, double *out_row)
{
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    double *w = (double *)malloc(sizeof(double) * (size_t)k);
    double *hrow = (double *)malloc(sizeof(double) * (size_t)I);
    double *yrow = (double *)malloc(sizeof(double) * (size_t)H);
    oracle_route(logits + (size_t)t * E, 1, E, k, ids, w);
    for (int n = 0; n < H; ++n) out_row[n] = 0.0;
    for (int j = 0; j < k; ++j) {
        expert_gate_up_nvfp4(x + (size_t)t * H, H, I, c13, b13, g13, ids[j], hrow);
        expert_down_nvfp4(hrow, H, I, c2, b2, g2, ids[j], yrow);
        for (int n = 0; n < H; ++n) out_row[n] += w[j] * yrow[n];
    }
    free(ids);
    free(w);
    free(hrow);
    free(yrow);
}

/* The four steps over a batch with NVFP4 weights (as oracle_moe_forward):
 * routing and grouping are those of the W4A16 layer; steps 3 and 4 read
 * the NVFP4 matrices. */
ORACLE_API void oracle_moe_forward_nvfp4(const float *logits, const uint16_t *x,
                                         int T, int E, int k, int H, int I,
                                         const uint32_t *c13, const uint8_t *b13,
                                         const float *g13,
                                         const uint32_t *c2, const uint8_t *b2,
                                         const float *g2,
                                         int32_t *topk_ids, double *topk_w,
                                         int32_t *expert_offsets, int32_t *sorted_pair,
                                         int32_t *active_experts, int32_t *num_active,
                                         double *h, double *out)
{
    int P = T * k;
    oracle_route(logits, T, E, k, topk_ids, topk_w);
    oracle_align(topk_ids, T, E, k, expert_offsets, sorted_pair, active_experts,
                 num_active);
    oracle_gate_up_silu_nvfp4(x, T, H, I, k, c13, b13, g13, expert_offsets,
                              sorted_pair, active_experts, num_active, h);
    double *y = (double *)malloc(sizeof(double) * (size_t)P * H);
    int *row_of_pair = (int *)malloc(sizeof(int) * (size_t)P);
    for (int a = 0; a < num_active[0]; ++a) {
        int e = active_experts[a];
        for (int r = expert_offsets[e]; r < expert_offsets[e + 1]; ++r) {
            expert_down_nvfp4(h + (size_t)r * I, H, I, c2, b2, g2, e, y + (size_t)r * H);
            row_of_pair[sorted_pair[r]] = r;
        }
    }
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += topk_w[(size_t)t * k + j] * y[(size_t)row_of_pair[t * k + j] * H + n];
            out[(size_t)t * H + n] = acc;
        }
    free(y);
    free(row_of_pair);
}

/* ---------------------------------------------------------------- router logits
 * The step ahead of routing.  The pages treat the router's fp32 logits as
 * given; the model's gate is a bias-free linear map from the hidden state to
 * one score per expert, so
 *     logits[t][e] = sum over h of x[t][h] * wr[e][h]
 * with x binary16 [T][H] and the router matrix wr binary16 [E][H] (one row
 * per expert, the layout of a linear layer's weight), evaluated in double. */
ORACLE_API void oracle_router_logits(const uint16_t *x, const uint16_t *wr,
                                     int T, int E, int H, double *logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += oracle_half_to_double(x[(size_t)t * H + c]) *
                       oracle_half_to_double(wr[(size_t)e * H + c]);
            logits[(size_t)t * E + e] = acc;
        }
}

/* ---------------------------------------------------------------- AWQ import
 * The grouped-decode work reads AWQ g32 checkpoints ("[Model][SM70] Support
 * Qwen3.8 Flash Next with PLE offload", section Purpose, names the AWQ g32
 * metadata adapter).  The pages do not restate the checkpoint layout; these
 * functions follow the public AWQ "GEMM" packing of one linear layer with
 * input size K and output size N:
 *     qweight u32  [K][N/8]    nibble i of word [kk][c] is q of output column 8c + ORDER[i]
 *     qzeros  u32  [K/32][N/8] nibble i of word [g][c]  is z of output column 8c + ORDER[i]
 *     scales  f16  [K/32][N]
 *     ORDER = (0, 2, 4, 6, 1, 3, 5, 7), w = (q - z) * s as in the layer.
 * Experts are stacked along a leading E axis.  The import writes the same
 * (q, z, s) into the layer's layout (header of this file) at rows
 * [row0, row0 + N) of a destination with Ndst rows per expert, so that the
 * gate and up layers of an expert land in the two halves of W13. */
static const int awq_column_of_nibble[8] = {0, 2, 4, 6, 1, 3, 5, 7};

/* The nibble slot (0..7) of a word that holds output column n. */
static int awq_slot_of_column(int n)
{
    for (int i = 0; i < 8; ++i)
        if (awq_column_of_nibble[i] == n % 8) return i;
    return -1;
}

ORACLE_API int oracle_awq_q(const uint32_t *aq, int K, int N, int e, int n, int kk)
{
    uint32_t w = aq[((size_t)e * K + kk) * (N / 8) + n / 8];
    return (int)((w >> (4 * awq_slot_of_column(n))) & 0xfu);
}

ORACLE_API int oracle_awq_z(const uint32_t *az, int K, int N, int e, int n, int kk)
{
    uint32_t w = az[((size_t)e * (K / 32) + kk / 32) * (N / 8) + n / 8];
    return (int)((w >> (4 * awq_slot_of_column(n))) & 0xfu);
}

ORACLE_API uint16_t oracle_awq_s(const uint16_t *as, int K, int N, int e, int n, int kk)
{
    return as[((size_t)e * (K / 32) + kk / 32) * N + n];
}

static void put_nibble(uint32_t *word, int slot, int v)
{
    *word = (*word & ~(0xfu << (4 * slot))) | ((uint32_t)v << (4 * slot));
}

/* Element by element: every (e, n, kk) of the AWQ matrices is read with the
 * accessors above and written to its place in the layer's layout. */
ORACLE_API void oracle_awq_import(const uint32_t *aq, const uint32_t *az, const uint16_t *as,
                                  int E, int K, int N, uint32_t *qweight, uint16_t *scales,
                                  uint32_t *qzeros, int Ndst, int row0)
{
    for (int e = 0; e < E; ++e)
        for (int n = 0; n < N; ++n) {
            int r = row0 + n;
            for (int kk = 0; kk < K; ++kk) {
                put_nibble(&qweight[((size_t)e * Ndst + r) * (K / 8) + kk / 8], kk % 8,
                           oracle_awq_q(aq, K, N, e, n, kk));
                put_nibble(&qzeros[((size_t)e * (Ndst / 8) + r / 8) * (K / 32) + kk / 32], r % 8,
                           oracle_awq_z(az, K, N, e, n, kk));
                scales[((size_t)e * Ndst + r) * (K / 32) + kk / 32] = oracle_awq_s(as, K, N, e, n, kk);
            }
        }
}
