/*
 * CPU oracle of the MXFP4 routed-expert MoE layer.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package's smoke() check and bench.py's cpu_baseline
 * (and --impl reference) leg may load or call this library.  The CUDA path
 * never links, loads or calls it, and the two share no code, header, table or
 * constant.
 *
 * Plain, slow, single-threaded C.  Floating point is fp64 wherever the pages
 * leave the precision free; fp32 exactly where a floating-point result decides
 * an integer (the Q8 codes, the router logits that decide the top-k), so that
 * the CUDA path can be held to those integers bit for bit.
 *
 * Sources (web pages on the DeepSeek-V4-Flash MXFP4 expert layer):
 *  [SH]  "Optimizing DeepSeek V4 Flash Inference on a Strix Halo Pair: An
 *        Engineering Record" -- sections "MXFP4 routed-expert kernels",
 *        "MXFP4 prefill tile vectorization", "The exact-rows contract".
 *  [GFX] "DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
 *        Performance Engineering" -- Execution structure and Fig. 1, §5.3
 *        (E8M0 scale layout, deterministic index selection), §6.1 (TP4/EP1
 *        decode route), §7.1 (sorter), §8.2 (down-consumer pilot), Table 4.
 *  [LB]  "feat(ds4): add concurrent serving on Strix Halo and R9700 + Strix"
 *        (Luce-Org/lucebox PR #598) -- "Reduce expert-route overhead".
 *
 * Readings where the pages are silent are marked READING.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* E2M1 code -> real value.  [GFX] §6.1 maps each FP4 nibble to
 * 0, ±1, ±2, ±3, ±4, ±6, ±8, ±12, i.e. twice the E2M1 values
 * {0, .5, 1, 1.5, 2, 3, 4, 6}.  READING: the bit encoding is the OCP MX one
 * (bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa; exponent 0 is
 * subnormal 0.5*m).  Code 8 is -0. */
double moe_oracle_e2m1(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E8M0 scale byte -> 2^(u-127); byte 255 is NaN.  [GFX] §6.1 ("E8M0
 * scaling"), one byte per 32 weights. */
double moe_oracle_e8m0(int u)
{
    return u == 255 ? NAN : ldexp(1.0, u - 127);
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float load_elem(const void *p, int is_bf16, int64_t i)
{
    return is_bf16 ? bf16_to_f32(((const uint16_t *)p)[i]) : ((const float *)p)[i];
}

/* ------------------------------------------------------------------ router */

/* Router logit l[t,e] = x_t . Wr_e in fp32.  The pages do not state the
 * router arithmetic ([GFX] Fig. 1 "Router Top-6").  READING: the logit is the
 * fp32 result of one fixed summation order, so that the selection it decides
 * is reproducible bit for bit: the H inputs are cut into chunks of 8
 * consecutive elements; chunk c feeds partial sum c mod 32; each partial sum
 * takes its chunks in increasing order and its elements in increasing order,
 * one fused multiply-add each; the 32 partial sums are then added pairwise,
 * p[l] += p[l+s] for s = 16, 8, 4, 2, 1, and l = p[0].  (A bf16 x bf16
 * product is exact in fp32, so for bf16 inputs the fused and unfused forms
 * agree.)  Requires H % 8 == 0. */
void moe_oracle_router_logits(const void *x, int x_bf16, int64_t ld_x,
                              const void *wr, int wr_bf16,
                              int T, int H, int E, float *logits)
{
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float p[32];
            for (int l = 0; l < 32; ++l) p[l] = 0.0f;
            for (int c = 0; c < H / 8; ++c) {
                int lane = c % 32;
                for (int j = 0; j < 8; ++j) {
                    int64_t kk = 8 * (int64_t)c + j;
                    float xv = load_elem(x, x_bf16, (int64_t)t * ld_x + kk);
                    float wv = load_elem(wr, wr_bf16, (int64_t)e * H + kk);
                    p[lane] = fmaf(xv, wv, p[lane]);
                }
            }
            for (int s = 16; s >= 1; s /= 2)
                for (int l = 0; l < s; ++l) p[l] = p[l] + p[l + s];
            logits[(int64_t)t * E + e] = p[0];
        }
    }
}

/* Top-k of E by score = logit (+ bias[e]), fp32 add.  [GFX] §5.3:
 * "deterministic index selection fixes membership ties using logical IDs and
 * presents selected positions in a fixed order".  READING: ties go to the
 * lower expert id; slots are ordered by descending score.  Weights are the
 * sigmoid of the selected scores renormalised to sum 1 (the tiny-layer
 * workload's "sigmoid scores, top-k renormalised"), computed in fp64.
 * READING (the pages say nothing of non-finite scores): a NaN score is never
 * selected, since it names no ordering; a slot for which only NaN scores are
 * left gets the id MOE_ORACLE_NO_EXPERT (0x7fffffff, an id no layer has) and
 * the score -inf, so its sigmoid, and its weight, is 0.  An infinite score is
 * an ordinary score (+inf first, -inf last, weight 0 for -inf). */
#define MOE_ORACLE_NO_EXPERT 0x7fffffff

void moe_oracle_topk(const float *logits, const float *bias, int T, int E, int k,
                     int32_t *ids, double *w)
{
    float *score = (float *)malloc(sizeof(float) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float s = logits[(int64_t)t * E + e];
            score[e] = bias ? s + bias[e] : s;
            taken[e] = 0;
        }
        double sig[64];
        double total = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e] || isnan(score[e])) continue;
                if (best < 0 || score[e] > score[best]) best = e; /* strict: lower id keeps ties */
            }
            double s;
            if (best < 0) {
                ids[(int64_t)t * k + j] = MOE_ORACLE_NO_EXPERT;
                s = -INFINITY;
            } else {
                taken[best] = 1;
                ids[(int64_t)t * k + j] = best;
                s = (double)score[best];
            }
            sig[j] = 1.0 / (1.0 + exp(-s));
            total += sig[j];
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = sig[j] / total;
    }
    free(score);
    free(taken);
}

/* ------------------------------------------------------------------ sorter */

/* Group the A = T*k assignments a = t*k + j by expert.  [GFX] §7.1 item 8
 * (expert sorter with row blocks of 32 or 64).  Stable: within one expert the
 * assignments keep increasing a.  Each expert's segment is padded to a
 * multiple of tile_rows with -1, the negative sentinel of [LB] "Reduce
 * expert-route overhead".  offsets[E+1] are segment starts; inv[a] is the
 * position of a.  Returns offsets[E], or -1 (bad id) / -2 (cap too small). */
int64_t moe_oracle_sort(const int32_t *ids, int T, int k, int E, int tile_rows,
                        int32_t *offsets, int32_t *sorted, int64_t cap, int32_t *inv)
{
    int64_t A = (int64_t)T * k;
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    for (int64_t a = 0; a < A; ++a) {
        if (ids[a] < 0 || ids[a] >= E) { free(count); return -1; }
        count[ids[a]]++;
    }
    int64_t pos = 0;
    for (int e = 0; e < E; ++e) {
        offsets[e] = (int32_t)pos;
        pos += (count[e] + tile_rows - 1) / tile_rows * tile_rows;
    }
    offsets[E] = (int32_t)pos;
    if (pos > cap) { free(count); return -2; }
    for (int64_t i = 0; i < pos; ++i) sorted[i] = -1;
    for (int e = 0; e < E; ++e) count[e] = 0;
    for (int64_t a = 0; a < A; ++a) {
        int e = ids[a];
        int64_t p = offsets[e] + count[e]++;
        sorted[p] = (int32_t)a;
        inv[a] = (int32_t)p;
    }
    free(count);
    return pos;
}

/* ------------------------------------------------------------------ Q8 */

/* Per row, per block of 32: amax = max|x|, d = amax / 127, codes
 * q = round(x * (1/d)) clamped to [-127, 127]; d = 0 gives q = 0.
 * [GFX] §6.1 "online BF16 activation quantization to INT8 per 32 elements";
 * [GFX] §8.2 "forms group32 INT8 values/scales".  READING: fp32 throughout,
 * IEEE division for d and for the reciprocal, round to nearest even. */
void moe_oracle_quant_q8(const void *x, int x_bf16, int rows, int cols, int64_t ld_x,
                         int8_t *q, int64_t ld_q, float *d, int64_t ld_d)
{
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < cols / 32; ++b) {
            float v[32];
            float amax = 0.0f;
            for (int l = 0; l < 32; ++l) {
                v[l] = load_elem(x, x_bf16, (int64_t)r * ld_x + 32 * b + l);
                float a = fabsf(v[l]);
                if (a > amax) amax = a;
            }
            float dd = amax / 127.0f;
            float inv = dd > 0.0f ? 1.0f / dd : 0.0f;
            for (int l = 0; l < 32; ++l) {
                float s = nearbyintf(v[l] * inv);
                if (s > 127.0f) s = 127.0f;
                if (s < -127.0f) s = -127.0f;
                q[(int64_t)r * ld_q + 32 * b + l] = (int8_t)s;
            }
            d[(int64_t)r * ld_d + b] = dd;
        }
    }
}

/* ------------------------------------------------------------------ MX dots */

/* Twice the E2M1 value of a nibble, an exact small integer; the 16 values
 * are taken once from moe_oracle_e2m1. */
static int e2m1_twice(int code)
{
    static int table[16];
    static int ready = 0;
    if (!ready) {
        for (int c = 0; c < 16; ++c) table[c] = (int)lround(2.0 * moe_oracle_e2m1(c));
        ready = 1;
    }
    return table[code];
}

/* Exact integer block dot I = sum_{l<32} q_l * 2*e2m1(c_l) over one 32-element
 * block; byte i of the 16 packed bytes holds element 2i in its low nibble and
 * 2i+1 in its high nibble (READING: OCP MX / float4_e2m1fn_x2 order).
 * [GFX] §6.1 "v_dot4_i32_i8 / mixed-dot accumulation". */
int32_t moe_oracle_block_dot(const int8_t *q, const uint8_t *nib)
{
    int64_t acc = 0;
    for (int l = 0; l < 32; ++l) {
        int code = (l & 1) ? (nib[l / 2] >> 4) : (nib[l / 2] & 15);
        acc += (int64_t)q[l] * e2m1_twice(code);
    }
    return (int32_t)acc;
}

/* One output of an MXFP4 projection against a Q8 row, in fp64:
 * y = sum_b I_b * d_b * 2^(u_b - 128), the integer block dot "followed by
 * activation and E8M0 scaling" ([GFX] §6.1).  2^(u-128) is the E8M0 factor
 * 2^(u-127) halved, because I_b counts twice the E2M1 values. */
static double mx_dot(const int8_t *q, const float *d, const uint8_t *wrow,
                     const uint8_t *srow, int K)
{
    double acc = 0.0;
    for (int b = 0; b < K / 32; ++b) {
        int32_t I = moe_oracle_block_dot(q + 32 * b, wrow + 16 * b);
        double ws = 0.5 * moe_oracle_e8m0(srow[b]);
        acc += (double)I * (double)d[b] * ws;
    }
    return acc;
}

/* silu(g) = g * sigmoid(g), fp64.  [GFX] Fig. 1 / [LB] "folds SwiGLU into
 * its second projection pass": h = silu(gate) * up. */
double moe_oracle_silu(double g)
{
    return g / (1.0 + exp(-g));
}

/* Gate/up of one Q8 row through one expert: G[i], U[i] for i < I.
 * wg, wu [I, H/2] packed, sg, su [I, H/32] E8M0. */
void moe_oracle_expert_gateup(const int8_t *xq, const float *xs,
                              const uint8_t *wg, const uint8_t *sg,
                              const uint8_t *wu, const uint8_t *su,
                              int H, int I, double *G, double *U)
{
    for (int i = 0; i < I; ++i) {
        G[i] = mx_dot(xq, xs, wg + (int64_t)i * (H / 2), sg + (int64_t)i * (H / 32), H);
        U[i] = mx_dot(xq, xs, wu + (int64_t)i * (H / 2), su + (int64_t)i * (H / 32), H);
    }
}

/* Down of one Q8 row through one expert: y[n] for n < H.
 * wd [H, I/2] packed, sd [H, I/32] E8M0. */
void moe_oracle_expert_down(const int8_t *hq, const float *hs,
                            const uint8_t *wd, const uint8_t *sd,
                            int H, int I, double *y)
{
    for (int n = 0; n < H; ++n)
        y[n] = mx_dot(hq, hs, wd + (int64_t)n * (I / 2), sd + (int64_t)n * (I / 32), I);
}

/* Routing-weighted combine, slot order, fp64 ([GFX] §8.2 "FP32 top-k partial
 * and fixed reduction"): out[t,n] = sum_{j<k} w[t,j] * y[t*k+j, n]. */
void moe_oracle_combine(const double *y, const double *w, int T, int k, int H, double *out)
{
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += w[(int64_t)t * k + j] * y[((int64_t)t * k + j) * H + n];
            out[(int64_t)t * H + n] = acc;
        }
}

/* ------------------------------------------------------------------ layer */

/* The routed-expert MoE layer for T tokens ([GFX] Fig. 1, [SH] "MXFP4
 * routed-expert kernels"): route -> Q8(x) -> per assignment gate/up + SwiGLU
 * -> Q8(h) -> down -> out[t] = sum_j w[t,j] * y[t*k+j], j in slot order
 * ([GFX] §8.2 "FP32 top-k partial and fixed reduction").
 *
 * Expert weights come as arrays of E pointers; only the experts the tokens
 * select need to be present (NULL otherwise).  READING: the intermediate h is
 * quantised from its fp32 rounding (the pages' pilot rounds it to bf16 first;
 * this build keeps fp32).  Every intermediate is returned for stage-wise
 * comparison:
 *   logits [T,E] f32, ids [T,k], w [T,k] f64, xq [T,H], xs [T,H/32] f32,
 *   h [A,I] f64, hq [A,I], hs [A,I/32] f32, y [A,H] f64, out [T,H] f64.
 * Returns 0, or -1 when a selected expert's weights are missing. */
int moe_oracle_layer(const void *x, int x_bf16, int T, int H,
                     const void *wr, int wr_bf16, const float *bias,
                     int E, int k, int I,
                     const uint8_t *const *wg, const uint8_t *const *sg,
                     const uint8_t *const *wu, const uint8_t *const *su,
                     const uint8_t *const *wd, const uint8_t *const *sd,
                     float *logits, int32_t *ids, double *w,
                     int8_t *xq, float *xs,
                     double *h, int8_t *hq, float *hs,
                     double *y, double *out)
{
    int64_t A = (int64_t)T * k;
    moe_oracle_router_logits(x, x_bf16, H, wr, wr_bf16, T, H, E, logits);
    moe_oracle_topk(logits, bias, T, E, k, ids, w);
    moe_oracle_quant_q8(x, x_bf16, T, H, H, xq, H, xs, H / 32);

    double *G = (double *)malloc(sizeof(double) * (size_t)I);
    double *U = (double *)malloc(sizeof(double) * (size_t)I);
    float *hf = (float *)malloc(sizeof(float) * (size_t)I);
    int rc = 0;
    for (int64_t a = 0; a < A && rc == 0; ++a) {
        int t = (int)(a / k), e = ids[a];
        if (e < 0 || e >= E) {
            /* READING: a slot with no expert (moe_oracle_topk's NaN rule)
             * contributes nothing: its h, Q8(h) and y rows are 0 (and its
             * weight is 0). */
            for (int i = 0; i < I; ++i) { h[a * I + i] = 0.0; hq[a * I + i] = 0; }
            for (int b = 0; b < I / 32; ++b) hs[a * (I / 32) + b] = 0.0f;
            for (int n = 0; n < H; ++n) y[a * H + n] = 0.0;
            continue;
        }
        if (!wg[e] || !sg[e] || !wu[e] || !su[e] || !wd[e] || !sd[e]) { rc = -1; break; }
        moe_oracle_expert_gateup(xq + (int64_t)t * H, xs + (int64_t)t * (H / 32),
                                 wg[e], sg[e], wu[e], su[e], H, I, G, U);
        for (int i = 0; i < I; ++i) {
            h[a * I + i] = moe_oracle_silu(G[i]) * U[i];
            hf[i] = (float)h[a * I + i];
        }
        moe_oracle_quant_q8(hf, 0, 1, I, I, hq + a * I, I, hs + a * (I / 32), I / 32);
        moe_oracle_expert_down(hq + a * I, hs + a * (I / 32), wd[e], sd[e], H, I, y + a * H);
    }
    if (rc == 0) moe_oracle_combine(y, w, T, k, H, out);
    free(G);
    free(U);
    free(hf);
    return rc;
}

/* ------------------------------------------------------------------ shared expert */

/* The shared expert ([GFX] Execution structure and Fig. 1: the layer has a
 * shared expert beside the routed experts, and both feed the join that adds
 * their partials).  READING: the pages give neither the shared expert's
 * weight format nor the join's arithmetic.  This build takes one expert in
 * the routed experts' MXFP4 format and shape, run on the same Q8(x) rows
 * with weight 1 -- per token the steps of one routed assignment: gate/up +
 * SwiGLU -> Q8(h) -> down -- and the join out[t] = routed[t] + ys[t].
 *   xq [T,H], xs [T,H/32]: Q8 of the tokens (as moe_oracle_layer's);
 *   h [T,I] f64, hq [T,I], hs [T,I/32] f32, ys [T,H] f64: outputs;
 *   out [T,H] f64: the routed output on entry, the joined output on return
 *   (NULL: ys only). */
void moe_oracle_shared_expert(const int8_t *xq, const float *xs, int T, int H, int I,
                              const uint8_t *wg, const uint8_t *sg, const uint8_t *wu, const uint8_t *su,
                              const uint8_t *wd, const uint8_t *sd,
                              double *h, int8_t *hq, float *hs, double *ys, double *out)
{
    double *G = (double *)malloc(sizeof(double) * (size_t)I);
    double *U = (double *)malloc(sizeof(double) * (size_t)I);
    float *hf = (float *)malloc(sizeof(float) * (size_t)I);
    for (int t = 0; t < T; ++t) {
        moe_oracle_expert_gateup(xq + (int64_t)t * H, xs + (int64_t)t * (H / 32), wg, sg, wu, su, H, I, G, U);
        for (int i = 0; i < I; ++i) {
            h[(int64_t)t * I + i] = moe_oracle_silu(G[i]) * U[i];
            hf[i] = (float)h[(int64_t)t * I + i];
        }
        moe_oracle_quant_q8(hf, 0, 1, I, I, hq + (int64_t)t * I, I, hs + (int64_t)t * (I / 32), I / 32);
        moe_oracle_expert_down(hq + (int64_t)t * I, hs + (int64_t)t * (I / 32), wd, sd, H, I, ys + (int64_t)t * H);
        if (out)
            for (int n = 0; n < H; ++n) out[(int64_t)t * H + n] += ys[(int64_t)t * H + n];
    }
    free(G);
    free(U);
    free(hf);
}
