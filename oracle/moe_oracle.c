/*
 * moe_oracle.c -- plain, slow, FP64 CPU oracle of the small-T Mixture-of-Experts
 * FFN layer with MXFP4 expert weights.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load or call this code.  It
 * shares no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it.
 *
 * What the layer computes, for every token t (x[t] is a bf16 row of length H):
 *
 *   1. Router logits        l[t,e] = sum_h x[t,h] * Wr[h,e] + b[e],  e < E.
 *   2. Top-k + shared slot  the k largest logits (ties: lower expert index),
 *                           ordered by descending logit then ascending index;
 *                           w = softmax over the k selected logits (the same
 *                           as softmax over all E followed by renormalising the
 *                           k kept ones); the shared expert (index E) is
 *                           appended as slot k with weight shared_weight.
 *   3. Grouping             the (t, slot) pairs sorted by (expert, t).
 *   4. Expert FFN           g = Wg x, u = Wu x, h = silu(g) * u, Y = Wd h,
 *                           silu(z) = z / (1 + e^-z), weights decoded from
 *                           MXFP4: W[r][c] = e2m1(code) * 2^(s - 127) with s the
 *                           E8M0 byte of block floor(c/32) of row r.
 *   5. Combine              y[t] = sum over slots s = 0..k of w[t,s] * Y_s.
 *
 * Passages followed:
 *   - shared expert fused as an extra expert that is always selected, top-9 of
 *     161 with the shared expert in the 9th position, all expert outputs
 *     weighted and aggregated: "Optimizing GLM4-MoE for production"
 *     (blogs.novita.ai), section 1 "Shared experts fusion".
 *   - MXFP4: blocks of 32 values sharing one exponent, per the OCP
 *     Microscaling (MX) specification: "How Xiaomi reached 1,000 tokens/s on a
 *     1T-parameter model" (molayo1419.me), section 2, "MXFP4 with QAT".  The
 *     page's "3-bit mantissa" is read as the E2M1 element of the OCP MX v1.0
 *     spec (1 sign, 2 exponent, 1 mantissa bit).
 *   - top-8 routed experts per token: GLM-5.2 on B300 (d9249.github.io),
 *     section "What it solves"; same novita section.
 * Readings where the pages are silent (all from the problem statement of the
 * layer): low nibble holds the even element; E8M0 = 2^(s-127); gate rows
 * 0..I-1 then up rows I..2I-1; blocks of 32 run along each row (the reduction
 * axis); the bias is part of the logit for both selection and weights.
 *
 * Precision: every product x*w is exact in double (8-bit x 24-bit and 8-bit x
 * 3-bit significands); sums are plain left-to-right double sums.
 *
 * MXFP8 activation mode (oracle_moe_tokens_act with mx = 1): x[t] is
 * MXFP8-quantised (OCP MX v1.0, E4M3 elements, blocks of 32 along H) before
 * the gate/up projection and h before the down projection; everything else
 * as above.  Pins: tests/test_oracle_mxfp8_pins.py.
 *
 * Parity pins (tests/test_oracle_pins.py): exhaustive E2M1 table and E8M0
 * exponents against the OCP bit-field definitions, a brute-force tiny layer
 * (top-k by enumerating every k-subset, dense numpy matmuls), a closed form
 * (all weights 1.0), zero weights, the single-expert dense SwiGLU case,
 * routing and grouping invariants, linearity over slots, and the tie rule.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the oracle's parallel loops use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- formats */

/* E2M1 magnitudes indexed by the low 3 bits (exponent:mantissa), OCP MX v1.0. */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(int code)
{
    double m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* E8M0 scale: 2^(s-127); s = 255 is NaN in the MX spec. */
double oracle_e8m0_value(int s)
{
    if (s == 255)
        return NAN;
    return ldexp(1.0, s - 127);
}

double oracle_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even. */
uint16_t oracle_bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    (void)frexp(a, &e);           /* a = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;                /* weight of the last of 8 significant bits */
    if (q < -133)
        q = -133;                 /* bf16 subnormal quantum */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);   /* ties to even */
    if (r > 0x1.FEp127)           /* largest finite bf16 */
        return sign | 0x7F80;
    float f = (float)r;           /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Element c of a packed row: byte c/2, low nibble for even c. */
static int row_code(const uint8_t *codes, int c)
{
    uint8_t byte = codes[c / 2];
    return (c & 1) ? (byte >> 4) : (byte & 15);
}

/* Decode one MXFP4 row of K elements (K/32 scales) into doubles. */
void oracle_decode_row(const uint8_t *codes, const uint8_t *scales, int K, double *out)
{
    for (int c = 0; c < K; ++c)
        out[c] = oracle_e2m1_value(row_code(codes, c)) * oracle_e8m0_value(scales[c / 32]);
}

/* ------------------------------------------------- MXFP8 activations */
/*
 * The live-activation-quantisation variant (GLM-5.2 on B300, d9249.github.io,
 * section 1 of its kernel part: FP8 activations quantised right before the
 * GEMM).  The page names FP8 but neither the element format nor the block
 * size; the reading taken here is MXFP8 of the OCP Microscaling v1.0 spec,
 * the same block structure as the MXFP4 weights: E4M3 elements, one E8M0
 * scale per 32 consecutive values along the reduction axis.
 *
 * E4M3 (OCP 8-bit floating point): 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; S.1111.111
 * is NaN; there are no infinities, so the largest magnitude is 1.75 * 2^8 =
 * 448.
 */
double oracle_e4m3_value(int b)
{
    int sign = (b >> 7) & 1, ex = (b >> 3) & 15, m = b & 7;
    double v;
    if (ex == 15 && m == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)m, -9);              /* m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, ex - 10);           /* (1 + m/8) * 2^(ex-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 code to v, ties to even, magnitudes above 448 saturated to
 * 448 (the OCP MX conversion clamps to the element's largest normal). */
int oracle_e4m3_round(double v)
{
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);                        /* a = f * 2^e, 0.5 <= f < 1 */
    int q = e - 4;                             /* weight of the last of 4 significant bits */
    if (q < -9)
        q = -9;                                /* subnormal quantum */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);   /* ties to even */
    /* encode r (exactly representable; at most 448 after the clamp above,
     * since 448 < a < 448 + 16 rounds to 448) */
    if (r < ldexp(1.0, -6))
        return sign | (int)ldexp(r, 9);        /* subnormal: m = r / 2^-9 */
    (void)frexp(r, &e);
    int ex = e - 1 + 7;                         /* r = (1 + m/8) * 2^(e-1) */
    int m = (int)(ldexp(r, 4 - e) - 8.0);
    return sign | (ex << 3) | m;
}

/*
 * OCP MX v1.0 conversion of n values (n a multiple of 32) to MXFP8: for
 * each block of 32, the shared exponent is floor(log2(max |v|)) minus the
 * largest exponent of E4M3 (8), kept inside E8M0's range [-127, 127] (an
 * all-zero block takes -127); the scale byte is that exponent + 127 and
 * each element is E4M3-rounded v / 2^exponent.  deq (nullable) receives the
 * dequantised values code * 2^exponent.
 */
void oracle_mxfp8_quantize(const double *v, int n, uint8_t *codes, uint8_t *scales, double *deq)
{
    for (int b = 0; b < n / 32; ++b) {
        const double *vb = v + 32 * b;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i)
            if (fabs(vb[i]) > amax)
                amax = fabs(vb[i]);
        int se = -127;
        if (amax > 0.0) {
            int e;
            (void)frexp(amax, &e);             /* floor(log2(amax)) = e - 1 */
            se = e - 1 - 8;
            if (se < -127)
                se = -127;
            if (se > 127)
                se = 127;
        }
        scales[b] = (uint8_t)(se + 127);
        for (int i = 0; i < 32; ++i) {
            int c = oracle_e4m3_round(ldexp(vb[i], -se));
            codes[32 * b + i] = (uint8_t)c;
            if (deq)
                deq[32 * b + i] = ldexp(oracle_e4m3_value(c), se);
        }
    }
}

/* ----------------------------------------------------------------- router */

/* l[t,e] = sum_h x[t,h] * Wr[h,e] + b[e]; abs_sum[t,e] = sum_h |x[t,h] * Wr[h,e]|. */
void oracle_router_logits(const uint16_t *x, const float *wr, const float *bias,
                          int T, int H, int E, double *logits, double *abs_sum)
{
    double *acc = calloc((size_t)E, sizeof(double));
    double *mag = calloc((size_t)E, sizeof(double));
    for (int t = 0; t < T; ++t) {
        memset(acc, 0, sizeof(double) * (size_t)E);
        memset(mag, 0, sizeof(double) * (size_t)E);
        for (int h = 0; h < H; ++h) {
            double xv = oracle_bf16_value(x[(size_t)t * H + h]);
            for (int e = 0; e < E; ++e) {
                double p = xv * (double)wr[(size_t)h * E + e];
                acc[e] += p;
                mag[e] += fabs(p);
            }
        }
        for (int e = 0; e < E; ++e) {
            logits[(size_t)t * E + e] = acc[e] + (bias ? (double)bias[e] : 0.0);
            if (abs_sum)
                abs_sum[(size_t)t * E + e] = mag[e];
        }
    }
    free(acc);
    free(mag);
}

/* Does expert a rank before expert b?  Larger logit first, ties to lower index. */
static int ranks_before(const double *l, int a, int b)
{
    return l[a] > l[b] || (l[a] == l[b] && a < b);
}

/*
 * Top-k selection, softmax over the selected logits, shared slot.
 * ids/w: [T, k + has_shared].  gap[t] (nullable): the smallest difference
 * between consecutive logits among the token's k+1 best, the margin that
 * decides both the chosen set and its order.
 */
void oracle_topk(const double *logits, int T, int E, int k, int has_shared,
                 double shared_weight, int32_t *ids, double *w, double *gap)
{
    int kps = k + has_shared;
    int nsel = k < E ? k + 1 : k;
    int *order = malloc(sizeof(int) * (size_t)nsel);
    char *taken = malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int i = 0; i < nsel; ++i) {       /* selection sort, one pick per slot */
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || ranks_before(l, e, best)))
                    best = e;
            order[i] = best;
            taken[best] = 1;
        }
        double lmax = l[order[0]], z = 0.0;
        for (int i = 0; i < k; ++i)
            z += exp(l[order[i]] - lmax);
        for (int i = 0; i < k; ++i) {
            ids[(size_t)t * kps + i] = order[i];
            w[(size_t)t * kps + i] = exp(l[order[i]] - lmax) / z;
        }
        if (has_shared) {
            ids[(size_t)t * kps + k] = E;
            w[(size_t)t * kps + k] = shared_weight;
        }
        if (gap) {
            double g = INFINITY;
            for (int i = 0; i + 1 < nsel; ++i)
                g = fmin(g, l[order[i]] - l[order[i + 1]]);
            gap[t] = g;
        }
    }
    free(order);
    free(taken);
}

/* Router + top-k for all T tokens. logits/abs_sum/gap are nullable outputs. */
void oracle_route(const uint16_t *x, const float *wr, const float *bias, int T, int H, int E,
                  int k, int has_shared, double shared_weight, int32_t *ids, double *w,
                  double *logits_out, double *abs_sum_out, double *gap_out)
{
    double *l = logits_out ? logits_out : malloc(sizeof(double) * (size_t)T * E);
    oracle_router_logits(x, wr, bias, T, H, E, l, abs_sum_out);
    oracle_topk(l, T, E, k, has_shared, shared_weight, ids, w, gap_out);
    if (!logits_out)
        free(l);
}

/* --------------------------------------------------------------- grouping */

/*
 * (t, slot) pairs sorted by (expert, t).  offsets [n_tot+1] (exclusive prefix
 * of the per-expert counts), sorted_tok / sorted_slot [T*kps], active [n_tot]
 * (experts with a nonzero count, ascending), *num_active.
 * Returns 0, or -1 if an id is out of range.
 */
int oracle_group(const int32_t *ids, int T, int kps, int n_tot, int32_t *offsets,
                 int32_t *sorted_tok, int32_t *sorted_slot, int32_t *active, int32_t *num_active)
{
    for (int i = 0; i < T * kps; ++i)
        if (ids[i] < 0 || ids[i] >= n_tot)
            return -1;
    int pos = 0, na = 0;
    for (int e = 0; e < n_tot; ++e) {
        offsets[e] = pos;
        for (int t = 0; t < T; ++t)
            for (int s = 0; s < kps; ++s)
                if (ids[t * kps + s] == e) {
                    sorted_tok[pos] = t;
                    sorted_slot[pos] = s;
                    ++pos;
                }
        if (pos > offsets[e])
            active[na++] = e;
    }
    offsets[n_tot] = pos;
    *num_active = na;
    return 0;
}

/* ------------------------------------------------------------- expert FFN */

/*
 * One expert on one token.  w13 [2I][H/2] (gate rows then up rows), s13
 * [2I][H/32], w2 [H][I/2], s2 [H][I/32].  x [H] in double.
 * h_out [I] (nullable), y_out [H].  With mx, h enters the down projection
 * MXFP8-quantised (blocks of 32 along I); h_out keeps the unquantised h.
 */
static void expert_token(const uint8_t *w13, const uint8_t *s13, const uint8_t *w2,
                         const uint8_t *s2, int H, int I, const double *x,
                         double *h_out, double *y_out, int mx)
{
    double *h = malloc(sizeof(double) * (size_t)I);
    double *hq = malloc(sizeof(double) * (size_t)I);
#pragma omp parallel for schedule(static)
    for (int j = 0; j < I; ++j) {
        double *row = malloc(sizeof(double) * (size_t)H);
        double g = 0.0, u = 0.0;
        oracle_decode_row(w13 + (size_t)j * (H / 2), s13 + (size_t)j * (H / 32), H, row);
        for (int c = 0; c < H; ++c)
            g += row[c] * x[c];
        oracle_decode_row(w13 + (size_t)(I + j) * (H / 2), s13 + (size_t)(I + j) * (H / 32), H, row);
        for (int c = 0; c < H; ++c)
            u += row[c] * x[c];
        h[j] = g / (1.0 + exp(-g)) * u;
        free(row);
    }
    if (mx) {
        uint8_t *codes = malloc((size_t)I), *scales = malloc((size_t)I / 32);
        oracle_mxfp8_quantize(h, I, codes, scales, hq);
        free(codes);
        free(scales);
    } else {
        memcpy(hq, h, sizeof(double) * (size_t)I);
    }
#pragma omp parallel for schedule(static)
    for (int n = 0; n < H; ++n) {
        double *row = malloc(sizeof(double) * (size_t)I);
        double acc = 0.0;
        oracle_decode_row(w2 + (size_t)n * (I / 2), s2 + (size_t)n * (I / 32), I, row);
        for (int j = 0; j < I; ++j)
            acc += row[j] * hq[j];
        y_out[n] = acc;
        free(row);
    }
    if (h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(h);
    free(hq);
}

void oracle_expert_token(const uint8_t *w13, const uint8_t *s13, const uint8_t *w2,
                         const uint8_t *s2, int H, int I, const double *x,
                         double *h_out, double *y_out)
{
    expert_token(w13, s13, w2, s2, H, I, x, h_out, y_out, 0);
}

/*
 * Expert FFNs and combine for the listed tokens, given the routing.
 * Expert e's arrays are w13[e], s13[e], w2[e], s2[e] (per-expert pointers, so
 * a caller may supply only the experts its tokens touch).
 * y [n_tokens][H]; hs [n_tokens][kps][I] and ys [n_tokens][kps][H] nullable.
 * mx = 1: MXFP8 activations -- x[t] is quantised (blocks of 32 along H)
 * before the gate/up projection and each h before the down projection.
 */
void oracle_moe_tokens_act(const uint16_t *x, int H, int I, int kps, const int32_t *ids,
                           const double *w, const uint8_t *const *w13, const uint8_t *const *s13,
                           const uint8_t *const *w2, const uint8_t *const *s2,
                           const int32_t *tokens, int n_tokens, double *y, double *hs, double *ys, int mx)
{
    double *xt = malloc(sizeof(double) * (size_t)H);
    double *yslot = malloc(sizeof(double) * (size_t)H);
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens[i];
        for (int c = 0; c < H; ++c)
            xt[c] = oracle_bf16_value(x[(size_t)t * H + c]);
        if (mx) {
            uint8_t *codes = malloc((size_t)H), *scales = malloc((size_t)H / 32);
            oracle_mxfp8_quantize(xt, H, codes, scales, xt);
            free(codes);
            free(scales);
        }
        double *yt = y + (size_t)i * H;
        for (int c = 0; c < H; ++c)
            yt[c] = 0.0;
        for (int s = 0; s < kps; ++s) {
            int e = ids[(size_t)t * kps + s];
            double *hdst = hs ? hs + ((size_t)i * kps + s) * I : NULL;
            expert_token(w13[e], s13[e], w2[e], s2[e], H, I, xt, hdst, yslot, mx);
            if (ys)
                memcpy(ys + ((size_t)i * kps + s) * H, yslot, sizeof(double) * (size_t)H);
            double ws = w[(size_t)t * kps + s];
            for (int c = 0; c < H; ++c)
                yt[c] += ws * yslot[c];
        }
    }
    free(xt);
    free(yslot);
}

void oracle_moe_tokens(const uint16_t *x, int H, int I, int kps, const int32_t *ids,
                       const double *w, const uint8_t *const *w13, const uint8_t *const *s13,
                       const uint8_t *const *w2, const uint8_t *const *s2,
                       const int32_t *tokens, int n_tokens, double *y, double *hs, double *ys)
{
    oracle_moe_tokens_act(x, H, I, kps, ids, w, w13, s13, w2, s2, tokens, n_tokens, y, hs, ys, 0);
}

/* bf16 rounding of a whole array (the layer's output format). */
void oracle_bf16_round_array(const double *v, size_t n, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_round(v[i]);
}
