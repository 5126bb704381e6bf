/* Plain C definition of the route plan and of the A16W16, A8W8-INT and FP8 x FP4 expert
 * feed-forward with top-k combine.
 *
 * TEST INFRASTRUCTURE ONLY: a second, independent statement of what oracle/moe.py computes for
 * the plan and the A16W16, A8W8-INT and FP8 x FP4 modes, written with plain loops in double precision (and
 * the fp32 roundings the readings fix), which the CPU tests compare with it. Nothing in the product path links or loads it; it shares no code with the
 * CUDA path.
 *
 * Ascend mega_moe page, "Computation Process", A16W16 use case:
 *   EP Dispatch: the rows routed to expert e, I_e = {(i, k) : E[i,k] = e}, N_e = |I_e|, stacked in
 *     ascending i*K + k (a stable counting sort: count, exclusive prefix sum, scatter);
 *   Linear1: H = X_e . W1[e] (W1[e] is hidden x 2*intermediate);
 *   SwiGLU: A = SiLU(H[:, :I]) * H[:, I:], SiLU(z) = z / (1 + e^-z);
 *   Linear2: Y_e = A . W2[e] with A rounded to bf16 (both GEMMs take bf16 operands);
 *   Token Combine: c[i,k] = bf16(fp32(G[i,k] * Y_e[row(i,k)])), y_i = bf16(sum over k = 0..K-1 of
 *     c[i,k] in fp32, in slot order). A masked route (id -1) contributes nothing.
 * Everything else runs in double precision. These are the readings oracle/moe.py states.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* Nearest bf16 value (ties to even) of a double, as a double: bf16 keeps 8 significant bits, the
 * spacing in [2^e, 2^(e+1)) is 2^(e-7), below 2^-126 it stays 2^-133; beyond the largest finite
 * bf16 (plus half a spacing) the value rounds to infinity. */
static double round_to_bf16(double v) {
    if (!isfinite(v)) return v;
    int ex;
    frexp(v, &ex); /* |v| in [2^(ex-1), 2^ex) */
    int e = ex - 1 < -126 ? -126 : ex - 1;
    const double q = ldexp(1.0, e - 7);
    const double r = nearbyint(v / q) * q; /* the default rounding mode: half to even */
    const double bf16_max = (2.0 - ldexp(1.0, -7)) * ldexp(1.0, 127);
    return fabs(r) > bf16_max ? copysign(INFINITY, v) : r;
}

/* Token Combine: y_t = bf16(sum over the slots k = 0..K-1 of the bf16 rows comb[t*K + k], in fp32 in
 * slot order); a masked slot's row is zero. */
static void combine_tokens(const double* comb, int64_t T, int64_t K, int64_t H, double* y) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) acc = acc + (float)comb[(t * K + k) * H + c];
            y[t * H + c] = round_to_bf16((double)acc);
        }
}

/* The weighted combine row of one routed row: bf16(fp32(G * Y)). */
static double gated(float g, double yv) { return round_to_bf16((double)(float)((double)g * yv)); }

/* counts[E], offsets[E+1], row_src[offsets[E]] of the T x K routing ids; returns 0, or -1 when an
 * id lies outside [-1, E). */
int oracle_plan(const int32_t* ids, int64_t T, int64_t K, int64_t E, int64_t* counts, int64_t* offsets,
                int64_t* row_src) {
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t r = 0; r < T * K; ++r) {
        if (ids[r] < -1 || ids[r] >= E) return -1;
        if (ids[r] >= 0) ++counts[ids[r]];
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t* cursor = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor) return -2;
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t r = 0; r < T * K; ++r)
        if (ids[r] >= 0) row_src[cursor[ids[r]]++] = r;
    free(cursor);
    return 0;
}

/* y [T, H] (bf16 values as doubles) of the A16W16 layer. x [T, H], w1 [E, H, 2I], w2 [E, I, H] hold
 * the decoded bf16 operands, g [T*K] the fp32 gate weights. Returns 0, -1 for a bad id, -2 when
 * memory runs out. */
int oracle_forward_a16w16(const double* x, const int32_t* ids, const float* g, const double* w1, const double* w2,
                          int64_t T, int64_t K, int64_t E, int64_t H, int64_t I, double* y) {
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    int64_t* offsets = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int64_t* row_src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * K > 0 ? T * K : 1));
    double* comb = (double*)calloc((size_t)(T * K * H > 0 ? T * K * H : 1), sizeof(double));
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    int st = (counts && offsets && row_src && comb && h && a) ? 0 : -2;
    if (st == 0) st = oracle_plan(ids, T, K, E, counts, offsets, row_src);
    for (int64_t e = 0; st == 0 && e < E; ++e) {
        const double* w1e = w1 + e * H * 2 * I;
        const double* w2e = w2 + e * I * H;
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            const double* xr = x + tok * H;
            for (int64_t j = 0; j < 2 * I; ++j) { /* Linear1 */
                double s = 0.0;
                for (int64_t c = 0; c < H; ++c) s += xr[c] * w1e[c * 2 * I + j];
                h[j] = s;
            }
            for (int64_t j = 0; j < I; ++j) /* SwiGLU, then the bf16 L2 operand */
                a[j] = round_to_bf16(h[j] / (1.0 + exp(-h[j])) * h[I + j]);
            for (int64_t c = 0; c < H; ++c) { /* Linear2, gate, the bf16 combine row */
                double s = 0.0;
                for (int64_t j = 0; j < I; ++j) s += a[j] * w2e[j * H + c];
                comb[src * H + c] = gated(g[src], s);
            }
        }
    }
    if (st == 0) combine_tokens(comb, T, K, H, y);
    free(counts);
    free(offsets);
    free(row_src);
    free(comb);
    free(h);
    free(a);
    return st;
}

/* y [T, H] of the A8W8-INT layer (Ascend mega_moe page, A8W8-INT use case). x int8 [T, H] with the
 * fp32 per-token scales x_scale [T]; w1 int8 [E, 2I, H] and w2 int8 [E, H, I] (output channel,
 * then input) with fp32 per-output-channel scales [E, 2I] and [E, H]; g [T*K] fp32.
 *   Linear1: C = Q . W1 in integers; H = (C * s^W1) * s^X, each product rounded to fp32;
 *   SwiGLU in double precision on H;
 *   Linear2 step (1): A rounded to fp32; s^A = max(fp32(max|A| / 127), 1e-8);
 *     q = clamp(round-half-even(fp32(A / s^A)), -127, 127);
 *   Linear2: D = q . W2 in integers; Y = (D * s^W2) * s^A, each product rounded to fp32;
 *   Token Combine as in the A16W16 layer.
 * Returns 0, -1 for a bad id, -2 when memory runs out. */
int oracle_forward_int8(const int8_t* x, const float* x_scale, const int32_t* ids, const float* g, const int8_t* w1,
                        const float* w1_scale, const int8_t* w2, const float* w2_scale, int64_t T, int64_t K, int64_t E,
                        int64_t H, int64_t I, double* y) {
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    int64_t* offsets = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int64_t* row_src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * K > 0 ? T * K : 1));
    double* comb = (double*)calloc((size_t)(T * K * H > 0 ? T * K * H : 1), sizeof(double));
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    float* a32 = (float*)malloc(sizeof(float) * (size_t)I);
    int32_t* q = (int32_t*)malloc(sizeof(int32_t) * (size_t)I);
    int st = (counts && offsets && row_src && comb && h && a32 && q) ? 0 : -2;
    if (st == 0) st = oracle_plan(ids, T, K, E, counts, offsets, row_src);
    for (int64_t e = 0; st == 0 && e < E; ++e) {
        const int8_t* w1e = w1 + e * 2 * I * H;
        const int8_t* w2e = w2 + e * H * I;
        const float* s1 = w1_scale + e * 2 * I;
        const float* s2 = w2_scale + e * H;
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            const int8_t* xr = x + tok * H;
            const float sx = x_scale[tok];
            for (int64_t j = 0; j < 2 * I; ++j) { /* Linear1 */
                int64_t c = 0;
                for (int64_t k = 0; k < H; ++k) c += (int64_t)xr[k] * (int64_t)w1e[j * H + k];
                float v = (float)c * s1[j];
                v = v * sx;
                h[j] = (double)v;
            }
            float amax = 0.0f;
            for (int64_t j = 0; j < I; ++j) { /* SwiGLU, in fp32 for the quantiser */
                a32[j] = (float)(h[j] / (1.0 + exp(-h[j])) * h[I + j]);
                const float m = fabsf(a32[j]);
                amax = m > amax ? m : amax;
            }
            float sa = amax / 127.0f;
            sa = sa > 1e-8f ? sa : 1e-8f;
            for (int64_t j = 0; j < I; ++j) {
                float t = rintf(a32[j] / sa);
                t = t < -127.0f ? -127.0f : (t > 127.0f ? 127.0f : t);
                q[j] = (int32_t)t;
            }
            for (int64_t c = 0; c < H; ++c) { /* Linear2, gate, the bf16 combine row */
                int64_t d = 0;
                for (int64_t j = 0; j < I; ++j) d += (int64_t)q[j] * (int64_t)w2e[c * I + j];
                float v = (float)d * s2[c];
                v = v * sa;
                comb[src * H + c] = gated(g[src], (double)v);
            }
        }
    }
    if (st == 0) combine_tokens(comb, T, K, H, y);
    free(counts);
    free(offsets);
    free(row_src);
    free(comb);
    free(h);
    free(a32);
    free(q);
    return st;
}

/* ---- FP8 (e4m3) activations x FP4 (e2m1) weights, block-scaled (DeepGEMM MegaMoE page §4: FP8
 * activations with 1x128 power-of-two fp32 scales, e2m1 weights with a UE8M0 scale per 32 of K; the
 * L1 output re-quantised to e4m3 with a UE8M0 exponent per 32, Ascend page "Q_MX") ---- */

/* e4m3fn code -> value: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal;
 * S.1111.111 is NaN. */
static double e4m3_value(uint8_t c) {
    const double s = (c & 0x80) ? -1.0 : 1.0;
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) return s * (m / 8.0) * ldexp(1.0, -6);
    return s * (1.0 + m / 8.0) * ldexp(1.0, e - 7);
}

/* Nearest e4m3fn code of v, ties to the even code, magnitudes above 448 taken as 448 (a saturating
 * conversion); the sign bit follows v, also when the magnitude rounds to zero. */
static uint8_t e4m3_encode(double v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0;
    double mag = fabs(v);
    if (mag > 448.0) mag = 448.0;
    if (mag < ldexp(1.0, -6)) {  /* subnormal range: spacing 2^-9; 8 * 2^-9 is the smallest normal */
        const int m = (int)nearbyint(mag / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    int ex;
    frexp(mag, &ex);  /* mag in [2^(ex-1), 2^ex) */
    const int e = ex - 1;
    int r = (int)nearbyint(mag / ldexp(1.0, e - 3));  /* 8 + mantissa, half to even */
    int be = e + 7;
    if (r == 16) r = 8, ++be;
    return (uint8_t)(sign | (be << 3) | (r - 8));
}

/* e2m1 code (4 bits) -> value: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal. */
static double e2m1_value(int c) {
    const double s = (c & 8) ? -1.0 : 1.0;
    const int e = (c >> 1) & 3, m = c & 1;
    if (e == 0) return s * 0.5 * m;
    return s * (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
}

/* UE8M0 scale byte -> 2^(b - 127); 255 is NaN. */
static double ue8m0_value(uint8_t b) { return b == 255 ? NAN : ldexp(1.0, (int)b - 127); }

/* Element k of a packed e2m1 row (element 2j in the low nibble of byte j) times its UE8M0 scale. */
static double fp4_weight(const uint8_t* row, const uint8_t* scales, int64_t k) {
    const int c = (k & 1) ? row[k >> 1] >> 4 : row[k >> 1] & 0xF;
    return e2m1_value(c) * ue8m0_value(scales[k / 32]);
}

/* y [T, H] of the FP8 x FP4 layer. x e4m3 [T, H] with fp32 scales [T, H/128]; w1 packed e2m1
 * [E, 2I, H/2] with UE8M0 [E, 2I, H/32]; w2 packed e2m1 [E, H, I/2] with UE8M0 [E, H, I/32]; g [T*K].
 *   Linear1: H = X_e . W1[e] on the decoded values, in double precision;
 *   SwiGLU in double precision;
 *   re-quantisation of A: A rounded to fp32; per 32 consecutive outputs the exponent e, the
 *     smallest integer with amax <= 448 * 2^e (clamped to [-127, 127], -127 for amax = 0), and
 *     codes e4m3(A / 2^e); the L2 operand is their value times 2^e;
 *   Linear2: Y = A~ . W2[e] in double precision; Token Combine as in the A16W16 layer.
 * Returns 0, -1 for a bad id, -2 when memory runs out. */
int oracle_forward_fp8_fp4(const uint8_t* x, const float* x_scale, const int32_t* ids, const float* g,
                           const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                           int64_t T, int64_t K, int64_t E, int64_t H, int64_t I, double* y) {
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    int64_t* offsets = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int64_t* row_src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * K > 0 ? T * K : 1));
    double* comb = (double*)calloc((size_t)(T * K * H > 0 ? T * K * H : 1), sizeof(double));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    int st = (counts && offsets && row_src && comb && xv && h && a) ? 0 : -2;
    if (st == 0) st = oracle_plan(ids, T, K, E, counts, offsets, row_src);
    for (int64_t e = 0; st == 0 && e < E; ++e) {
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            for (int64_t k = 0; k < H; ++k)
                xv[k] = e4m3_value(x[tok * H + k]) * (double)x_scale[tok * (H / 128) + k / 128];
            for (int64_t j = 0; j < 2 * I; ++j) { /* Linear1 */
                const uint8_t* wr = w1 + (e * 2 * I + j) * (H / 2);
                const uint8_t* sr = w1_scale + (e * 2 * I + j) * (H / 32);
                double s = 0.0;
                for (int64_t k = 0; k < H; ++k) s += xv[k] * fp4_weight(wr, sr, k);
                h[j] = s;
            }
            for (int64_t j = 0; j < I; ++j) /* SwiGLU, rounded to fp32 for the quantiser */
                a[j] = (double)(float)(h[j] / (1.0 + exp(-h[j])) * h[I + j]);
            for (int64_t b = 0; b < I; b += 32) { /* MX e4m3 re-quantisation, blocks of 32 */
                double amax = 0.0;
                for (int64_t j = b; j < b + 32; ++j) amax = fabs(a[j]) > amax ? fabs(a[j]) : amax;
                int ex = -127;
                if (amax > 0.0) {
                    int fe;
                    const double fm = frexp(amax / 448.0, &fe);
                    ex = fm == 0.5 ? fe - 1 : fe;
                    ex = ex < -127 ? -127 : (ex > 127 ? 127 : ex);
                }
                for (int64_t j = b; j < b + 32; ++j) a[j] = e4m3_value(e4m3_encode(a[j] / ldexp(1.0, ex))) * ldexp(1.0, ex);
            }
            for (int64_t c = 0; c < H; ++c) { /* Linear2, gate, the bf16 combine row */
                const uint8_t* wr = w2 + (e * H + c) * (I / 2);
                const uint8_t* sr = w2_scale + (e * H + c) * (I / 32);
                double s = 0.0;
                for (int64_t j = 0; j < I; ++j) s += a[j] * fp4_weight(wr, sr, j);
                comb[src * H + c] = gated(g[src], s);
            }
        }
    }
    if (st == 0) combine_tokens(comb, T, K, H, y);
    free(counts);
    free(offsets);
    free(row_src);
    free(comb);
    free(xv);
    free(h);
    free(a);
    return st;
}

/* The e4m3 encoder on its own, for the codec test. */
uint8_t oracle_e4m3_encode(double v) { return e4m3_encode(v); }
