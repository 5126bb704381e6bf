/* Plain C definition of the route plan, the shared-expert slots and the expert feed-forward with
 * top-k combine in every dtype mode: A16W16, A8W8-FP8 (e4m3 or e5m2), A8W8-INT, A8W4-INT and FP8 x FP4.
 *
 * TEST INFRASTRUCTURE ONLY: a second, independent statement of what oracle/moe.py computes, written
 * with plain loops in double precision (and the fp32 roundings the readings fix), which the CPU tests
 * compare with it. Every number format is decoded from its bit fields here (no table shared with the
 * numpy oracle), and the integer modes multiply the codes directly. Nothing in the product path links
 * or loads it; it shares no code with the CUDA path.
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

/* Integer weight code k of a row: int8 (one per byte), or int4 (two's complement nibbles, two per byte,
 * element 2j in the low nibble: the Ascend page's int4 packing). */
static int64_t int_weight(const int8_t* row, int64_t k, int bits) {
    if (bits == 8) return (int64_t)row[k];
    const int nib = (k & 1) ? ((uint8_t)row[k >> 1] >> 4) : ((uint8_t)row[k >> 1] & 0xF);
    return (int64_t)(nib >= 8 ? nib - 16 : nib);
}

/* y [T, H] of the integer layers (Ascend mega_moe page, A8W8-INT use case; the A8W4-INT use case with
 * int4 weights). x int8 [T, H] with the fp32 per-token scales x_scale [T]; w1 [E, 2I, H] and w2 [E, H, I]
 * (output channel, then input) as int8 codes (weight_bits 8) or packed int4 codes (weight_bits 4, rows of
 * H/2 and I/2 bytes) with fp32 per-output-channel scales [E, 2I] and [E, H]; g [T*K] fp32.
 *   Linear1: C = Q . W1 in integers; H = (C * s^W1) * s^X, each product rounded to fp32;
 *   SwiGLU in double precision on H;
 *   Linear2 step (1): A rounded to fp32; s^A = max(fp32(max|A| / 127), 1e-8);
 *     q = clamp(round-half-even(fp32(A / s^A)), -127, 127);
 *   Linear2: D = q . W2 in integers; Y = (D * s^W2) * s^A, each product rounded to fp32;
 *   Token Combine as in the A16W16 layer.
 * The int4 products are formed directly (the page's MSD split of the activations into nibbles with a
 * compensation bias reaches the same integers). When c_out, q_out, sa_out, d_out are not NULL they receive,
 * per pool row p (the plan's order), C [R, 2I], the codes q [R, I], s^A [R] and D [R, H].
 * Returns 0, -1 for a bad id, -2 when memory runs out, -3 when an accumulator leaves int32 (the pages
 * require int32 results). */
int oracle_forward_int(int weight_bits, const int8_t* x, const float* x_scale, const int32_t* ids, const float* g,
                       const int8_t* w1, const float* w1_scale, const int8_t* w2, const float* w2_scale, int64_t T,
                       int64_t K, int64_t E, int64_t H, int64_t I, double* y, int64_t* c_out, int32_t* q_out,
                       float* sa_out, int64_t* d_out) {
    if (weight_bits != 8 && weight_bits != 4) return -1;
    const int64_t row1 = weight_bits == 8 ? H : H / 2, row2 = weight_bits == 8 ? I : I / 2; /* bytes per row */
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
        const int8_t* w1e = w1 + e * 2 * I * row1;
        const int8_t* w2e = w2 + e * H * row2;
        const float* s1 = w1_scale + e * 2 * I;
        const float* s2 = w2_scale + e * H;
        for (int64_t p = offsets[e]; st == 0 && p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            const int8_t* xr = x + tok * H;
            const float sx = x_scale[tok];
            for (int64_t j = 0; j < 2 * I; ++j) { /* Linear1 */
                int64_t c = 0;
                for (int64_t k = 0; k < H; ++k) c += (int64_t)xr[k] * int_weight(w1e + j * row1, k, weight_bits);
                if (c < INT32_MIN || c > INT32_MAX) st = -3;
                if (c_out) c_out[p * 2 * I + j] = c;
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
            if (sa_out) sa_out[p] = sa;
            for (int64_t j = 0; j < I; ++j) {
                float t = rintf(a32[j] / sa);
                t = t < -127.0f ? -127.0f : (t > 127.0f ? 127.0f : t);
                q[j] = (int32_t)t;
                if (q_out) q_out[p * I + j] = q[j];
            }
            for (int64_t c = 0; c < H; ++c) { /* Linear2, gate, the bf16 combine row */
                int64_t d = 0;
                for (int64_t j = 0; j < I; ++j) d += (int64_t)q[j] * int_weight(w2e + c * row2, j, weight_bits);
                if (d < INT32_MIN || d > INT32_MAX) st = -3;
                if (d_out) d_out[p * H + c] = d;
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

/* The routing with S shared experts (DeepGEMM MegaMoE page §6): a shared expert takes no routed id, runs
 * on every token and writes the combine slot after the K routed ones. Shared expert j is expert E + j of
 * the weight tensors, its slot K + j carries weight 1 (the page gives it no gate). ids [T, K], g [T, K]
 * -> ids_out [T, K + S], g_out [T, K + S]; the forward functions then run with K + S slots and E + S
 * experts. */
void oracle_shared_slots(const int32_t* ids, const float* g, int64_t T, int64_t K, int64_t E, int64_t S,
                         int32_t* ids_out, float* g_out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < K; ++k) {
            ids_out[t * (K + S) + k] = ids[t * K + k];
            g_out[t * (K + S) + k] = g[t * K + k];
        }
        for (int64_t j = 0; j < S; ++j) {
            ids_out[t * (K + S) + K + j] = (int32_t)(E + j);
            g_out[t * (K + S) + K + j] = 1.0f;
        }
    }
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

/* e5m2 code -> value: sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent 0 is subnormal;
 * exponent 31 is infinity (mantissa 0) or NaN. */
static double e5m2_value(uint8_t c) {
    const double s = (c & 0x80) ? -1.0 : 1.0;
    const int e = (c >> 2) & 0x1F, m = c & 3;
    if (e == 0x1F) return m ? NAN : s * INFINITY;
    if (e == 0) return s * (m / 4.0) * ldexp(1.0, -14);
    return s * (1.0 + m / 4.0) * ldexp(1.0, e - 15);
}

/* Nearest e5m2 code of v, ties to the even code, magnitudes above 57344 (the largest finite value)
 * taken as 57344; the sign bit follows v. */
static uint8_t e5m2_encode(double v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0;
    double mag = fabs(v);
    if (mag > 57344.0) mag = 57344.0;
    if (mag < ldexp(1.0, -14)) { /* subnormal range: spacing 2^-16; 4 * 2^-16 is the smallest normal */
        const int m = (int)nearbyint(mag / ldexp(1.0, -16));
        return (uint8_t)(sign | m);
    }
    int ex;
    frexp(mag, &ex);
    const int e = ex - 1;
    int r = (int)nearbyint(mag / ldexp(1.0, e - 2)); /* 4 + mantissa, half to even */
    int be = e + 15;
    if (r == 8) r = 4, ++be;
    return (uint8_t)(sign | (be << 2) | (r - 4));
}

/* The two FP8 formats by name: fmt 0 is e4m3 (largest finite 448), 1 is e5m2 (57344). */
static double fp8_value(int fmt, uint8_t c) { return fmt ? e5m2_value(c) : e4m3_value(c); }
static uint8_t fp8_encode(int fmt, double v) { return fmt ? e5m2_encode(v) : e4m3_encode(v); }
static double fp8_max(int fmt) { return fmt ? 57344.0 : 448.0; }

/* Q_MX of n consecutive values of A (Ascend mega_moe page, A8W8-FP use case: groups of 32, one shared
 * power-of-two exponent per group, FP8 codes): each value is first rounded to fp32; per group of 32 the
 * exponent e is the smallest integer with amax <= fp8_max * 2^e (clamped to [-127, 127]; -127 for
 * amax = 0), the codes are fp8(a / 2^e). a is replaced by the values the codes stand for; codes and
 * UE8M0 bytes (e + 127) go to codes_out / exp_out when not NULL. */
static void mx_requant(double* a, int64_t n, int fmt, uint8_t* codes_out, uint8_t* exp_out) {
    for (int64_t j = 0; j < n; ++j) a[j] = (double)(float)a[j];
    for (int64_t b = 0; b < n; b += 32) {
        double amax = 0.0;
        for (int64_t j = b; j < b + 32; ++j) amax = fabs(a[j]) > amax ? fabs(a[j]) : amax;
        int ex = -127;
        if (amax > 0.0) {
            int fe;
            const double fm = frexp(amax / fp8_max(fmt), &fe); /* amax / max = fm * 2^fe, fm in [0.5, 1) */
            ex = fm == 0.5 ? fe - 1 : fe;
            ex = ex < -127 ? -127 : (ex > 127 ? 127 : ex);
        }
        if (exp_out) exp_out[b / 32] = (uint8_t)(ex + 127);
        for (int64_t j = b; j < b + 32; ++j) {
            const uint8_t c = fp8_encode(fmt, a[j] / ldexp(1.0, ex));
            if (codes_out) codes_out[j] = c;
            a[j] = fp8_value(fmt, c) * ldexp(1.0, ex);
        }
    }
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
 * a_codes_out [R, I] and a_exp_out [R, I/32], when not NULL, receive the re-quantised A per pool row.
 * Returns 0, -1 for a bad id, -2 when memory runs out. */
int oracle_forward_fp8_fp4(const uint8_t* x, const float* x_scale, const int32_t* ids, const float* g,
                           const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                           int64_t T, int64_t K, int64_t E, int64_t H, int64_t I, double* y, uint8_t* a_codes_out,
                           uint8_t* a_exp_out) {
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    int64_t* offsets = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int64_t* row_src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * K > 0 ? T * K : 1));
    double* comb = (double*)calloc((size_t)(T * K * H > 0 ? T * K * H : 1), sizeof(double));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* w1d = (double*)malloc(sizeof(double) * (size_t)(2 * I * H)); /* the expert's weights, decoded */
    double* w2d = (double*)malloc(sizeof(double) * (size_t)(H * I));
    int st = (counts && offsets && row_src && comb && xv && h && a && w1d && w2d) ? 0 : -2;
    if (st == 0) st = oracle_plan(ids, T, K, E, counts, offsets, row_src);
    for (int64_t e = 0; st == 0 && e < E; ++e) {
        if (offsets[e + 1] == offsets[e]) continue; /* no rows */
        for (int64_t j = 0; j < 2 * I; ++j)         /* decode W1[e] and W2[e] to their values once */
            for (int64_t k = 0; k < H; ++k)
                w1d[j * H + k] = fp4_weight(w1 + (e * 2 * I + j) * (H / 2), w1_scale + (e * 2 * I + j) * (H / 32), k);
        for (int64_t c = 0; c < H; ++c)
            for (int64_t j = 0; j < I; ++j)
                w2d[c * I + j] = fp4_weight(w2 + (e * H + c) * (I / 2), w2_scale + (e * H + c) * (I / 32), j);
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            for (int64_t k = 0; k < H; ++k)
                xv[k] = e4m3_value(x[tok * H + k]) * (double)x_scale[tok * (H / 128) + k / 128];
            for (int64_t j = 0; j < 2 * I; ++j) { /* Linear1 */
                double s = 0.0;
                for (int64_t k = 0; k < H; ++k) s += xv[k] * w1d[j * H + k];
                h[j] = s;
            }
            for (int64_t j = 0; j < I; ++j) /* SwiGLU */
                a[j] = h[j] / (1.0 + exp(-h[j])) * h[I + j];
            /* the e4m3 re-quantisation of A, blocks of 32 */
            mx_requant(a, I, 0, a_codes_out ? a_codes_out + p * I : NULL, a_exp_out ? a_exp_out + p * (I / 32) : NULL);
            for (int64_t c = 0; c < H; ++c) { /* Linear2, gate, the bf16 combine row */
                double s = 0.0;
                for (int64_t j = 0; j < I; ++j) s += a[j] * w2d[c * I + j];
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
    free(w1d);
    free(w2d);
    return st;
}

/* y [T, H] of the A8W8-FP layer (Ascend mega_moe page, A8W8-FP use case), fmt 0 for FLOAT8_E4M3FN and 1
 * for FLOAT8_E5M2: x FP8 codes [T, H] with UE8M0 scales [T, H/32]; w1 FP8 [E, 2I, H] with UE8M0
 * [E, 2I, H/32]; w2 FP8 [E, H, I] with UE8M0 [E, H, I/32] (output channel, then input; one scale per 32
 * along the contraction axis); g [T*K].
 *   GMM1: H = X_e . W1[e] on the decoded values, in double precision; SwiGLU in double precision;
 *   Q_MX of A to the same FP8 format (mx_requant); GMM2: Y = A~ . W2[e] in double precision;
 *   Token Combine as in the A16W16 layer.
 * a_codes_out [R, I] and a_exp_out [R, I/32], when not NULL, receive the re-quantised A per pool row.
 * Returns 0, -1 for a bad id or format, -2 when memory runs out. */
int oracle_forward_fp8(int fmt, const uint8_t* x, const uint8_t* x_scale, const int32_t* ids, const float* g,
                       const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                       int64_t T, int64_t K, int64_t E, int64_t H, int64_t I, double* y, uint8_t* a_codes_out,
                       uint8_t* a_exp_out) {
    if (fmt != 0 && fmt != 1) return -1;
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    int64_t* offsets = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    int64_t* row_src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * K > 0 ? T * K : 1));
    double* comb = (double*)calloc((size_t)(T * K * H > 0 ? T * K * H : 1), sizeof(double));
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* w1d = (double*)malloc(sizeof(double) * (size_t)(2 * I * H)); /* the expert's weights, decoded */
    double* w2d = (double*)malloc(sizeof(double) * (size_t)(H * I));
    int st = (counts && offsets && row_src && comb && xv && h && a && w1d && w2d) ? 0 : -2;
    if (st == 0) st = oracle_plan(ids, T, K, E, counts, offsets, row_src);
    for (int64_t e = 0; st == 0 && e < E; ++e) {
        if (offsets[e + 1] == offsets[e]) continue; /* no rows */
        for (int64_t j = 0; j < 2 * I; ++j)         /* decode W1[e] and W2[e] to their values once */
            for (int64_t k = 0; k < H; ++k)
                w1d[j * H + k] = fp8_value(fmt, w1[(e * 2 * I + j) * H + k]) *
                                 ue8m0_value(w1_scale[(e * 2 * I + j) * (H / 32) + k / 32]);
        for (int64_t c = 0; c < H; ++c)
            for (int64_t j = 0; j < I; ++j)
                w2d[c * I + j] = fp8_value(fmt, w2[(e * H + c) * I + j]) * ue8m0_value(w2_scale[(e * H + c) * (I / 32) + j / 32]);
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const int64_t src = row_src[p], tok = src / K;
            for (int64_t k = 0; k < H; ++k)
                xv[k] = fp8_value(fmt, x[tok * H + k]) * ue8m0_value(x_scale[tok * (H / 32) + k / 32]);
            for (int64_t j = 0; j < 2 * I; ++j) { /* GMM1 */
                double s = 0.0;
                for (int64_t k = 0; k < H; ++k) s += xv[k] * w1d[j * H + k];
                h[j] = s;
            }
            for (int64_t j = 0; j < I; ++j) /* SwiGLU */
                a[j] = h[j] / (1.0 + exp(-h[j])) * h[I + j];
            mx_requant(a, I, fmt, a_codes_out ? a_codes_out + p * I : NULL, a_exp_out ? a_exp_out + p * (I / 32) : NULL);
            for (int64_t c = 0; c < H; ++c) { /* GMM2, gate, the bf16 combine row */
                double s = 0.0;
                for (int64_t j = 0; j < I; ++j) s += a[j] * w2d[c * I + j];
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
    free(w1d);
    free(w2d);
    return st;
}

/* The e5m2 encoder on its own, for the codec test. */
uint8_t oracle_e5m2_encode(double v) { return e5m2_encode(v); }

/* The e4m3 encoder on its own, for the codec test. */
uint8_t oracle_e4m3_encode(double v) { return e4m3_encode(v); }
