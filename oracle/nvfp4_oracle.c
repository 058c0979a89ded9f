/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the small-M NVFP4 W4A4 linear.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * What it computes (source: "ReSET: Accurate Latency-Critical NVFP4 Reasoning
 * via Step-Aware Temperature Scaling", abstract, and the ReSET README,
 * "Core components" item 2): the linear layer Y[M,N] = X[M,K] . W[N,K]^T of
 * latency-critical decode, with both operands in NVFP4 ("W4A4") and M <= 8.
 * The pages name the format but do not define its bits, its scales or its
 * rounding.  This file fixes the plainest public reading, step by step:
 *
 *   E2M1   4 bits: sign | 2 exponent bits (bias 1) | 1 mantissa bit.
 *          Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (OCP microscaling FP4).
 *   E4M3   8 bits, the "FN" variant: sign | 4 exponent bits (bias 7) |
 *          3 mantissa bits, subnormals at exponent 0, S.1111.111 = NaN,
 *          no infinity, largest finite 448 (OCP FP8).
 *   Block  one E4M3 scale per 16 consecutive elements along K.
 *   Global one FP32 per-tensor scale g = amax(|T|) / (6 * 448).
 *
 * Quantisation recipe, applied alike to W and X (all FP32 ops correctly
 * rounded, no fused multiply-add):
 *   1. g given (weights: amax / 2688 computed here; activations: an input).
 *   2. per row r and 16-block b: bmax = max |t|;  s = bmax / (6 * g)
 *      with 6 * g rounded to FP32 first.  If 6 * g == 0 the scale is 0.
 *   3. sc = E4M3 round-to-nearest-even, saturating at 448.
 *   4. S  = dec(sc) * g in FP32.  If S == 0 every element is a signed zero.
 *   5. q  = E2M1 round-to-nearest-even of t / S, saturating at 6.  The sign
 *      of t is kept, also when the magnitude rounds to 0 (-0 -> code 0x8).
 *   6. element 2j goes in the low nibble of byte j, 2j+1 in the high nibble.
 * GEMM (FP64 throughout; every decoded value is exact in double):
 *   y[m,n] = gX * gW * sum_b dec(sx[m,b]) * dec(sw[n,b])
 *                        * sum_{i in b} e2m1(qx[m,i]) * e2m1(qw[n,i]).
 *
 * Encoders are brute force: every finite code is decoded by its closed form
 * and the nearest one wins; on an exact tie the code with mantissa LSB 0
 * (the even code) wins.  That is round-to-nearest-even read off the grid,
 * with no bit tricks to get wrong.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no -ffast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- element formats ---------------------------------------------------- */

/* E2M1 closed form: e = bits 2..1, m = bit 0; e == 0 is subnormal (m * 0.5),
 * else 2^(e-1) * (1 + m/2).  Bit 3 is the sign. */
double oracle_e2m1_value(int code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* E4M3 (FN) closed form: e = bits 6..3, m = bits 2..0; e == 0 is subnormal
 * m/8 * 2^-6, else (1 + m/8) * 2^(e-7); exponent and mantissa all ones is
 * NaN.  Bit 7 is the sign. */
double oracle_e4m3_value(int code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp(m / 8.0, -6);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest E2M1 code to v by exhaustive search over the 8 magnitudes, ties to
 * the even code, saturating at 6 (the nearest finite value beyond the grid). */
int oracle_e2m1_encode(float v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    int best = 0;
    double best_d = INFINITY;
    if (a >= 6.0) /* saturate: 6 is the nearest finite magnitude; also keeps
                     huge inputs out of the distance search, where the FP64
                     differences would all round to the same number */
        return (neg << 3) | 7;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - oracle_e2m1_value(c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (neg << 3) | best;
}

/* Nearest non-negative finite E4M3 code to s >= 0 (codes 0x00..0x7E), ties to
 * the even code; anything at or above the largest finite value maps to it. */
int oracle_e4m3_encode(float s)
{
    double a = (double)s;
    int best = 0;
    double best_d = INFINITY;
    if (!(a >= 0.0))
        return 0; /* negative or NaN never reach here; define as 0 */
    if (a >= oracle_e4m3_value(0x7E))
        return 0x7E;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(a - oracle_e4m3_value(c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* ---- per-tensor scale --------------------------------------------------- */

float oracle_amax(const float* t, int64_t count)
{
    float a = 0.0f;
    for (int64_t i = 0; i < count; ++i) {
        float v = fabsf(t[i]);
        if (v > a)
            a = v;
    }
    return a;
}

/* g = amax / (6 * 448) in FP32. */
float oracle_global_scale(const float* t, int64_t count)
{
    return oracle_amax(t, count) / 2688.0f;
}

/* ---- quantise one matrix (recipe steps 2..6) ------------------------------ */

void oracle_quantize(const float* t, int64_t rows, int64_t k, float g,
                     uint8_t* q, uint8_t* s)
{
    const int64_t nb = k / 16;
    const float six_g = 6.0f * g;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* blk = t + r * k + b * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float v = fabsf(blk[i]);
                if (v > bmax)
                    bmax = v;
            }
            int sc = 0;
            if (six_g > 0.0f) {
                float ratio = bmax / six_g;
                sc = oracle_e4m3_encode(ratio);
            }
            s[r * nb + b] = (uint8_t)sc;
            float S = (float)oracle_e4m3_value(sc) * g;
            for (int i = 0; i < 16; ++i) {
                int code;
                if (S == 0.0f) {
                    code = signbit(blk[i]) ? 8 : 0;
                } else {
                    float v = blk[i] / S;
                    code = oracle_e2m1_encode(v);
                }
                uint8_t* byte = q + r * (k / 2) + b * 8 + i / 2;
                if ((i & 1) == 0)
                    *byte = (uint8_t)((*byte & 0xF0) | code);
                else
                    *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
            }
        }
    }
}

/* Weight packing: global scale from the tensor itself, then quantise. */
void oracle_pack_weight(const float* w, int64_t n, int64_t k,
                        uint8_t* wq, uint8_t* ws, float* wg)
{
    float g = oracle_global_scale(w, n * k);
    *wg = g;
    oracle_quantize(w, n, k, g, wq, ws);
}

/* Dequantise to FP64: out[r,i] = e2m1(q) * e4m3(s) * g. */
void oracle_dequantize(const uint8_t* q, const uint8_t* s, float g,
                       int64_t rows, int64_t k, double* out)
{
    const int64_t nb = k / 16;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < k; ++i) {
            uint8_t byte = q[r * (k / 2) + i / 2];
            int code = (i & 1) ? (byte >> 4) : (byte & 15);
            out[r * k + i] = oracle_e2m1_value(code)
                           * oracle_e4m3_value(s[r * nb + i / 16]) * (double)g;
        }
}

/* ---- GEMM --------------------------------------------------------------- */

static double block_dot(const uint8_t* xq_row, const uint8_t* wq_row, int64_t b)
{
    double acc = 0.0;
    for (int i = 0; i < 16; ++i) {
        int64_t e = b * 16 + i;
        uint8_t xb = xq_row[e / 2], wb = wq_row[e / 2];
        int xc = (e & 1) ? (xb >> 4) : (xb & 15);
        int wc = (e & 1) ? (wb >> 4) : (wb & 15);
        acc += oracle_e2m1_value(xc) * oracle_e2m1_value(wc);
    }
    return acc;
}

/* One output element, from the packed bytes; rows [n0, n1) of the output
 * row m.  Used for full outputs on small shapes and for sampled outputs on
 * large ones. */
double oracle_gemm_one(const uint8_t* xq, const uint8_t* xs, float gx,
                       const uint8_t* wq, const uint8_t* ws, float gw,
                       int64_t k, int64_t m, int64_t n)
{
    const int64_t nb = k / 16;
    const uint8_t* xr = xq + m * (k / 2);
    const uint8_t* wr = wq + n * (k / 2);
    double acc = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        double scale = oracle_e4m3_value(xs[m * nb + b])
                     * oracle_e4m3_value(ws[n * nb + b]);
        acc += scale * block_dot(xr, wr, b);
    }
    return (double)gx * (double)gw * acc;
}

void oracle_gemm(const uint8_t* xq, const uint8_t* xs, float gx,
                 const uint8_t* wq, const uint8_t* ws, float gw,
                 int64_t m, int64_t n, int64_t k, double* y)
{
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            y[i * n + j] = oracle_gemm_one(xq, xs, gx, wq, ws, gw, k, i, j);
}

/* Sampled outputs: y[t] = element (ms[t], ns[t]). */
void oracle_gemm_sampled(const uint8_t* xq, const uint8_t* xs, float gx,
                         const uint8_t* wq, const uint8_t* ws, float gw,
                         int64_t k, const int64_t* ms, const int64_t* ns,
                         int64_t count, double* y)
{
    for (int64_t t = 0; t < count; ++t)
        y[t] = oracle_gemm_one(xq, xs, gx, wq, ws, gw, k, ms[t], ns[t]);
}

/* ---- BF16, the production activation and output dtype -------------------
 * BF16 is the upper half of an IEEE binary32: sign | 8 exponent bits | 7
 * mantissa bits.  Widening puts the 16 bits on top of 16 zero bits, which is
 * exact.  Narrowing (finite values below the largest BF16) takes the two
 * BF16 neighbours of v -- v's upper half (towards zero) and the next BF16
 * away from zero -- and keeps the nearer one, on an exact tie the one whose
 * last bit is 0: round-to-nearest-even, again read off the grid. */
float oracle_bf16_to_f32(uint16_t b)
{
    const uint32_t bits = (uint32_t)b << 16;
    float v;
    memcpy(&v, &bits, sizeof v);
    return v;
}

uint16_t oracle_f32_to_bf16(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, sizeof bits);
    const uint16_t lo = (uint16_t)(bits >> 16);
    const uint16_t hi = (uint16_t)(lo + 1);
    const double d = v;
    const double elo = fabs(d - (double)oracle_bf16_to_f32(lo));
    const double ehi = fabs((double)oracle_bf16_to_f32(hi) - d);
    if (elo < ehi)
        return lo;
    if (ehi < elo)
        return hi;
    return (lo & 1u) ? hi : lo;
}

void oracle_bf16_widen(const uint16_t* b, int64_t count, float* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = oracle_bf16_to_f32(b[i]);
}

void oracle_bf16_round(const float* v, int64_t count, uint16_t* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = oracle_f32_to_bf16(v[i]);
}
