/*
 * oracle.c -- plain, single-threaded CPU oracle for the FP8 block-scaled linear path.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's CPU
 * baseline; never by the product path. It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * The oracle follows the pages' steps in their order and writes each rounding out:
 *   - e4m3fn values come from the format's bit fields; the encoder picks the nearest code by
 *     brute force over the finite codes (ties to the even code) and saturates at +-448,
 *     the largest e4m3fn magnitude ("DeepSeek-V3 Administrator & Developer Guide",
 *     §8.5.1: "448.0 is the maximum representable magnitude in e4m3fn").
 *   - A binary32 division is formed in binary64 and rounded once to binary32. Because
 *     53 >= 2*24 + 2, this double rounding is innocuous (S. Figueroa, "When is double
 *     rounding innocuous?", SIGNUM Newsletter 30(3), 1995): the result is the correctly
 *     rounded binary32 quotient, i.e. what an IEEE binary32 divide returns.
 *   - A binary32 product of an e4m3 value (4 significant bits) and a binary32 scale
 *     (24 bits) is exact in binary64 (28 bits), so rounding it once to binary32 gives the
 *     correctly rounded binary32 product.
 *   - The GEMM is accumulated entirely in binary64; each 128-long block sum of e4m3 products
 *     is exact there (products span 2^-18 .. 2^17.6, so 128 of them need < 53 bits).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

/* ---------------------------------------------------------------- e4m3fn codec ---- */

/* e4m3fn: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0. Exponent field 0
   holds the subnormals mant * 2^-9; S.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exp_field = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (exp_field == 0xF && mant == 0x7) return NAN;
    if (exp_field == 0)
        mag = ldexp((double)mant, -9);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, exp_field - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even, saturating (satfinite) conversion of a binary32 value to e4m3fn.
   NaN -> 0x7F. |v| >= 448 (including infinity) -> sign | 0x7E. Otherwise the finite
   non-negative code nearest |v|, the even code on a tie, with v's sign bit (so -0 and
   negative values that round to zero give 0x80). */
uint8_t oracle_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* values of the finite non-negative codes 0x00..0x7E, filled on first use */
    static double code_value[0x7F];
    static int have_values = 0;
    if (!have_values) {
        for (int c = 0; c <= 0x7E; ++c) code_value[c] = oracle_e4m3_decode((uint8_t)c);
        have_values = 1;
    }
    int best = 0;
    double best_err = a; /* distance to code 0x00 (value 0) */
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(code_value[c] - a);
        /* adjacent codes tie only at their midpoint: take the one with even mantissa LSB */
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------- bf16 --------------- */

float oracle_bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Nearest bf16 to f, ties to the even pattern. The two candidates are the bf16 patterns
   that bracket f (truncation of f's bits, and the next one away from zero); their values
   and f are compared in binary64. NaN stays a quiet NaN. */
uint16_t oracle_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040);
    uint16_t lo = (uint16_t)(u >> 16);       /* toward zero */
    if ((u & 0xFFFFu) == 0) return lo;       /* already a bf16 value */
    uint16_t hi = (uint16_t)(lo + 1);        /* away from zero (may become infinity) */
    double v = fabs((double)f);
    double vlo = fabs((double)oracle_bf16_to_float(lo));
    double vhi = fabs((double)oracle_bf16_to_float(hi));
    double elo = v - vlo, ehi = vhi - v;
    if (elo < ehi) return lo;
    if (ehi < elo) return hi;
    return (lo & 1) ? hi : lo;
}

/* ---------------------------------------------------------------- arithmetic -------- */

float oracle_f32_div(float a, float b) { return (float)((double)a / (double)b); }

/* Smallest power of two >= s (s > 0, finite): 2^ceil(log2 s), exact. frexp gives
   s = f * 2^e with f in [0.5, 1); s is a power of two exactly when f == 0.5. */
static float pow2_ceil(float s) {
    int e;
    double f = frexp((double)s, &e);
    if (f == 0.5) return s;
    return (float)ldexp(1.0, e);
}

/* ---------------------------------------------------------------- act_quant --------- */

/* "DeepSeek-V3 Administrator & Developer Guide", §8.5.1 act_quant_kernel: per 128-element
   block along K, load as float32, take the absolute max, clamp it to 1e-4, divide by 448 to
   get the scale s; with scale_fmt "ue8m0" round s up to a power of two (2^ceil(log2 s);
   "DeepSeek-V3 User Guide", FAQ on ue8m0); then y = x / s cast to float8_e4m3fn; store y, s. */
void oracle_act_quant(const uint16_t* x, uint8_t* y, float* s, int64_t M, int64_t K,
                      int scale_fmt) {
    const int64_t nblk = K / ORACLE_BLOCK;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nblk; ++b) {
            const uint16_t* xb = x + m * K + b * ORACLE_BLOCK;
            uint8_t* yb = y + m * K + b * ORACLE_BLOCK;
            float amax = 0.0f;
            for (int j = 0; j < ORACLE_BLOCK; ++j) {
                float v = fabsf(oracle_bf16_to_float(xb[j]));
                if (v > amax) amax = v;
            }
            float clamped = amax > 1e-4f ? amax : 1e-4f;
            float sc = oracle_f32_div(clamped, 448.0f);
            if (scale_fmt == ORACLE_SCALE_UE8M0) sc = pow2_ceil(sc);
            for (int j = 0; j < ORACLE_BLOCK; ++j)
                yb[j] = oracle_e4m3_encode(oracle_f32_div(oracle_bf16_to_float(xb[j]), sc));
            s[m * nblk + b] = sc;
        }
    }
}

/* ---------------------------------------------------------------- weight_dequant ---- */

/* "DeepSeek-V3 Administrator & Developer Guide", §8.5.2 weight_dequant_kernel and §6.3:
   one fp32 scale per 128x128 block (scale tensor (ceil(N/128), ceil(K/128))); the e4m3 value
   is loaded as float32, multiplied by its block's scale and stored as bf16. */
void oracle_weight_dequant(const uint8_t* w, const float* s, uint16_t* y, int64_t N,
                           int64_t K) {
    const int64_t kblk = (K + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            double sc = (double)s[(n / ORACLE_BLOCK) * kblk + k / ORACLE_BLOCK];
            float prod = (float)(oracle_e4m3_decode(w[n * K + k]) * sc);
            y[n * K + k] = oracle_bf16_rne(prod);
        }
    }
}

/* ---------------------------------------------------------------- fp8_gemm ---------- */

/* "DeepSeek-V3 Administrator & Developer Guide", §8.5.3 fp8_gemm_kernel: C = A B^T where each
   128-wide K block's partial dot product is multiplied by a_s (per row, per K block) and b_s
   (per 128x128 block of B) and accumulated. Here every step is binary64. */
static double gemm_one(const uint8_t* a, const float* a_s, const uint8_t* b, const float* b_s,
                       const double* dec, int64_t m, int64_t n, int64_t K) {
    const int64_t nkb = K / ORACLE_BLOCK;
    const uint8_t* arow = a + m * K;
    const uint8_t* brow = b + n * K;
    double acc = 0.0;
    for (int64_t kb = 0; kb < nkb; ++kb) {
        double p = 0.0;
        for (int64_t k = kb * ORACLE_BLOCK; k < (kb + 1) * ORACLE_BLOCK; ++k)
            p += dec[arow[k]] * dec[brow[k]];
        double sa = (double)a_s[m * nkb + kb];
        double sb = (double)b_s[(n / ORACLE_BLOCK) * nkb + kb];
        acc += p * sa * sb;
    }
    return acc;
}

static void decode_table(double* dec) {
    for (int c = 0; c < 256; ++c) dec[c] = oracle_e4m3_decode((uint8_t)c);
}

void oracle_gemm(const uint8_t* a, const float* a_s, const uint8_t* b, const float* b_s,
                 double* c, int64_t M, int64_t N, int64_t K) {
    double dec[256];
    decode_table(dec);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) c[m * N + n] = gemm_one(a, a_s, b, b_s, dec, m, n, K);
}

void oracle_gemm_at(const uint8_t* a, const float* a_s, const uint8_t* b, const float* b_s,
                    const int64_t* mi, const int64_t* ni, int64_t count, double* out,
                    int64_t M, int64_t N, int64_t K) {
    double dec[256];
    decode_table(dec);
    (void)M;
    (void)N;
    for (int64_t i = 0; i < count; ++i) out[i] = gemm_one(a, a_s, b, b_s, dec, mi[i], ni[i], K);
}
