/* Exhaustive host check of the quotient identity used by the act_quant kernel.
 *
 * For every bf16 block maximum `amax` (positive, finite) the kernel forms
 *     s = RN32(max(amax, 1e-4f) / 448)     (and, for ue8m0, s = 2^ceil(log2 s))
 *     r = RN32(1 / s)
 * and for every bf16 element x with |x| <= amax the quotient
 *     q0 = RN32(x r),  rem = RN32(x - q0 s) (one FMA),  q = RN32(q0 + rem r) (one FMA),
 * then ORs the sign bit of x into q. Every operation is symmetric in the sign of x, so x >= 0
 * and x = -0 cover both signs.
 *
 * Compared with the correctly rounded binary32 quotient RN32(x / s) (formed in binary64 and
 * rounded once, which is exact for binary32 operands):
 *   - wherever RN32(x / s) >= 2^-11 in magnitude the two must be bit-identical;
 *   - below that (the remainder can underflow for subnormal x) both must still be below 2^-10,
 *     half the smallest e4m3 subnormal, so both convert to a zero e4m3 code of x's sign.
 * Prints the counts and exits nonzero on any violation.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fopenmp quotient_check.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float kernel_quotient(float x, float s, float r) {
    float q0 = x * r;
    float rem = fmaf(-q0, s, x);
    float q = fmaf(rem, r, q0);
    return from_bits(to_bits(q) | (to_bits(x) & 0x80000000u));
}

static float pow2_ceil(float s) {
    uint32_t b = to_bits(s);
    if (b & 0x007FFFFFu) b = (b & 0xFF800000u) + 0x00800000u;
    return from_bits(b);
}

int main(void) {
    const float tiny = 0x1p-11f, zero_code = 0x1p-10f;
    long long checked = 0, exact = 0, small = 0, bad = 0;
    for (int fmt = 0; fmt < 2; ++fmt) {
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : checked, exact, small, bad)
        for (int a = 0x0001; a < 0x7F80; ++a) { /* positive finite bf16 amax */
            float amax = from_bits((uint32_t)a << 16);
            float clamped = amax > 1e-4f ? amax : 1e-4f;
            float s = (float)((double)clamped / 448.0);
            if (fmt == 1) s = pow2_ceil(s);
            float r = (float)(1.0 / (double)s);
            for (int xb = -1; xb <= a; ++xb) { /* -1 stands for x = -0 */
                float x = xb < 0 ? -0.0f : from_bits((uint32_t)xb << 16);
                float want = (float)((double)x / (double)s);
                float got = kernel_quotient(x, s, r);
                ++checked;
                if (fabsf(want) >= tiny) {
                    if (to_bits(want) == to_bits(got)) {
                        ++exact;
                    } else {
                        ++bad;
#pragma omp critical
                        printf("mismatch fmt=%d amax=%a x=%a want=%a got=%a\n", fmt, amax, x,
                               want, got);
                    }
                } else if (fabsf(got) < zero_code && signbit(got) == signbit(x)) {
                    ++small;
                } else {
                    ++bad;
#pragma omp critical
                    printf("small mismatch fmt=%d amax=%a x=%a want=%a got=%a\n", fmt, amax,
                           x, want, got);
                }
            }
        }
    }
    printf("checked %lld: identical %lld, below 2^-11 and zero-coded %lld, violations %lld\n",
           checked, exact, small, bad);
    return bad ? 1 : 0;
}
