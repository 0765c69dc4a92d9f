/* Exhaustive check of the divisions the FP8 dispatch kernel does without a
 * divide instruction.
 * 1. The scale: with y448 = RN(1/448), q0 = RN(amax*y448),
 *    r = RN(amax - q0*448) (fmaf), RN(q0 + r*y448) must equal the IEEE
 *    quotient amax/448 bit for bit, for every finite bf16 amax >= 0.
 * 2. The codes, for groups with amax >= 2^-60: with s = RN(amax/448) and
 *    y = RN(1/s), q = copysign(RN(q0 + r*y), x), q0 = RN(x*y),
 *    r = RN(x - q0*s) (fmaf), must give the same E4M3 code as the IEEE
 *    quotient RN(x/s), for every bf16 x with |x| <= amax and every bf16
 *    amax >= 2^-60 (Markstein's correction; the remainder is exact while it
 *    stays a normal number).  Codes come from the oracle's encoder.
 * Test infrastructure: links oracle/ep_oracle.c.  Arguments: amax stride
 * (1 = every amax).  Prints "pairs N mismatches M scale_mismatches K". */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

uint8_t ep_oracle_f32_to_e4m3(float v);

static float bf16(uint32_t h) { uint32_t u = h << 16; float f; memcpy(&f, &u, 4); return f; }

int main(int argc, char **argv) {
    const uint32_t stride = argc > 1 ? (uint32_t)atoi(argv[1]) : 1u;
    const float lim = ldexpf(1.0f, -60);
    long long pairs = 0, bad = 0;
    for (uint32_t ah = 0x0001; ah < 0x7f80; ah += stride) {
        const float amax = bf16(ah);
        if (amax < lim) continue;
        const float s = amax / 448.0f;
        const float y = 1.0f / s;
        for (uint32_t xh = 0; xh < 0x7f80; ++xh) {
            const float xa = bf16(xh);
            if (xa > amax) break; /* positive bf16 values grow with their bits */
            for (int sg = 0; sg < 2; ++sg) {
                const float x = sg ? -xa : xa;
                const float ref = x / s;
                const float q0 = x * y;
                const float r = fmaf(-q0, s, x);
                const float q = copysignf(fmaf(r, y, q0), x);
                ++pairs;
                if (memcmp(&q, &ref, 4) != 0 && ep_oracle_f32_to_e4m3(q) != ep_oracle_f32_to_e4m3(ref)) {
                    if (bad < 5) printf("mismatch amax=%a x=%a ieee=%a fast=%a\n", amax, x, ref, q);
                    ++bad;
                }
            }
        }
    }
    long long scale_bad = 0;
    const float y448 = 1.0f / 448.0f;
    for (uint32_t ah = 0; ah < 0x7f80; ++ah) {
        const float amax = bf16(ah);
        const float ref = amax / 448.0f;
        const float q0 = amax * y448;
        const float r = fmaf(-q0, 448.0f, amax);
        const float q = copysignf(fmaf(r, y448, q0), amax);
        if (memcmp(&q, &ref, 4) != 0) {
            if (scale_bad < 5) printf("scale mismatch amax=%a ieee=%a fast=%a\n", amax, ref, q);
            ++scale_bad;
        }
    }
    printf("pairs %lld mismatches %lld scale_mismatches %lld\n", pairs, bad, scale_bad);
    return bad != 0 || scale_bad != 0;
}
