/* Exhaustive check of the reciprocal refinement used by the SwiGLU kernels:
 * from a seed y0 within a few ulp of 1/d, two Newton-Raphson steps in
 * Markstein's residual form (e = fma(-d, y, 1); y = fma(y, e, y)), then
 * d = (2 - 2^-23) 2^k mapped to (1 + 2^-23) 2^-(k+1).  For every
 * significand of d in [1, 2) and every seed offset in [-R, R] ulp, the
 * result must equal the correctly rounded 1/d (IEEE division).  Prints the
 * number of mismatches; exit status 0 when there are none. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float refine(float d, float y)
{
    float e = fmaf(-d, y, 1.0f);
    y = fmaf(y, e, y);
    e = fmaf(-d, y, 1.0f);
    y = fmaf(y, e, y);
    const uint32_t bd = u_of(d);
    if ((bd & 0x7FFFFFu) == 0x7FFFFFu)
        y = f_of(0x7E800001u - (bd & 0x7F800000u));
    return y;
}

int main(int argc, char **argv)
{
    const int R = argc > 1 ? atoi(argv[1]) : 8;
    /* exponents: 0 (d in [1,2)) plus a few scaled binades up to 2^125 */
    const int ks[] = {0, 1, 17, 64, 100, 125};
    long bad = 0, n = 0;
    for (size_t ki = 0; ki < sizeof ks / sizeof ks[0]; ++ki) {
        const uint32_t step = ks[ki] == 0 ? 1u : 97u;  /* all significands in [1, 2) */
        for (uint32_t m = 0; m < (1u << 23); m += step) {
            const float d = f_of(((uint32_t)(127 + ks[ki]) << 23) | m);
            const float ref = 1.0f / d;
            for (int k = -R; k <= R; ++k) {
                const float y = refine(d, f_of(u_of(ref) + (uint32_t)k));
                ++n;
                if (u_of(y) != u_of(ref))
                    ++bad;
            }
        }
    }
    printf("%ld cases, %ld mismatches\n", n, bad);
    return bad != 0;
}
