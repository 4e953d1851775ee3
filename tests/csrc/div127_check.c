/*
 * CPU proof of the quantizer's division by 127 (the device helper div127 in
 * the library): for every finite non-negative binary32 a, Markstein's
 * correction step from r = RN(1/127),
 *     q0 = RN(a r),  rem = fma(-q0, 127, a),  q = fma(rem, r, q0),
 * equals the IEEE quotient RN(a / 127).  The arithmetic is IEEE binary32 with
 * round to nearest even and no flush to zero on both the host and the GPU
 * (the device helper uses __fmul_rn / __fmaf_rn), so this exhaustive check
 * covers the device as well.  Prints the number of mismatches (0 expected)
 * and the first one.  Build: gcc -O2 -ffp-contract=off -fopenmp div127_check.c -lm
 * (P. Markstein, "Computation of elementary functions on the IBM RISC
 * System/6000 processor", IBM J. Res. Develop. 34(1), 1990.)
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float as_f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t as_u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

int main(void)
{
    const float r = 0x1.020408p-7f; /* RN(1/127) */
    unsigned long long bad = 0;
    uint32_t first = 0xFFFFFFFFu;
#pragma omp parallel for schedule(static) reduction(+ : bad) reduction(min : first)
    for (long long i = 0; i <= 0x7F7FFFFFLL; ++i) {
        const uint32_t u = (uint32_t)i;
        const float a = as_f(u);
        const float ref = a / 127.0f;
        const float q0 = a * r;
        const float q = fmaf(fmaf(-q0, 127.0f, a), r, q0);
        if (as_u(q) != as_u(ref)) {
            ++bad;
            if (u < first) first = u;
        }
    }
    printf("%llu %08x\n", bad, bad ? first : 0u);
    return 0;
}
