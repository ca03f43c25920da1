/* The quantize kernel's scale division, (mx - mn) / 15, is computed as
 * q0 = x * RN(1/15) followed by one fused multiply-add correction with the
 * exact residual x - 15 q0.  This program compares that sequence with IEEE
 * division for every finite non-negative fp32 x and prints the number of
 * mismatches (expected: 0).  Build without contraction: -ffp-contract=off. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

int main(void) {
    const float c = 1.0f / 15.0f;
    unsigned long long bad = 0;
    for (uint64_t u = 0; u < 0x7F800000ull; ++u) {
        const uint32_t b = (uint32_t)u;
        float x;
        memcpy(&x, &b, sizeof x);
        const float ref = x / 15.0f;
        const float q0 = x * c;
        const float q1 = fmaf(fmaf(-q0, 15.0f, x), c, q0);
        if (q1 != ref) ++bad;
    }
    printf("%llu\n", bad);
    return 0;
}
