/* The q8_1 quantizers' amax / 127 -- Markstein's correction for a known divisor: a quotient
 * q0 = a * RN(1/127), its exact residual a - 127 q0 by one fused multiply-add, and
 * q0 + residual * RN(1/127) by another -- against IEEE division, for every non-negative finite
 * binary32 value a (+inf is selected separately by the kernels).  Prints the mismatch count. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

int main(void)
{
    const float c = 1.0f / 127.0f;
    long long bad = 0;
#pragma omp parallel for reduction(+ : bad) schedule(static)
    for (long long u = 0; u < 0x7F800000LL; ++u) {
        const uint32_t b = (uint32_t)u;
        float a;
        memcpy(&a, &b, 4);
        const float ref = a / 127.0f;
        const float q0 = a * c;
        const float q1 = fmaf(fmaf(-q0, 127.0f, a), c, q0);
        uint32_t rb, qb;
        memcpy(&rb, &ref, 4);
        memcpy(&qb, &q1, 4);
        if (rb != qb) ++bad;
    }
    printf("mismatches %lld\n", bad);
    return 0;
}
