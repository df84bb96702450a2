/*
 * Host check of the division method the FP8 and 4-bit quantizer kernels use
 * (rowquant.cuh, nvfp4.cu): with y = fl(1 / b) correctly rounded and
 * q0 = fl(a * y), the residual r = fma(-q0, b, a) is exact and
 * q1 = fma(r, y, q0) is the correctly rounded quotient fl(a / b)
 * (Markstein's theorem for FMA-based division, round to nearest) while the
 * residual does not underflow.  The kernels use it for scales b in
 * [2^-80, 2^100], where every quotient that can give a nonzero code (2^-11
 * and up) has |a| >= 2^-91.  Compares q1 with the IEEE quotient for n seeded
 * random pairs in that domain (quotients from 2^-12 to 2^10); prints the
 * number of mismatches.  Usage: fma_quotient_check n seed
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint64_t st;
static uint64_t next(void) {
    st ^= st << 13;
    st ^= st >> 7;
    st ^= st << 17;
    return st;
}
static float from_bits(uint32_t b) {
    float f;
    memcpy(&f, &b, 4);
    return f;
}
static uint32_t bits(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    return b;
}

int main(int argc, char** argv) {
    long long n = argc > 1 ? atoll(argv[1]) : 1000000;
    st = argc > 2 ? strtoull(argv[2], NULL, 10) * 2654435761ull + 1 : 1;
    long long bad = 0;
    for (long long i = 0; i < n; ++i) {
        uint64_t r = next();
        uint32_t mb = (uint32_t)(r & 0x7FFFFF);
        if ((i & 15) == 0) mb = 0x7FFFFF; /* all-ones significands */
        if ((i & 15) == 1) mb = 0;
        int eb = 47 + (int)((r >> 23) % 180); /* scales in [2^-80, 2^100) */
        float b = from_bits(((uint32_t)eb << 23) | mb);
        uint32_t ma = (uint32_t)((r >> 30) & 0x7FFFFF);
        if ((i & 7) == 2) ma = 0x7FFFFF;
        int ea = eb + 9 - (int)((r >> 53) % 22); /* |a / b| in [2^-12, 2^11) */
        if (ea < 1) continue;
        float a = from_bits(((uint32_t)ea << 23) | ma | ((uint32_t)(r >> 63) << 31));
        float y = 1.0f / b;
        float q0 = a * y;
        float res = fmaf(-q0, b, a);
        float q1 = fmaf(res, y, q0);
        if (bits(q1) != bits(a / b)) ++bad;
    }
    printf("%lld\n", bad);
    return 0;
}
