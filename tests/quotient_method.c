/*
 * The quotient correction the fp8 quantiser uses, checked in plain C against
 * IEEE division (gcc, -ffp-contract=off; fmaf is the IEEE fused
 * multiply-add): with rd = RN(1/d), q0 = RN(x*rd), r = fma(-q0, d, x) and
 * q = RN(q0 + r*rd) (also one fma), q must equal RN(x/d) for
 *   - d = 448 and every x = max(amax, 1e-4) over all finite bf16 amax >= 0;
 *   - d = every block scale RN(max(amax, 1e-4)/448) of a bf16 amax, and x over
 *     a stride of the finite bf16 values with |x| <= amax and |x/d| >= 2^-10;
 *   - a stride of scales against every finite bf16 x in that range.
 * Prints the number of pairs checked and of mismatches.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_value(uint32_t bits)
{
    uint32_t w = bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

static uint32_t bits_of(float f)
{
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return w;
}

static float corrected(float x, float d, float rd)
{
    float q0 = x * rd;
    float r = fmaf(-q0, d, x);
    return copysignf(fmaf(r, rd, q0), x);
}

int main(void)
{
    const float r448 = 1.0f / 448.0f;
    unsigned long long pairs = 0, bad = 0;
    for (uint32_t mb = 0; mb <= 0x7F7F; ++mb) {
        float m = bf16_value(mb);
        float a = m > 1e-4f ? m : 1e-4f;
        float s = a / 448.0f;
        ++pairs;
        if (bits_of(corrected(a, 448.0f, r448)) != bits_of(s)) ++bad;
        float rs = 1.0f / s;
        uint32_t stride = (mb % 61 == 0) ? 1 : 7;
        for (uint32_t xb = 0; xb < 0x10000; xb += stride) {
            float x = bf16_value(xb);
            if (!isfinite(x) || fabsf(x) > m) continue;
            float q = x / s;
            if (fabsf(q) < 0x1p-10f) continue;
            ++pairs;
            if (bits_of(corrected(x, s, rs)) != bits_of(q)) ++bad;
        }
    }
    printf("pairs=%llu mismatches=%llu\n", pairs, bad);
    return 0;
}
