/* Host check of the V encoder's arithmetic (test infrastructure).
 *
 * The V^T encoder forms the E4M3 code of fl(x / sv) without a division:
 * with nr = -fl(1/sv), z = fl(x nr), r = fma(z, sv, x) and y = fma(r, nr, z),
 * the code of fl(x / sv) is the code of y with its sign bit flipped
 * (Markstein's correction step for correctly rounded quotients, IBM J. Res.
 * Dev. 34(1), 1990, with the reciprocal negated so that signed zeros come
 * out right).  The kernel takes this path for sv in [2^-100, 2^125].
 *
 * For each positive finite bf16 amax in the chosen set, sv = fl(amax / 448)
 * as the kernel forms it, and for every bf16 x with |x| <= amax, this
 * compares that code with the oracle's E4M3 code of the IEEE quotient
 * fl(x / sv) and prints "pairs N differ D".
 *
 *   v_quotient_check sample   every amax mantissa at a spread of exponents,
 *                             the range's end binades included
 *   v_quotient_check all      every positive finite bf16 amax (about 1e9 pairs)
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

uint8_t oracle_e4m3_encode(float y);

static float bf16_value(uint32_t bits) {
    uint32_t u = bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int in_sample(uint32_t amax_bits) {
    /* bf16 exponent field e (amax ~ 2^(e - 127)); sv ~ amax / 448 ~ 2^(e - 136). */
    static const int exps[] = {36, 37, 38, 39, 60, 100, 120, 127, 128, 131, 140, 160, 200, 250, 254};
    int e = (int)(amax_bits >> 7) & 0xFF;
    for (unsigned k = 0; k < sizeof exps / sizeof exps[0]; ++k)
        if (e == exps[k]) return 1;
    return 0;
}

int main(int argc, char **argv) {
    const int all = argc > 1 && strcmp(argv[1], "all") == 0;
    long long pairs = 0, differ = 0;
    for (uint32_t ab = 0x0001; ab < 0x7F80; ++ab) {
        if (!all && !in_sample(ab)) continue;
        const float amax = bf16_value(ab);
        const float sv = amax / 448.0f;
        if (!(sv >= 0x1p-100f && sv <= 0x1p125f)) continue;
        const float nr = -(1.0f / sv);
        for (uint32_t xb = 0; xb < 0x10000; ++xb) {
            const float x = bf16_value(xb);
            if (!(fabsf(x) <= amax)) continue;
            volatile float z = x * nr;
            volatile float r = fmaf(z, sv, x);
            volatile float y = fmaf(r, nr, z);
            const uint8_t got = (uint8_t)(oracle_e4m3_encode(y) ^ 0x80);
            const uint8_t want = oracle_e4m3_encode(x / sv);
            ++pairs;
            if (got != want) {
                if (++differ <= 5)
                    printf("amax %a sv %a x %a: %02x, division %02x\n", amax, sv, x, got, want);
            }
        }
    }
    printf("pairs %lld differ %lld\n", pairs, differ);
    return differ != 0;
}
