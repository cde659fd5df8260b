/*
 * Exhaustive check of the quantizer's division method against IEEE division.
 *
 * The GPU quantizer computes x / s (s = fl32(amax / 448), one per tile) as
 *   r = RN(1 / s);  q0 = RN(x * r);  e = RN(q0 * s - x);  q = RN(q0 - e * r)
 * (a reciprocal plus one exact-residual correction, Markstein 1990) when the
 * tile's amax >= 2^-90, and with an IEEE divide otherwise. Inputs are bf16,
 * so every (amax, x) pair with |x| <= amax can be enumerated: for amax >= 2^-90
 * this program checks that q equals the IEEE quotient bit for bit whenever
 * |x / s| >= 2^-12, and that smaller quotients keep the IEEE sign and stay
 * below 2^-11 (every such value encodes to the same signed E4M3 zero).
 * It also checks the tile scale s = amax / 448, computed the same way with
 * the constant reciprocal RN(1/448), against the IEEE quotient for every
 * finite non-negative bf16 amax.
 * Prints "pairs mismatches scale_mismatches" and exits 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_to_f32(uint32_t h) {
    uint32_t u = h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

int main(void) {
    const float min_amax = 0x1p-90f;
    long long pairs = 0, bad = 0;
#pragma omp parallel for reduction(+ : pairs, bad) schedule(dynamic, 64)
    for (uint32_t ab = 1; ab < 0x7F80; ++ab) { /* every finite positive bf16 amax */
        const float amax = bf16_to_f32(ab);
        if (amax < min_amax) continue;
        const float s = amax / 448.0f;
        const float r = 1.0f / s;
        for (uint32_t xb = 0; xb <= ab; ++xb) {
            for (int neg = 0; neg < 2; ++neg) {
                const float x = neg ? -bf16_to_f32(xb) : bf16_to_f32(xb);
                const float ref = x / s;
                const float q0 = x * r;
                const float e = fmaf(q0, s, -x);
                const float q = fmaf(-e, r, q0);
                ++pairs;
                if (fabsf(ref) >= 0x1p-12f) {
                    if (bits(q) != bits(ref)) ++bad;
                } else if (signbit(q) != signbit(ref) || fabsf(q) >= 0x1p-11f) {
                    ++bad;
                }
            }
        }
    }
    long long scale_bad = 0;
    const float r448 = 1.0f / 448.0f;
    for (uint32_t ab = 0; ab < 0x7F80; ++ab) {
        const float amax = bf16_to_f32(ab);
        const float q0 = amax * r448;
        const float e = fmaf(q0, 448.0f, -amax);
        const float s = fmaf(-e, r448, q0);
        if (bits(s) != bits(amax / 448.0f)) ++scale_bad;
    }
    printf("%lld %lld %lld\n", pairs, bad, scale_bad);
    return 0;
}
