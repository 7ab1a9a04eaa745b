// Host check of draft_verification_02_b300/csrc/fp64_exact.cuh: every
// integer form against the host's IEEE binary64 arithmetic (x86-64 SSE2 or
// AArch64 scalar: round to nearest-even, no fused operations), on random
// operands and on constructed exact ties.  Prints "mismatches N" and exits
// non-zero when N > 0.  Built and run by tests/test_fp64_exact.py.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cmath>
#include <random>

#include "fp64_exact.cuh"

using namespace sv;

static uint64_t bits_of(double x)
{
    uint64_t b;
    std::memcpy(&b, &x, 8);
    return b;
}


static uint32_t fbits_of(float x)
{
    uint32_t b;
    std::memcpy(&b, &x, 4);
    return b;
}

// The same operations as the kernel's host table (separate roundings).
static double latency_cost(int d)
{
    const double at_pow2[5] = {1.0, 1.2, 1.5, 2.0, 3.0};
    if (d <= 1)
        return at_pow2[0];
    if (d >= 16)
        return at_pow2[4];
    int k = 0;
    while ((2 << k) < d)
        ++k;
    const double frac = (double)(d - (1 << k)) / (double)(1 << k);
    volatile double rise = at_pow2[k + 1] - at_pow2[k];
    volatile double step = rise * frac;
    return at_pow2[k] + step;
}

static long mismatches = 0;

static void expect(uint64_t got, uint64_t want, const char *what, double a, double b)
{
    if (got != want) {
        if (mismatches < 10)
            std::printf("%s: %.17g op %.17g: got %016llx want %016llx\n", what, a, b,
                        (unsigned long long)got, (unsigned long long)want);
        ++mismatches;
    }
}

static void check_mul(double P, float c)
{
    Dbl a, b;
    if (!dbl_unpack(bits_of(P), a) || !flt_unpack(fbits_of(c), b))
        return;
    volatile double want = P * (double)c;
    uint64_t got;
    if (!dbl_pack(mul_round(a, b), got))
        return;  // outside the normal range: the kernel takes the hardware path
    expect(got, bits_of(want), "mul", P, c);
}

static void check_mul_int(double P, int d)
{
    Dbl a;
    if (!dbl_unpack(bits_of(P), a))
        return;
    volatile double want = P * (double)d;
    uint64_t got;
    if (!dbl_pack(mul_round(a, int_unpack((uint32_t)d)), got))
        return;
    expect(got, bits_of(want), "mul_int", P, d);
}

static void check_div(double x, double y)
{
    Dbl a, b;
    if (!dbl_unpack(bits_of(x), a) || !dbl_unpack(bits_of(y), b))
        return;
    volatile double want = x / y;
    uint64_t got;
    if (!dbl_pack(div_round(a, b, recip116(b.m)), got))
        return;
    expect(got, bits_of(want), "div", x, y);
}

static void check_add(double t, double c)
{
    // t is 0 or >= 1, c >= 1: both multiples of 2^-52
    volatile double want = t + c;
    const uint64_t got = add_units_round(t == 0.0 ? 0 : to_units(bits_of(t)), to_units(bits_of(c)));
    const uint64_t w = to_units(bits_of(want));
    if (got != w) {
        if (mismatches < 10)
            std::printf("add: %.17g + %.17g\n", t, c);
        ++mismatches;
    }
}

int main()
{
    std::mt19937_64 rng(12345);
    std::uniform_real_distribution<double> u01(0.0, 1.0);
    long n = 0;
    // products of confidences: P in (2^-60, 1], c in (0, 1]
    for (int i = 0; i < 2000000; ++i, ++n) {
        double P = std::ldexp(1.0 + u01(rng), -1 - (int)(rng() % 60));
        float c = (float)u01(rng);
        if (c == 0.f)
            c = 0.5f;
        check_mul(P, c);
        check_mul(P, 1.0f);
        check_mul_int(P, 1 + (int)(rng() % 32));
    }
    // constructed ties: c = 1 + 2^-23 and P's low 23 bits exactly half
    for (int i = 0; i < 200000; ++i, ++n) {
        uint64_t m = (1ull << 52) | (rng() & ((1ull << 52) - 1));
        m = (m & ~((1ull << 23) - 1)) | (1ull << 22);
        const double P = std::ldexp((double)m, -52 - 1 - (int)(rng() % 20));
        check_mul(P, 1.0f + 0x1p-23f);
        check_mul(P, 1.0f - 0x1p-24f);
    }
    // benefits: x / cost(d) for the table's costs, and random divisors in [1, 3]
    double costs[33];
    for (int d = 1; d <= 32; ++d)
        costs[d] = latency_cost(d);
    for (int i = 0; i < 2000000; ++i, ++n) {
        const double x = std::ldexp(1.0 + u01(rng), -(int)(rng() % 60) + 4);
        check_div(x, costs[1 + rng() % 32]);
        check_div(x, 1.0 + 2.0 * u01(rng));
    }
    // quotients landing exactly halfway: x = y * (q + 1/2 ulp) cannot be
    // formed in doubles, so exactness is shown by x = y * q exactly (a zero
    // remainder) for small-significand y
    for (int i = 0; i < 200000; ++i, ++n) {
        const double y = 1.0 + (double)(rng() % 64) / 64.0;
        const double q = 1.0 + (double)(rng() % (1ull << 40)) * 0x1p-40;
        const double x = y * q;  // exact: 7 + 41 significant bits
        check_div(x, y);
    }
    // admission sums: running totals of table costs, as the scheduler adds
    // them, up to the units path's bound (totals below 2^11)
    for (int i = 0; i < 20000; ++i) {
        double t = 0.0;
        for (int k = 0; k < 600; ++k, ++n) {
            const double c = costs[1 + rng() % 32];
            check_add(t, c);
            t = t + c;
        }
    }
    std::printf("checked %ld cases, mismatches %ld\n", n, mismatches);
    return mismatches ? 1 : 0;
}
