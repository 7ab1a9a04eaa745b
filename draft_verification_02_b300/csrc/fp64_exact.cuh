// fp64_exact.cuh - exact integer forms of the few IEEE binary64 operations
// the cost-unit D-cut scheduler takes (multiply, divide by a fixed divisor,
// add), each rounded to nearest-even exactly as the hardware's __dmul_rn,
// __ddiv_rn and __dadd_rn round.  B300's fp64 pipe has a small fraction of
// its fp32 rate and a long latency; these forms run on the 64-bit integer
// paths with short dependency chains.
//
// A positive normal double is m * 2^e with m in [2^52, 2^53).  A product or
// quotient is formed exactly (a 53 x 24-bit product, or a 56-bit quotient
// with its remainder) and rounded once to 53 significant bits; a result
// outside the normal range (and a subnormal operand) is reported, so that
// the caller can take the hardware path instead.  Compiled for the host too:
// the tests check every form against the host's IEEE arithmetic.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define SV_HD __host__ __device__ __forceinline__
#else
#define SV_HD inline
#endif

namespace sv {

struct Dbl {
    uint64_t m;  // in [2^52, 2^53)
    int e;       // value m * 2^e
};

SV_HD int clz64(uint64_t x)
{
#ifdef __CUDA_ARCH__
    return __clzll((long long)x);
#else
    return x ? __builtin_clzll(x) : 64;
#endif
}

SV_HD uint64_t mulhi64(uint64_t a, uint64_t b)
{
#ifdef __CUDA_ARCH__
    return __umul64hi(a, b);
#else
    return (uint64_t)(((unsigned __int128)a * b) >> 64);
#endif
}

// The double's fields: true for a positive normal value.
SV_HD bool dbl_unpack(uint64_t bits, Dbl &d)
{
    const int be = (int)((bits >> 52) & 0x7ff);
    if ((bits >> 63) || be == 0 || be == 0x7ff)
        return false;
    d.m = (bits & ((1ull << 52) - 1)) | (1ull << 52);
    d.e = be - 1075;
    return true;
}

// A positive normal float as m * 2^e with m in [2^23, 2^24); false otherwise.
SV_HD bool flt_unpack(uint32_t bits, Dbl &d)
{
    const int be = (int)((bits >> 23) & 0xff);
    if ((bits >> 31) || be == 0 || be == 0xff)
        return false;
    d.m = (bits & 0x7fffffu) | 0x800000u;
    d.e = be - 150;
    return true;
}

// A positive integer below 2^24 as m * 2^e with m in [2^23, 2^24).
SV_HD Dbl int_unpack(uint32_t v)
{
    const int up = clz64(v) - 40;  // 64 - 24
    return {(uint64_t)v << up, -up};
}

// The bits of m * 2^e; false when that is not a normal double.
SV_HD bool dbl_pack(const Dbl &d, uint64_t &bits)
{
    const int be = d.e + 1075;
    if (be < 1 || be > 2046)
        return false;
    bits = ((uint64_t)be << 52) | (d.m & ((1ull << 52) - 1));
    return true;
}

// p * 2^e (2^53 <= p < 2^64), plus a positive tail below one unit of p when
// `sticky`, rounded to 53 significant bits, ties to even.
SV_HD Dbl round53(uint64_t p, int e, bool sticky)
{
    const int s = 11 - clz64(p);  // bits below the 53 kept
    uint64_t m = p >> s;
    const uint64_t rem = p & ((1ull << s) - 1), half = 1ull << (s - 1);
    if (rem > half || (rem == half && (sticky || (m & 1)))) {
        if (++m == (1ull << 53))
            return {1ull << 52, e + s + 1};
    }
    return {m, e + s};
}

// a * b for b with a 24-bit significand (b.m in [2^23, 2^24)), rounded once.
// The exact product has 76 or 77 bits: with a.m = ah 2^32 + al it is
// (ah b) 2^32 + al b, two 32 x 32-bit products; then its top 53 bits and a
// remainder.
SV_HD Dbl mul_round(const Dbl &a, const Dbl &b)
{
    const uint32_t al = (uint32_t)a.m, ah = (uint32_t)(a.m >> 32), bm = (uint32_t)b.m;
    const uint64_t pl = (uint64_t)al * bm, ph = (uint64_t)ah * bm;  // < 2^56, < 2^45
    const uint64_t t = ph + (pl >> 32);
    const uint64_t hi = t >> 32;                                   // < 2^13
    const uint64_t lo = (t << 32) | (pl & 0xffffffffu);
    const int s = hi >> 12 ? 24 : 23;  // 77 or 76 bits
    uint64_t m = (hi << (64 - s)) | (lo >> s);
    const uint64_t rem = lo & ((1ull << s) - 1), half = 1ull << (s - 1);
    const int e = a.e + b.e + s;
    if (rem > half || (rem == half && (m & 1))) {
        if (++m == (1ull << 53))
            return {1ull << 52, e + 1};
    }
    return {m, e};
}

// floor((2^116 - 1) / y.m): with it, a quotient by y needs no division.
// Host only (a 128-bit division, once per divisor).
inline uint64_t recip116(uint64_t ym)
{
    return (uint64_t)((((unsigned __int128)1 << 116) - 1) / ym);
}

// x / y rounded once, given r = recip116(y.m).  t = x.m 2^55 / y.m lies in
// (2^54, 2^56); x.m * r / 2^61 is below t by less than 2^-8, so its floor is
// floor(t) or one less, and one exact remainder step settles it.  The
// remainder is below 2^54, so it is exact in wrapping 64-bit arithmetic.
SV_HD Dbl div_round(const Dbl &x, const Dbl &y, uint64_t r)
{
    const uint64_t lo = x.m * r, hi = mulhi64(x.m, r);
    uint64_t q = (hi << 3) | (lo >> 61);
    uint64_t rem = (x.m << 55) - q * y.m;
    if (rem >= y.m) {
        ++q;
        rem -= y.m;
    }
    return round53(q, x.e - y.e - 55, rem != 0);
}

// Values that are 0 or doubles in [1, 2^11) as integers in units of 2^-52
// (exact: such doubles are multiples of 2^-52): a + b rounded once to 53
// significant bits, in the same units.  Valid while a + b < 2^63 (below
// 2^11 in value): then at most 10 bits are rounded away, all in the low
// 32-bit word, which keeps the chain of an admission loop short.
SV_HD uint64_t add_units_round(uint64_t a, uint64_t b)
{
    const uint64_t s = a + b;
    const uint32_t hi = (uint32_t)(s >> 32), lo = (uint32_t)s;
    if (hi < (1u << 21))  // below 2^53: exact
        return s;
#ifdef __CUDA_ARCH__
    const int k = 11 - __clz(hi);  // bits below the 53 kept, 1..10
#else
    const int k = 11 - __builtin_clz(hi);
#endif
    const uint32_t unit = 1u << k, rem = lo & (unit - 1), half = unit >> 1;
    const uint64_t t = s - rem;
    return rem > half || (rem == half && (lo & unit)) ? t + unit : t;
}

// A double in [1, 2^11) in units of 2^-52.
SV_HD uint64_t to_units(uint64_t bits)
{
    Dbl d;
    if (!dbl_unpack(bits, d))
        return 0;
    return d.m << (d.e + 52);
}

}  // namespace sv
