// Host check of the plan-time divisor magic (make_fastdiv): floor(n / d) by multiply-high
// and shift against hardware division, for every d up to 70000 at random n, multiples of d
// and their neighbours, and divisors near powers of two up to 2^30.
#include "internal.h"
#include <cstdio>
#include <random>
using namespace convfwd;
static uint32_t mulhi(uint32_t a, uint32_t b) { return (uint32_t)(((uint64_t)a * b) >> 32); }
int main() {
    std::mt19937_64 rng(1);
    long long bad = 0, n_tests = 0;
    auto check = [&](uint32_t d, uint32_t n) {
        FastDiv f = make_fastdiv(d);
        uint32_t q = (mulhi(n, f.m) + n) >> f.s;
        ++n_tests;
        if (q != n / d) { if (bad < 5) printf("d=%u n=%u got %u want %u\n", d, n, q, n / d); ++bad; }
    };
    for (uint32_t d = 1; d <= 70000; ++d) {
        for (uint32_t k = 0; k < 40; ++k) {
            uint32_t n = (uint32_t)(rng() & 0x7FFFFFFFu);
            check(d, n);
            uint32_t mult = (uint32_t)(rng() % (0x7FFFFFFFu / d + 1)) * d;   // a multiple of d and its neighbours
            check(d, mult); if (mult) check(d, mult - 1); if (mult + 1 < 0x80000000u) check(d, mult + 1);
        }
        check(d, 0x7FFFFFFFu); check(d, d - 1); check(d, d);
    }
    for (int e = 16; e < 31; ++e) for (int k = -3; k <= 3; ++k) {
        uint32_t d = (1u << e) + k;
        for (int j = 0; j < 2000; ++j) check(d, (uint32_t)(rng() & 0x7FFFFFFFu));
        check(d, 0x7FFFFFFFu);
    }
    printf("%lld checks, %lld wrong\n", n_tests, bad);
    return bad != 0;
}
