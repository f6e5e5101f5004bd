// Host-side check of the invariant-divisor division used by the cost builder:
// compares nest::divide / nest::divide_up with the C++ operators on edge values
// (including both sides of 2^41, where the multiplier's long division changes from
// three 64-bit steps to bit by bit) and on random values across the ranges the
// solver uses.
#include <cstdint>
#include <cstdio>
#include <random>

#include "../../memory_aware_device_gb300/csrc/nest_divide.cuh"

int main() {
    std::mt19937_64 rng(12345);
    const uint64_t edge_d[] = {1, 2, 3, 5, 7, 10, 999, 1000, 1001, 1024, 4095, 4096, 4097, 6250, 12500, 25000,
                               50000, 900000, (1ull << 20) - 1, 1ull << 20, (1ull << 40) - 1, 1ull << 40,
                               (1ull << 40) + 1, (1ull << 41) - 1, 1ull << 41, (1ull << 41) + 1,
                               (1ull << 63) - 1, 1ull << 63, ~0ull};
    const uint64_t edge_n[] = {0, 1, 2, 999, 1000, 1001, (1ull << 32) - 1, 1ull << 32, (1ull << 59) + 12345,
                               (1ull << 62) - 1, (1ull << 63) - 1, 1ull << 63, ~0ull - 1, ~0ull};
    long bad = 0, count = 0;
    auto check = [&](uint64_t n, uint64_t d) {
        const nest::Divisor v = nest::make_divisor(d);
        count++;
        if (nest::divide(n, v) != n / d) {
            if (bad++ < 10) std::printf("divide(%llu, %llu) wrong\n", (unsigned long long)n, (unsigned long long)d);
        }
        if (n <= ~0ull - d + 1 && nest::divide_up(n, d, v) != n / d + (n % d != 0)) {
            if (bad++ < 10) std::printf("divide_up(%llu, %llu) wrong\n", (unsigned long long)n, (unsigned long long)d);
        }
    };
    for (uint64_t d : edge_d)
        for (uint64_t n : edge_n) check(n, d);
    for (int t = 0; t < 2000000; t++) {
        const int bits_d = 1 + int(rng() % 64), bits_n = 1 + int(rng() % 64);
        uint64_t d = rng() >> (64 - bits_d);
        if (d == 0) d = 1;
        const uint64_t n = rng() >> (64 - bits_n);
        check(n, d);
        check(d * (n % 1000) , d);              // exact multiples
        if (n > 0) check(d * (n % 1000) - 1, d);
    }
    std::printf("%ld checks, %ld wrong\n", count, bad);
    return bad != 0;
}
