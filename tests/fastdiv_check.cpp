// Host-side check of fsdp_emulated_ranks_gb300/csrc/fastdiv.h: the
// multiply-shift quotient must equal n / d for every divisor and dividend
// tried (edge values around powers of two, the workloads' chunk lengths,
// and pseudo-random ones).  Prints the number of mismatches.
#include <cstdint>
#include <cstdio>

#include "fastdiv.h"

static uint64_t s = 0x9E3779B97F4A7C15ull;
static uint64_t rnd() {
  s ^= s << 13;
  s ^= s >> 7;
  s ^= s << 17;
  return s;
}

int main() {
  uint64_t bad = 0, checks = 0;
  uint64_t divisors[4096];
  int nd = 0;
  for (uint64_t d = 1; d <= 300; ++d) divisors[nd++] = d;
  for (int b = 2; b <= 32; ++b) {
    const uint64_t p = 1ull << b;
    divisors[nd++] = p - 1;
    divisors[nd++] = p;
    divisors[nd++] = p + 1;
  }
  const uint64_t workload[] = {262144, 4194304, 162500000, 2097152, 16777216, 1638400};
  for (uint64_t d : workload) divisors[nd++] = d;
  while (nd < 4000) divisors[nd++] = 1 + rnd() % 0xffffffffull;
  for (int k = 0; k < nd; ++k) {
    const uint64_t d = divisors[k];
    const cr::FastDiv f = cr::fastdiv_make(d, 0xffffffffull);
    auto check = [&](uint64_t n) {
      ++checks;
      if (cr::fastdiv_div(f, n) != n / d) {
        if (bad < 10) printf("d=%llu n=%llu got %llu\n", (unsigned long long)d,
                             (unsigned long long)n, (unsigned long long)cr::fastdiv_div(f, n));
        ++bad;
      }
    };
    for (uint64_t n = 0; n < 2048; ++n) check(n);
    for (int q = 0; q < 64; ++q) {  // around multiples of d
      const uint64_t m = d * (rnd() % (0xffffffffull / d + 1));
      for (int64_t o = -2; o <= 2; ++o)
        if ((int64_t)m + o >= 0 && m + o <= 0xffffffffull) check(m + o);
    }
    for (int q = 0; q < 2000; ++q) check(rnd() & 0xffffffffull);
    check(0xffffffffull);
    check(0xfffffffeull);
  }
  // Dividends beyond 32 bits take the plain division.
  const cr::FastDiv big = cr::fastdiv_make(162500000, 1ull << 40);
  for (int q = 0; q < 100000; ++q) {
    const uint64_t n = rnd() & ((1ull << 40) - 1);
    ++checks;
    if (cr::fastdiv_div(big, n) != n / 162500000) ++bad;
  }
  printf("checks=%llu mismatches=%llu\n", (unsigned long long)checks, (unsigned long long)bad);
  return bad != 0;
}
