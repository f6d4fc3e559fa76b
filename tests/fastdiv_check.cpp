// fastdiv_check.cpp — CPU check of swa::FastDiv (swa_kernels.h), the multiply-high division the
// persistent kernels use to split their tile index, against the C++ division and remainder.
//
// Every divisor 1..3000 against every dividend below 12,000 and a set of dividends near 2^31; a
// list of larger divisors (up to 2^31 - 1) against dividends spread over [0, 2^31).  Prints
// "ok <checks>" and exits 0, or prints the first mismatch and exits 1.
#include <cstdint>
#include <cstdio>

#include "swa_kernels.h"

namespace {

int check(const swa::FastDiv& f, uint32_t n, uint32_t d) {
  if (f.div(n) != n / d || f.mod(n) != n % d) {
    std::printf("mismatch: %u / %u gave %u rem %u, want %u rem %u\n", n, d, f.div(n), f.mod(n),
                n / d, n % d);
    return 1;
  }
  return 0;
}

}  // namespace

int main() {
  long long checks = 0;
  const uint32_t near_top[] = {(1u << 31) - 1, (1u << 31) - 2, 1u << 30, (1u << 30) + 12345,
                               999999999u, 2147480000u};
  for (uint32_t d = 1; d <= 3000; ++d) {
    const swa::FastDiv f(d);
    for (uint32_t n = 0; n < 12000; ++n, ++checks)
      if (check(f, n, d)) return 1;
    for (uint32_t n : near_top) {
      if (check(f, n, d) || check(f, n - d, d)) return 1;
      checks += 2;
    }
  }
  const uint32_t large[] = {4095, 4096, 4097, 65535, 65536, 1u << 20, 12345678, 1u << 30,
                            (1u << 31) - 1};
  for (uint32_t d : large) {
    const swa::FastDiv f(d);
    for (uint64_t n = 0; n < (1ull << 31); n += 104729, ++checks)
      if (check(f, static_cast<uint32_t>(n), d)) return 1;
  }
  std::printf("ok %lld\n", checks);
  return 0;
}
