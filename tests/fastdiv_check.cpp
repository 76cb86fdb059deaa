// Checks fa::FastDiv against exact division: every divisor 1..4096 with
// numerators 0..65535 and the top of the range, then random 31-bit
// numerators for random divisors.  Exit status 0 when all agree.
#include <cstdint>
#include <cstdio>
#include <random>

#include "fa_fastdiv.h"

int main() {
  auto check = [](uint32_t d, uint32_t n) {
    const fa::FastDiv f = fa::FastDiv::make(d);
    const uint32_t q = f.div(n);
    if (q != n / d || f.mod(n, q) != n % d) {
      std::printf("mismatch d=%u n=%u got %u want %u\n", d, n, q, n / d);
      return false;
    }
    return true;
  };
  for (uint32_t d = 1; d <= 4096; ++d) {
    for (uint32_t n = 0; n < 65536; n += (d < 64 ? 1 : 7)) if (!check(d, n)) return 1;
    for (uint32_t n = 0x7fffffffu - 4096; n <= 0x7fffffffu && n >= 0x7fffffffu - 4096; ++n)
      if (!check(d, n)) return 1;
  }
  std::mt19937_64 rng(12345);
  for (int i = 0; i < 2000000; ++i) {
    const uint32_t d = 1 + (uint32_t)(rng() % 0x7fffffffu);
    const uint32_t n = (uint32_t)(rng() & 0x7fffffffu);
    if (!check(d, n)) return 1;
  }
  std::printf("ok\n");
  return 0;
}
