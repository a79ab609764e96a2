// Host check of make_fastdiv (wgrad_params.h): for divisors 1..4096, a set of
// larger ones and numerators up to 2^31 - 1, umulhi(x, mul) >> shift must equal
// x / d.  Prints "ok <cases>" or the first mismatch and exits non-zero.
#include <cstdint>
#include <cstdio>

#include "wgrad_params.h"

static uint32_t umulhi_host(uint32_t a, uint32_t b) {
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
}

int main() {
  uint64_t cases = 0;
  uint64_t lcg = 12345;
  auto next = [&]() {
    lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
    return static_cast<uint32_t>(lcg >> 33);   // 31 bits
  };
  for (int pass = 0; pass < 2; ++pass) {
    const uint32_t dmax = pass == 0 ? 4096 : 2000;
    for (uint32_t i = 1; i <= dmax; ++i) {
      const uint32_t d = pass == 0 ? i : (next() % 0x7FFFFFFFu) + 1;
      const dg::FastDiv f = dg::make_fastdiv(d);
      const uint32_t edge[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 0x7FFFFFFEu, 0x7FFFFFFFu,
                               (0x7FFFFFFFu / d) * d, (0x7FFFFFFFu / d) * d - 1};
      for (int k = 0; k < 10 + 200; ++k) {
        const uint32_t x = k < 10 ? edge[k] : next();
        if (x > 0x7FFFFFFFu) continue;
        const uint32_t q = f.mul == 0 ? x : (umulhi_host(x, f.mul) >> f.shift);
        if (q != x / d) {
          std::printf("mismatch d=%u x=%u q=%u want=%u\n", d, x, q, x / d);
          return 1;
        }
        ++cases;
      }
    }
  }
  std::printf("ok %llu\n", static_cast<unsigned long long>(cases));
  return 0;
}
