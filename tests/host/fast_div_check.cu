// Host-side check of the kernel's multiply-high division (FastDiv in
// attn_fwd_kernel.cuh): for divisors over the whole int range and dividends over
// [0, 2^31), fast_div(x, make_fast_div(d)) must equal x / d.  Built and run by
// tests/test_fast_div.py; prints the number of cases and exits non-zero on a
// mismatch.
#include <cstdint>
#include <cstdio>
#include <random>

#include "attn_fwd_kernel.cuh"

int main() {
  std::mt19937_64 rng(2024);
  long long cases = 0, bad = 0;
  auto check = [&](int x, int d) {
    const eca::FastDiv f = eca::make_fast_div(d);
    if (eca::fast_div(x, f) != x / d) {
      if (bad < 5) std::printf("mismatch: %d / %d\n", x, d);
      ++bad;
    }
    ++cases;
  };
  for (int d = 1; d <= 2048; ++d) {  // every small divisor: all small dividends, random and extreme large ones
    for (int x = 0; x < 4096; ++x) check(x, d);
    for (int k = 0; k < 256; ++k) check(static_cast<int>(rng() & 0x7fffffff), d);
    check(0x7fffffff, d);
    check(0x7fffffff - (0x7fffffff % d), d);      // the largest multiple of d
    check(0x7fffffff - (0x7fffffff % d) - 1, d);  // just below it
  }
  for (int l = 1; l < 31; ++l) {  // powers of two and their neighbours
    for (int d : {(1 << l) - 1, 1 << l, (1 << l) + 1}) {
      for (int k = 0; k < 256; ++k) check(static_cast<int>(rng() & 0x7fffffff), d);
      check(0x7fffffff, d);
      check(d, d);
      check(d - 1, d);
    }
  }
  for (int k = 0; k < 200000; ++k) {  // random pairs over the whole range
    const int d = 1 + static_cast<int>(rng() % 0x7ffffffe);
    check(static_cast<int>(rng() & 0x7fffffff), d);
    check(d, d);
    check(d - 1, d);
  }
  std::printf("%lld cases, %lld mismatches\n", cases, bad);
  return bad == 0 ? 0 : 1;
}
