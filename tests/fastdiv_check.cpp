// Host check of the multiply-and-shift division (csrc/fastdiv.h) against the division itself.
// Exit status 0 when every case agrees; prints the first disagreement otherwise.
#include <stdio.h>
#include <stdlib.h>

#include <initializer_list>
#include "fastdiv.h"

using engram::FastDiv;
using engram::fast_div;
using engram::make_fastdiv;

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint32_t next31() {                    // xorshift64, 31-bit outputs
  rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
  return (uint32_t)(rng >> 33);
}

static int check(uint32_t n, uint32_t d, FastDiv f) {
  if (fast_div(n, f) != n / d) {
    printf("mismatch: n %u d %u got %u want %u\n", n, d, fast_div(n, f), n / d);
    return 1;
  }
  return 0;
}

int main() {
  const uint32_t top = 0x7FFFFFFFu;           // largest numerator
  // every numerator below 2^24 for the divisors the gathers meet (chunks per row, columns)
  const uint32_t small[] = {1, 2, 3, 4, 5, 7, 8, 9, 16, 24, 32, 48, 64, 96};
  for (uint32_t d : small) {
    const FastDiv f = make_fastdiv(d);
    for (uint32_t n = 0; n < (1u << 24); ++n)
      if (check(n, d, f)) return 1;
  }
  // divisors 1 .. 2^17 and a spread up to 2^31 - 1: multiples of d and their neighbours near
  // 0 and near the top, and random numerators
  for (uint64_t d64 = 1; d64 <= top; d64 = d64 < (1u << 17) ? d64 + 1 : d64 * 3 / 2 + 1) {
    const uint32_t d = (uint32_t)d64;
    const FastDiv f = make_fastdiv(d);
    const uint32_t q_top = top / d;
    for (uint32_t k = 0; k < 4; ++k) {
      const uint64_t lo = (uint64_t)k * d, hi = (uint64_t)(q_top - (k < q_top ? k : q_top)) * d;
      for (uint64_t base : {lo, hi})
        for (int e = -1; e <= 1; ++e) {
          const int64_t n = (int64_t)base + e;
          if (n >= 0 && n <= top && check((uint32_t)n, d, f)) return 1;
        }
    }
    if (check(top, d, f) || check(top - 1, d, f)) return 1;
    for (int r = 0; r < 64; ++r)
      if (check(next31(), d, f)) return 1;
  }
  printf("ok\n");
  return 0;
}
