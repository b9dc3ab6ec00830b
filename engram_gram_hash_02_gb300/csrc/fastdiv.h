// Division of n in [0, 2^31) by a divisor that is fixed for a whole launch, as one multiply and
// one shift. The method is Granlund and Montgomery's ("Division by invariant integers using
// multiplication", PLDI 1994, the round-up multiplier): with l = ceil(log2 d) and
// m = ceil(2^(31 + l) / d), the error m * d - 2^(31 + l) is below d <= 2^l, so
// floor(n / d) = floor(n * m / 2^(31 + l)) for every n < 2^31, and m < 2^32 (d > 2^(l - 1)).
// Plain C++ (host and device), so that a host program can check it against the division.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define ENGRAM_HD __host__ __device__ __forceinline__
#else
#define ENGRAM_HD inline
#endif

namespace engram {

struct FastDiv {
  uint32_t m;       // multiplier; 0 for d = 1 (the quotient is n)
  uint32_t s;       // l - 1: the quotient is the high word of n * m shifted right by s
};

// d in [1, 2^31)
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  if (d == 1) {
    f.m = 0;
    f.s = 0;
    return f;
  }
  uint32_t l = 0;
  while (((uint64_t)1 << l) < d) ++l;           // l >= 1
  const uint64_t p = (uint64_t)1 << (31 + l);
  f.m = (uint32_t)((p + d - 1) / d);
  f.s = l - 1;
  return f;
}

// floor(n / d) for n in [0, 2^31): (n * m) >> (31 + l) as the high word of n * m, >> (l - 1)
ENGRAM_HD uint32_t fast_div(uint32_t n, FastDiv f) {
#ifdef __CUDA_ARCH__
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
  return f.m != 0 ? hi >> f.s : n;
}

}  // namespace engram
