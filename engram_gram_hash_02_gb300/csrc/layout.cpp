// Host-side layout of the Engram hash tables: the prime bucket sizes and their offsets.
//
// Follows the vLLM "deepseek_v41.common.engram" page (EngramLayout.__init__: per layer and
// n-gram size the search restarts above engram_vocab_size - 1 and takes n_heads successive
// primes never handed out before; find_next_prime; _is_prime: deterministic Miller-Rabin
// with witnesses 2, 7, 61 after trial division by the primes up to 37, valid below 2^32).
#include <stdint.h>
#include <stdio.h>

#include <set>
#include <string>

#include "../../include/engram.h"

namespace engram {
void set_error(const char* fmt, ...);
}

namespace {

uint64_t mulmod(uint64_t a, uint64_t b, uint64_t n) { return (a * b) % n; }  // a, b < n < 2^32

uint64_t powmod(uint64_t a, uint64_t e, uint64_t n) {
  uint64_t r = 1 % n;
  a %= n;
  while (e) {
    if (e & 1) r = mulmod(r, a, n);
    a = mulmod(a, a, n);
    e >>= 1;
  }
  return r;
}

bool is_prime_u32(uint64_t n) {
  if (n < 2) return false;
  static const uint64_t small[] = {2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37};
  for (uint64_t p : small) {
    if (n % p == 0) return n == p;
  }
  uint64_t d = n - 1;
  int r = 0;
  while ((d & 1) == 0) {
    d >>= 1;
    ++r;
  }
  static const uint64_t witnesses[] = {2, 7, 61};
  for (uint64_t a : witnesses) {
    if (a % n == 0) continue;
    uint64_t x = powmod(a, d, n);
    if (x == 1 || x == n - 1) continue;
    bool composite = true;
    for (int i = 1; i < r; ++i) {
      x = mulmod(x, x, n);
      if (x == n - 1) {
        composite = false;
        break;
      }
    }
    if (composite) return false;
  }
  return true;
}

}  // namespace

extern "C" int engram_layout(int64_t vocab_size, int32_t layers, int32_t max_ngram, int32_t n_heads,
                             int64_t* primes_out, int64_t* offsets_out, int64_t* rows_out) {
  if (vocab_size < 1 || vocab_size >= ((int64_t)1 << 32) || layers < 1 || max_ngram < 2 || n_heads < 1 ||
      primes_out == nullptr || offsets_out == nullptr || rows_out == nullptr) {
    engram::set_error("engram_layout: bad arguments (vocab %lld, layers %d, max_ngram %d, heads %d)",
                      (long long)vocab_size, layers, max_ngram, n_heads);
    return ENGRAM_EINVAL;
  }
  const int cols = (max_ngram - 1) * n_heads;
  std::set<uint64_t> seen;
  for (int l = 0; l < layers; ++l) {
    int64_t running = 0;
    for (int o = 0; o < max_ngram - 1; ++o) {
      uint64_t current = (uint64_t)vocab_size - 1;
      for (int h = 0; h < n_heads; ++h) {
        uint64_t c = current + 1;
        while (!is_prime_u32(c) || seen.count(c)) {
          ++c;
          if (c >= ((uint64_t)1 << 32)) {
            engram::set_error("engram_layout: prime search passed 2^32");
            return ENGRAM_EINVAL;
          }
        }
        seen.insert(c);
        current = c;
        const int idx = l * cols + o * n_heads + h;
        primes_out[idx] = (int64_t)c;
        offsets_out[idx] = running;
        running += (int64_t)c;
      }
    }
    rows_out[l] = running;
  }
  return ENGRAM_OK;
}
