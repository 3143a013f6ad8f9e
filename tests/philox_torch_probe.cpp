// Test helper: prints the Philox4x32-10 word that PyTorch's header-only
// engine (ATen/core/PhiloxRNGEngine.h) gives for each "seed g" pair read from
// stdin, using key = seed and the 64-bit offset g >> 2 in counter words 0-1;
// word g & 3 of that block is printed.  Used to pin the oracle's generator
// to an independent implementation.
#include <ATen/core/PhiloxRNGEngine.h>

#include <cstdint>
#include <cstdio>

int main() {
  unsigned long long seed = 0, g = 0;
  while (std::scanf("%llu %llu", &seed, &g) == 2) {
    at::philox_engine eng(seed, /*subsequence=*/0, /*offset=*/g >> 2);
    uint32_t w = 0;
    for (unsigned i = 0; i <= (unsigned)(g & 3u); ++i) w = eng();
    std::printf("%u\n", w);
  }
  return 0;
}
