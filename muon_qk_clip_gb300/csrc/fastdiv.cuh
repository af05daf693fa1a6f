// Division by a run-time divisor as a multiply and a shift, for the work-item
// decoding of the persistent attention-side kernels: a hardware division
// sequence costs their single-thread issue loops hundreds of cycles per item.
#pragma once

#include <stdint.h>

namespace mc {

// floor(n / d) = (n * m) >> sh for every n < 2^31, with sh = 31 + s,
// s = floor(log2 d) + 1 (so d < 2^s) and m = ceil(2^sh / d): the rounding
// error n (m - 2^sh / d) / 2^sh stays below 2^31 / 2^sh = 2^-s < 1 / d, and
// m <= 2^33 keeps n * m below 2^64.
struct FastDiv {
  unsigned long long m;
  int sh;
};

inline FastDiv make_fastdiv(uint32_t d) {
  int s = 0;
  while ((1ull << s) <= d) ++s;
  FastDiv f;
  f.sh = 31 + s;
  f.m = ((1ull << f.sh) + d - 1) / d;
  return f;
}

#ifdef __CUDACC__
__device__ inline uint32_t fastdiv(uint32_t n, const FastDiv& f) {
  return (uint32_t)(((unsigned long long)n * f.m) >> f.sh);
}
#endif

}  // namespace mc
