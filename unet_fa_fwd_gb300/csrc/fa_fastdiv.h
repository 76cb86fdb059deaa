// fa_fastdiv.h — division by a divisor fixed for a whole launch, as one
// multiply-high, one add and one shift (the divisor's magic number is computed
// once on the host).  Round-up method: for d >= 1, l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, the quotient of any n < 2^31 is
// (mulhi(n, m) + n) >> l.  Plain C++ on the host (it is checked there
// exhaustively for small divisors and at random for large ones) and inline
// device code in the kernels.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

struct FastDiv {
  uint32_t d, m, l;

  FastDiv() = default;
  // d >= 1 (callers pass launch sizes, all >= 1).
  static FastDiv make(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    f.l = l;
    f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
    return f;
  }
  FA_HD uint32_t div(uint32_t n) const {  // n < 2^31
#if defined(__CUDA_ARCH__)
    const uint32_t hi = __umulhi(n, m);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)n * m) >> 32);
#endif
    return (hi + n) >> l;
  }
  FA_HD uint32_t mod(uint32_t n, uint32_t q) const { return n - q * d; }
};

}  // namespace fa
