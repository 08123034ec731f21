// fastdiv.h -- exact division of element indices by a run-time chunk length.
//
// Every kernel maps an element index e to its chunk j = e / L.  A 64-bit
// integer division is a long software sequence on the GPU, and its result
// is needed before the first load can be addressed (the ring order starts
// at rank j + 1).  For dividends below 2^32 the quotient is instead taken
// as a multiply-high and two shifts, with a magic number computed once on
// the host: Granlund & Montgomery, "Division by Invariant Integers using
// Multiplication" (PLDI 1994), the unsigned round-up method.  For a divisor
// d >= 2 with l = ceil(log2 d):
//     m = floor(2^32 * (2^l - d) / d) + 1            (fits in 32 bits)
//     t = floor(m * n / 2^32);  q = (t + ((n - t) >> 1)) >> (l - 1)
// which equals floor(n / d) for every 32-bit n.  Larger dividends, and
// d == 1, fall back to ordinary division.
//
// Plain C++ usable from host and device code (the CPU tests compile it
// with the host compiler alone).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define CR_HD __host__ __device__ __forceinline__
#else
#define CR_HD inline
#endif

namespace cr {

struct FastDiv {
  uint64_t d;      // divisor (>= 1)
  uint32_t magic;  // m of the round-up method
  uint32_t shift;  // l - 1
  uint32_t fast;   // 1: every dividend used is below 2^32 and d >= 2
  uint32_t pad;
};

// max_n: the largest dividend the kernels will divide.
inline FastDiv fastdiv_make(uint64_t d, uint64_t max_n) {
  FastDiv f;
  f.d = d ? d : 1;
  f.magic = 0;
  f.shift = 0;
  f.fast = 0;
  f.pad = 0;
  if (f.d >= 2 && max_n < (1ull << 32) && f.d <= (1ull << 32)) {
    uint32_t l = 0;
    while ((1ull << l) < f.d) ++l;  // l = ceil(log2 d), 1 <= l <= 32
    const uint64_t num = (1ull << 32) * ((1ull << l) - f.d);  // < 2^64: 2^l - d < d <= 2^32
    f.magic = (uint32_t)(num / f.d + 1);
    f.shift = l - 1;
    f.fast = 1;
  }
  return f;
}

CR_HD uint32_t fastdiv_mulhi(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return (uint32_t)(((uint64_t)a * (uint64_t)b) >> 32);
#endif
}

CR_HD uint64_t fastdiv_div(const FastDiv& f, uint64_t n) {
  if (f.fast) {
    const uint32_t n32 = (uint32_t)n;
    const uint32_t t = fastdiv_mulhi(n32, f.magic);
    return (uint64_t)((t + ((n32 - t) >> 1)) >> f.shift);
  }
  return n / f.d;
}

}  // namespace cr
