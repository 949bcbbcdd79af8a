// fastdiv.h -- division by a divisor fixed at launch time, as a multiply-high
// and a shift, for the index arithmetic that maps a work item to its batch,
// head and rows.  Host and device share the code; it also compiles as plain
// C++ (no CUDA), so the host tests check it exhaustively on small divisors.
//
// Method: Granlund and Montgomery, "Division by invariant integers using
// multiplication" (PLDI 1994), section 4, for 32-bit unsigned words.  With
// s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1 (which fits 32 bits,
// because 2^s - d < d), floor(n / d) = floor((mulhi(n, m) + n) / 2^s) for every
// 32-bit n; the sum stays below 2^32 when n < 2^31, the range used here.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

struct FastDiv {
  uint32_t d;  // divisor, >= 1
  uint32_t m;  // magic multiplier
  uint32_t s;  // shift, ceil(log2 d)
};

// Host: the constants for divisor d (d >= 1, d < 2^31).
inline FastDiv fastdiv_make(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.s = 0;
  while ((uint64_t(1) << f.s) < d) ++f.s;
  f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << f.s) - d)) / d + 1);
  return f;
}

// floor(n / f.d) for 0 <= n < 2^31.
ATTN_HD uint32_t fastdiv_div(const FastDiv &f, uint32_t n) {
#if defined(__CUDA_ARCH__)
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> 32);
#endif
  return (hi + n) >> f.s;
}

// q = floor(n / f.d), r = n - q * f.d.
ATTN_HD void fastdiv_divmod(const FastDiv &f, int n, int &q, int &r) {
  q = static_cast<int>(fastdiv_div(f, static_cast<uint32_t>(n)));
  r = n - q * static_cast<int>(f.d);
}

}  // namespace attn
