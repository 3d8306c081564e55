// Division by a divisor fixed for a kernel launch, shared by host (which
// prepares the constants) and device (which divides).
#pragma once

namespace attn {

// Division of 0 <= x < 2^31 by a divisor d >= 1 fixed for the launch, as a
// multiply-high, an add and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, the round-up method
// with a 33-bit multiplier 2^32 + m): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1,  x / d = (umulhi(x, m) + x) >> l.
// A work unit's decode takes five such divisions.  As plain integer
// divisions (each a dependent chain of about 20 instructions) they made
// every role's step from one unit to the next about 300 (MMA issuer) to
// 800 (softmax warps) cycles longer, which cost up to 5 % on launches of
// few K/V steps per unit.
struct FastDiv {
  int d;
  unsigned int m;
  unsigned int l;
};

inline FastDiv make_fast_div(int d) {
  FastDiv f;
  f.d = d;
  unsigned int l = 0;
  while ((1ull << l) < static_cast<unsigned long long>(d)) ++l;
  f.l = l;
  f.m = static_cast<unsigned int>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ int fast_div(int x, const FastDiv& f) {
  const unsigned int ux = static_cast<unsigned int>(x);
  return static_cast<int>((__umulhi(ux, f.m) + ux) >> f.l);
}
#else
inline int fast_div(int x, const FastDiv& f) {
  const unsigned int ux = static_cast<unsigned int>(x);
  const unsigned int hi = static_cast<unsigned int>(
      (static_cast<unsigned long long>(ux) * f.m) >> 32);
  return static_cast<int>((hi + ux) >> f.l);
}
#endif

}  // namespace attn
