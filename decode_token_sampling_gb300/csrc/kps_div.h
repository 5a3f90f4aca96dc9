// kps_div.h — x / T rounded to nearest for a fixed divisor T, by a multiply and one
// FMA correction (Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990: with rT = RN(1/T) and
// q = RN(x * rT), the residual r = x - T*q is exact under FMA and RN(q + r*rT) is
// RN(x/T) when no step under- or overflows).  The callers fall back to the IEEE
// division outside a safe range of dividends and quotients, or when T is extreme.  Plain C++: host
// code and a CPU test include it too.

#ifndef KPS_DIV_H_
#define KPS_DIV_H_

#include <cmath>

#if defined(__CUDACC__)
#define KPS_DHD __host__ __device__ __forceinline__
#else
#define KPS_DHD inline
#endif

namespace kps {

// Divisor T with its rounded reciprocal; usable when both are normal numbers.
struct FixedDivisor {
  float T;
  float rT;
  bool fast;
};

KPS_DHD FixedDivisor make_divisor(float T) {
  FixedDivisor d;
  d.T = T;
#if defined(__CUDA_ARCH__)
  d.rT = __frcp_rn(T);
#else
  d.rT = 1.0f / T;
#endif
  const float aT = std::fabs(T), ar = std::fabs(d.rT);
  d.fast = aT >= 1.2621774e-29f && aT <= 7.9228163e+28f && ar >= 1.2621774e-29f && ar <= 7.9228163e+28f;
  return d;
}

// The corrected quotient; equal to RN(x / T) when div_ok(x, q) holds (the callers
// check that and otherwise use the IEEE division).
KPS_DHD float div_fast(float x, const FixedDivisor& d) {
#if defined(__CUDA_ARCH__)
  const float q = __fmul_rn(x, d.rT);
  const float r = __fmaf_rn(-d.T, q, x);
  return __fmaf_rn(r, d.rT, q);
#else
  const float q = x * d.rT;
  const float r = std::fma(-d.T, q, x);
  return std::fma(r, d.rT, q);
#endif
}

// True when a quotient q = div_fast(x, d) may be used as is: the dividend and the quotient
// lie well inside the normal range, so the product T*q and the residual are exact.
KPS_DHD bool div_ok(float x, float q) {
  const float ax = std::fabs(x), aq = std::fabs(q);
  return ax >= 1.2621774e-29f && aq >= 1.2621774e-29f && aq <= 7.9228163e+28f;  // 2^-96, 2^96
}

}  // namespace kps

#endif  // KPS_DIV_H_
