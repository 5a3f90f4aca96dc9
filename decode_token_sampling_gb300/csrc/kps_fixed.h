// kps_fixed.h — softmax mass in 2^-40 fixed point, from the bits of an fp32 weight.
//
// round(w * 2^40), to nearest with ties to even, for a weight 0 <= w <= 2^23, computed
// with integer shifts of the significand instead of a float -> 64-bit integer conversion
// (which runs on the slow FP64 pipe of this GPU).  w * 2^40 is exact in fp32, so this is
// the plain IEEE rounding of that product.  Plain C++: host code and a CPU test include
// it too.

#ifndef KPS_FIXED_H_
#define KPS_FIXED_H_

#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define KPS_HD __host__ __device__ __forceinline__
#else
#define KPS_HD inline
#endif

namespace kps {

KPS_HD uint32_t fixed_bits(float x) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(x);
#else
  uint32_t u;
  std::memcpy(&u, &x, sizeof(u));
  return u;
#endif
}

KPS_HD unsigned long long fixed_mass_of(float w) {
  const uint32_t u = fixed_bits(w);
  const int e = static_cast<int>((u >> 23) & 0xFFu);
  if (e == 0) return 0ull;                                  // zero or below 2^-126
  const unsigned long long m = (u & 0x7FFFFFu) | 0x800000u;  // w = m * 2^(e - 150)
  const int s = e - 110;                                    // w * 2^40 = m * 2^s
  if (s >= 0) return m << s;
  const int r = -s;
  if (r > 25) return 0ull;  // below 2^-1: rounds to zero
  const unsigned long long q = m >> r;
  const unsigned long long rem = m & ((1ull << r) - 1ull);
  const unsigned long long half = 1ull << (r - 1);
  return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

}  // namespace kps

#endif  // KPS_FIXED_H_
