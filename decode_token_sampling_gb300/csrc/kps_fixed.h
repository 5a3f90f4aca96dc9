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

// The high 64 bits of a * b.
KPS_HD unsigned long long mul_hi_u64(unsigned long long a, unsigned long long b) {
#if defined(__CUDA_ARCH__)
  return __umul64hi(a, b);
#else
  return static_cast<unsigned long long>((static_cast<unsigned __int128>(a) * b) >> 64);
#endif
}

// ceil(p * total) for 0 < p < 1 (a finite float), exactly: p's significand times total in
// 128 bits, shifted right with the bits shifted out rounding up; clamped to [1, total].
// (The top-p target of a fixed-point total mass, without FP64: a float -> 64-bit integer
// conversion and double arithmetic run on the slow FP64 pipe of this GPU.)
KPS_HD unsigned long long ceil_mul_p(float p, unsigned long long total) {
  if (total == 0ull) return 0ull;
  const uint32_t u = fixed_bits(p);
  const int e = static_cast<int>((u >> 23) & 0xFFu);
  if (e >= 127) return total;  // p >= 1 (or not finite): everything
  const unsigned long long m = e ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);  // p = m * 2^-s
  const int s = e ? 150 - e : 149;  // >= 24 for p < 1
  const unsigned long long lo = m * total, hi = mul_hi_u64(m, total);
  unsigned long long t;
  if (s >= 128) {
    t = (lo | hi) ? 1ull : 0ull;
  } else if (s >= 64) {
    const int r = s - 64;
    const unsigned long long q = r ? (hi >> r) : hi;
    const bool rem = lo != 0ull || (r && (hi & ((1ull << r) - 1ull)) != 0ull);
    t = q + (rem ? 1ull : 0ull);
  } else {
    const unsigned long long q = (lo >> s) | (hi << (64 - s));
    const bool rem = (lo & ((1ull << s) - 1ull)) != 0ull;
    t = q + (rem ? 1ull : 0ull);
  }
  if (t < 1ull) t = 1ull;
  if (t > total) t = total;
  return t;
}

}  // namespace kps

#endif  // KPS_FIXED_H_
