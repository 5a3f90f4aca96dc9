// kps_weights.cuh — the softmax weights and race quotients of the sampling kernels, the
// arithmetic that decides the top-p boundary and the race winner.
//
// Top-k rows weigh a survivor y against the row maximum M as softmax_weight(y, M) =
// exp(y - M) (the rounding of y - M corrected to first order) and race it as
// weight / (q + eps) in IEEE division.  Top-p-only rows weigh an element of bin b (bins of
// width 1/32 below a reference H) as w24 * 2^-24 * exp(-b/32), with w24 = w24_weight(frac)
// the 24-bit weight of its position frac inside the bin and exp(-b/32) from a table
// (kExpBin), and race it as w24 * rcp(q + eps) * 2^-24 * exp(-b/32).
//
// The relative error of each factor bounds how far a kernel's decision can stray from
// the exact one: a top-p boundary can move only where the exact prefix mass lies within
// 2 (1 - p) e of p * S, and a race winner change only where the two best scores lie within
// 2 e of each other, e being the largest relative error of one element's mass (or score).
// The bounds of each factor, taken over its whole input domain on the GPU, are pinned by a
// GPU test (tests/weight_error_scan.cu).

#ifndef KPS_WEIGHTS_CUH_
#define KPS_WEIGHTS_CUH_

#include <cstdint>

namespace kps {

// 2^x by the hardware approximation (ex2.approx.f32).
__device__ __forceinline__ float rex2(float x) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// 1/x by the hardware approximation (rcp.approx.f32).
__device__ __forceinline__ float rrcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

constexpr float kLog2e = 1.4426950408889634f;

// exp(y - M) for y <= M: 1 at the maximum, 0 below exp's range; the rounding error of
// s = y - M is recovered exactly (two-sum) and applied to first order, exp(s + lo) =
// exp(s) (1 + lo).
__device__ __forceinline__ float softmax_weight(float x, float M) {
  if (x == M) return 1.0f;
  float s = __fsub_rn(x, M);
  if (!(s > -INFINITY)) return 0.0f;
  float bb = __fsub_rn(s, x);
  float lo = __fadd_rn(__fsub_rn(x, __fsub_rn(s, bb)), __fsub_rn(-M, bb));
  float e = expf(s);
  return __fmaf_rn(e, lo, e);
}

// The weight of a position frac (in [0, 1/32), possibly a rounding outside it) inside a
// bin, exp(-frac), in units of 2^-24: an integer-valued float in [2^23, 2^24).  ex2 of the
// small argument -frac log2(e) lands in [1/2, 1), where the float spacing is 2^-24, so the
// scaling by 2^24 is exact and already an integer; the top weight 2^24 is clamped to
// 2^24 - 1 so that the weight fits 24 bits.
__device__ __forceinline__ float w24_weight(float frac) {
  return fminf(__fmul_rn(rex2(__fmul_rn(frac, -kLog2e)), 16777216.0f), 16777215.0f);
}

// exp(-b/32) for b = 0 .. 2047 to the nearest float, evaluated by the compiler: exp(-1/32)
// by its Taylor series in double, then its powers by repeated multiplication (relative
// error below 2^-35 before the rounding to float, so each entry is within 2^-24 + 2^-35
// relative).
constexpr int kExpBins = 2048;
struct ExpBinTable {
  float v[kExpBins];
};
constexpr double exp_neg_1_32() {
  double term = 1.0, sum = 1.0;
  for (int k = 1; k < 24; ++k) {
    term = term * (-1.0 / 32.0) / static_cast<double>(k);
    sum += term;
  }
  return sum;
}
constexpr ExpBinTable make_exp_bin_table() {
  ExpBinTable t{};
  const double f = exp_neg_1_32();
  double e = 1.0;
  for (int b = 0; b < kExpBins; ++b) {
    t.v[b] = static_cast<float>(e);
    e *= f;
  }
  return t;
}
__device__ const ExpBinTable kExpBin = make_exp_bin_table();

}  // namespace kps

#endif  // KPS_WEIGHTS_CUH_
