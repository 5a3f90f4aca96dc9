// weight_error_scan.cu — the largest relative error of each factor of the sampling
// kernels' weights and race quotients, taken over its whole input domain on the GPU (a
// test program: tests/test_weight_error.py builds and runs it and checks the results
// against the error budget of the top-p boundary and the race).
//
// Every factor comes from the kernels' own header (kps_weights.cuh); the exact value is
// the double-precision function of the same input.  Prints one JSON object.

#include "kps_weights.cuh"

#include <cstdint>
#include <cstdio>
#include <cstring>

using kps::kExpBin;

__device__ void max_into(unsigned long long* slot, double v) {
  // non-negative doubles order like their bit patterns
  atomicMax(slot, static_cast<unsigned long long>(__double_as_longlong(v)));
}

enum { kW24, kExpBinErr, kRcp, kSwGrid, kSwPairs, kSlots };

// w24_weight over every float frac in [0, 1/32] (bit patterns 0 .. bits(1/32))
__global__ void scan_w24(unsigned long long* out, uint32_t n) {
  double worst = 0.0;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float frac = __uint_as_float(i);
    const double ex = exp(-static_cast<double>(frac));
    const double got = static_cast<double>(kps::w24_weight(frac)) * 5.9604644775390625e-8;
    worst = fmax(worst, fabs(got - ex) / ex);
  }
  max_into(out + kW24, worst);
}

// the bin factors exp(-b/32)
__global__ void scan_exp_bin(unsigned long long* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < kps::kExpBins) {
    const double ex = exp(-static_cast<double>(b) / 32.0);
    max_into(out + kExpBinErr, fabs(static_cast<double>(kExpBin.v[b]) - ex) / ex);
  }
}

// rcp.approx over every float in [1, 2) (its relative error repeats in every binade of
// normal numbers)
__global__ void scan_rcp(unsigned long long* out) {
  double worst = 0.0;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (1u << 23); i += gridDim.x * blockDim.x) {
    const float x = __uint_as_float(0x3F800000u + i);
    const double got = static_cast<double>(kps::rrcp_approx(x));
    worst = fmax(worst, fabs(got * static_cast<double>(x) - 1.0));
  }
  max_into(out + kRcp, worst);
}

// softmax_weight(s, 0) over every float s in [-87, 0) (no rounding in s - M: expf alone)
__global__ void scan_sw_grid(unsigned long long* out, uint32_t lo_bits, uint32_t n) {
  double worst = 0.0;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float s = -__uint_as_float(lo_bits + i);
    const double ex = exp(static_cast<double>(s));
    worst = fmax(worst, fabs(static_cast<double>(kps::softmax_weight(s, 0.0f)) - ex) / ex);
  }
  max_into(out + kSwGrid, worst);
}

// softmax_weight(x, M) on pseudo-random pairs: M in [-32, 32), x = fl(M + s) with s in
// [-80, 0], against exp(x - M) of the exact difference (so the rounding of x - M counts)
__device__ __forceinline__ uint32_t mix32(uint32_t x) {  // an integer hash (lowbias32)
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}
__global__ void scan_sw_pairs(unsigned long long* out, uint32_t n) {
  double worst = 0.0;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const uint32_t h1 = mix32(2u * i + 1u), h2 = mix32(2u * i + 2u);
    const float M = static_cast<float>(static_cast<int32_t>(h1)) * 1.4901161193847656e-8f;  // [-32, 32)
    const float s = -static_cast<float>(h2 >> 8) * 4.76837158203125e-6f;                   // [-80, 0]
    const float x = __fadd_rn(M, s);
    if (!(x <= M)) continue;
    const double d = static_cast<double>(x) - static_cast<double>(M);  // exact
    if (d < -87.0) continue;
    const double ex = exp(d);
    worst = fmax(worst, fabs(static_cast<double>(kps::softmax_weight(x, M)) - ex) / ex);
  }
  max_into(out + kSwPairs, worst);
}

static uint32_t float_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
}

int main() {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, kSlots * sizeof(unsigned long long)) != cudaSuccess) return 2;
  cudaMemset(d, 0, kSlots * sizeof(unsigned long long));
  const int grid = 152 * 8, block = 256;
  scan_w24<<<grid, block>>>(d, float_bits(0.03125f) + 1u);
  scan_exp_bin<<<(kps::kExpBins + 255) / 256, 256>>>(d);
  scan_rcp<<<grid, block>>>(d);
  scan_sw_grid<<<grid, block>>>(d, 1u, float_bits(87.0f));  // s = -(smallest subnormal) .. -87
  scan_sw_pairs<<<grid, block>>>(d, 1u << 28);
  unsigned long long h[kSlots];
  const cudaError_t e = cudaMemcpy(h, d, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    std::printf("{\"error\": \"%s\"}\n", cudaGetErrorString(e));
    return 1;
  }
  double v[kSlots];
  std::memcpy(v, h, sizeof v);
  std::printf("{\"w24\": %.6e, \"exp_bin\": %.6e, \"rcp\": %.6e, \"softmax_weight_grid\": %.6e, "
              "\"softmax_weight_pairs\": %.6e}\n", v[kW24], v[kExpBinErr], v[kRcp], v[kSwGrid], v[kSwPairs]);
  cudaFree(d);
  return 0;
}
