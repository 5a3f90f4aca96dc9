"""The GPU path's fixed-point softmax mass: round(w * 2^40), nearest with ties to even.

kps_fixed.h computes it with integer shifts of the fp32 significand (a float -> 64-bit
integer conversion is slow on the GPU).  This checks it, on the CPU, against the IEEE
definition for every fp32 weight in [0, 1] and for larger weights up to 2^23.
"""

import os
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_token_sampling_gb300", "csrc")

PROGRAM = r"""
#include <cmath>
#include <cstdio>
#include <cstring>
#include "kps_fixed.h"
int main() {
  // every fp32 bit pattern from +0 up to 2^23 (weights are never negative)
  const uint32_t hi = 0x4B000000u;  // 2^23
  unsigned long long bad = 0;
  for (uint32_t u = 0; u <= hi; ++u) {
    float w;
    std::memcpy(&w, &u, 4);
    const double exact = std::ldexp(static_cast<double>(w), 40);  // exact in double
    const unsigned long long want = static_cast<unsigned long long>(std::nearbyint(exact));
    if (kps::fixed_mass_of(w) != want) {
      if (bad < 5) std::printf("mismatch at %08x: %llu vs %llu\n", u, kps::fixed_mass_of(w), want);
      ++bad;
    }
  }
  std::printf("bad=%llu\n", bad);
  return bad == 0 ? 0 : 1;
}
"""


def test_fixed_mass_matches_ieee_rounding_exhaustively():
    gxx = "g++"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.cpp")
        exe = os.path.join(d, "t")
        with open(src, "w") as f:
            f.write(PROGRAM)
        r = subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, src, "-o", exe], capture_output=True, text=True)
        if r.returncode != 0:
            pytest.fail(r.stderr)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout
        assert "bad=0" in r.stdout
