"""The GPU path's division by a per-row temperature: a multiply by RN(1/T) and one FMA
correction (Markstein), used only inside a safe range of dividends and quotients.

Checked on the CPU against the IEEE quotient x / T: every fp32 significand (both signs)
at exponents near both ends of the safe range and in between, plus 2^24 random bit
patterns, for temperatures that include the workloads' range, all-ones and all-zeros
significands, and extremes.
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
#include <cstdint>
#include <cstdlib>
#include <random>
#include "kps_div.h"
static float from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
static unsigned long long bad = 0, used = 0;
static void check(float x, const kps::FixedDivisor& d) {
  const float q = kps::div_fast(x, d);
  if (!kps::div_ok(x, q)) return;
  ++used;
  const float want = x / d.T;
  uint32_t a, b;
  std::memcpy(&a, &q, 4);
  std::memcpy(&b, &want, 4);
  if (a != b) {
    if (bad < 5) std::printf("T=%a x=%a fast=%a ieee=%a\n", d.T, x, q, want);
    ++bad;
  }
}
int main(int argc, char** argv) {
  for (int i = 1; i < argc; ++i) {
    const float T = from_bits(static_cast<uint32_t>(std::strtoul(argv[i], nullptr, 16)));
    const kps::FixedDivisor d = kps::make_divisor(T);
    if (!d.fast) continue;
    // every significand, both signs, at exponents near both ends of the safe range and in between
    const int exps[] = {-95, -94, -60, -1, 0, 1, 20, 60, 94, 95};
    for (int e : exps)
      for (uint32_t m = 0; m < (1u << 23); ++m)
        for (uint32_t s = 0; s < 2; ++s) check(from_bits((s << 31) | (static_cast<uint32_t>(e + 127) << 23) | m), d);
    // and random bit patterns
    std::mt19937 rng(1234 + i);
    for (int k = 0; k < (1 << 24); ++k) check(from_bits(rng()), d);
  }
  std::printf("used=%llu bad=%llu\n", used, bad);
  return bad == 0 ? 0 : 1;
}
"""

# temperatures (fp32 bit patterns): 0.5, 0.7, 0.85, 1.0, 1.1, 1.2, 3.0 (odd significand),
# the largest float below 1 and below 2 (all-ones significands), 1e-3, 1e3, 2.0, 0.1
TEMPS = ["3f000000", "3f333333", "3f59999a", "3f800000", "3f8ccccd", "3f99999a", "40400000",
         "3f7fffff", "3fffffff", "3a83126f", "447a0000", "40000000", "3dcccccd"]


@pytest.fixture(scope="module")
def divtest():
    d = tempfile.mkdtemp()
    src = os.path.join(d, "t.cpp")
    exe = os.path.join(d, "t")
    with open(src, "w") as f:
        f.write(PROGRAM)
    r = subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC, src, "-o", exe],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.fail(r.stderr)
    return exe


def test_fixed_divisor_matches_ieee_division(divtest):
    r = subprocess.run([divtest, *TEMPS], capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout
    assert "bad=0" in r.stdout
