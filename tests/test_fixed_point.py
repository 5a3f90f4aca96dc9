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


CEIL_PROGRAM = r"""
#include <cstdio>
#include <cstring>
#include <cstdint>
#include "kps_fixed.h"
// reads lines "pbits total", prints ceil_mul_p for each
int main() {
  unsigned u; unsigned long long t;
  while (std::scanf("%x %llu", &u, &t) == 2) {
    float p;
    std::memcpy(&p, &u, 4);
    std::printf("%llu\n", kps::ceil_mul_p(p, t));
  }
  return 0;
}
"""


def test_ceil_mul_p_against_exact_fractions():
    """ceil(p * total) clamped to [1, total], against exact rational arithmetic, on p from
    subnormals to just below 1 and totals up to 2^63."""
    import random
    import struct
    from fractions import Fraction
    rng = random.Random(7)
    cases = []
    specials = [0x00000001, 0x00000100, 0x007FFFFF, 0x00800000, 0x33800000, 0x3F000000, 0x3F7FFFFF,
                0x3F4CCCCD, 0x3E99999A, 0x3F733333]
    totals = [1, 2, 3, 1023, 2**24 + 1, 2**40, 2**40 * 150000 + 12345, 2**62 + 7, 2**63 - 1]
    for pb in specials:
        for t in totals:
            cases.append((pb, t))
    for _ in range(20000):
        pb = rng.randrange(1, 0x3F800000)
        t = rng.choice([rng.randrange(1, 2**20), rng.randrange(1, 2**45), rng.randrange(1, 2**63)])
        cases.append((pb, t))
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "c.cpp")
        exe = os.path.join(tmp, "c")
        open(src, "w").write(CEIL_PROGRAM)
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", CSRC, "-o", exe, src])
        inp = "".join(f"{pb:x} {t}\n" for pb, t in cases)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout.split()
    assert len(out) == len(cases)
    for (pb, t), got in zip(cases, out):
        p = Fraction(struct.unpack("<f", struct.pack("<I", pb))[0])
        x = p * t
        want = -((-x.numerator) // x.denominator)  # ceil
        want = min(max(want, 1), t)
        assert int(got) == want, (hex(pb), t, got, want)
