"""Builds the in-tree CUDA library libkps.so for GB300 (sm_103a) with nvcc.

One translation unit, one -gencode, compiled in seconds; the product is
decode_token_sampling_gb300/libkps.so (git-ignored).  No torch extension
machinery is involved: the library exports a plain C ABI (include/kps.h).
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "kps.cu")
HDR = os.path.join(ROOT, "include", "kps.h")
LIB = os.path.join(PKG, "libkps.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkps.so")
    return cand


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out: str = LIB) -> str:
    """Compile libkps.so (or, with extra_flags and another `out`, a variant of it) if it is
    missing or older than its sources; returns its path."""
    srcs = [HDR] + [os.path.join(PKG, "csrc", f) for f in sorted(os.listdir(os.path.join(PKG, "csrc")))
                    if f.endswith((".cu", ".cuh", ".h"))]
    if not force and os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in srcs):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(extra_flags or []), "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


# Test-only variant: the cluster kernel's first copy wait in each CTA goes to a barrier that
# no copy completes, bounded by this many clock cycles, so that its timeout path (status
# KPS_ERR_TIMEOUT, one more bounded wait for the real copy) runs on every call.
SPIN_TEST_LIB = os.path.join(PKG, "libkps_spin_test.so")
SPIN_TEST_CYCLES = 20000


def build_spin_test(force: bool = False) -> str:
    return build(force=force, extra_flags=[f"-DKPS_TEST_SPIN_CYCLES={SPIN_TEST_CYCLES}LL"], out=SPIN_TEST_LIB)


# Debug variant: every kernel's dynamic shared memory starts as a NaN pattern
# (KPS_DEBUG_SENTINEL), so a read of shared memory that nothing in the launch wrote shows
# up as a wrong result.
SENTINEL_LIB = os.path.join(PKG, "libkps_sentinel.so")


def build_sentinel(force: bool = False) -> str:
    return build(force=force, extra_flags=["-DKPS_DEBUG_SENTINEL"], out=SENTINEL_LIB)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
