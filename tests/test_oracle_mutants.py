"""The oracle's pins catch planted mistakes (CPU only).

Each mutant below is one plausible slip in oracle/kps_oracle.cpp (a flipped sign,
a dropped term, the wrong tie rule, an off-by-one boundary).  The mutant is
written into a temporary copy of the oracle package next to a copy of the pin
tests, and the pin suite is run against it in a separate process: at least one
pin must fail for every mutant.  A mutant that passes every pin would mean the
pins do not constrain that part of the oracle.  The mutants run in parallel and
the pin suite stops at its first failure, so this takes seconds.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kps_oracle.cpp")

# (name, text in the oracle, replacement): each text occurs exactly once.
MUTANTS = [
    ("top-k cap 2048", "std::min<int64_t>(V, 1024)", "std::min<int64_t>(V, 2048)"),
    ("NaN not -inf", "if (std::isnan(x[v])) x[v] = NEG_INF;", ";"),
    ("duplicate ids applied twice", "if (id < 0 || id >= V || seen[id]) continue;", "if (id < 0 || id >= V) continue;"),
    ("penalty sign flipped", "(s > 0.0f) ? (s / pen) : (s * pen)", "(s > 0.0f) ? (s * pen) : (s / pen)"),
    ("temperature multiplies", "x[v] = x[v] / T;", "x[v] = x[v] * T;"),
    ("ties by higher index", "(x[a] == x[b] && a < b)", "(x[a] == x[b] && a > b)"),
    ("softmax not shifted", "std::exp(xv - M)", "std::exp(xv)"),
    ("top_p <= 0 keeps all", "if (greedy || p <= 0.0f) {", "if (greedy) {"),
    ("top-p boundary inclusive", "while (nP < nK && c < target) {", "while (nP < nK && c <= target) {"),
    ("race without eps", "(static_cast<double>(qrow[v]) + static_cast<double>(eps))", "(static_cast<double>(qrow[v]) + 1.0)"),
    ("race takes the minimum", "r > rbest || (r == rbest && v < best)", "r < rbest || (r == rbest && v < best)"),
    ("race tie to higher index", "r > rbest || (r == rbest && v < best)", "r > rbest || (r == rbest && v > best)"),
    ("Philox Weyl increment", "k0 += 0x9E3779B9u;", "k0 += 0x9E3779B1u;"),
    ("finished rows keep their token", "if (finished[b]) idx[b] = eos;", ";"),
    ("seen append to the wrong bit", "1u << (idx[b] % 32)", "1u << ((idx[b] + 1) % 32)"),
    ("bf16 widened one bit short", "static_cast<uint32_t>(h) << 16", "static_cast<uint32_t>(h) << 15"),
    ("non-positive temperature divides", "t.greedy = !(T > 0.0f) || std::isinf(T);", "t.greedy = false;"),
    ("top-k keeps one more", "    nK = k;\n", "    nK = std::min<int64_t>(V, k + 1);\n"),
    ("sampling off takes the last kept", "return RowResult{order[0], nP,", "return RowResult{order[nP - 1], nP,"),
    ("top-p drops the crossing element", "while (nP < nK && c < target) {", "while (nP < nK && c + e[nP] < target) {"),
    ("race over the top-k set", "for (int64_t i = 0; i < nP; ++i) {\n    int64_t v = order[i];",
     "for (int64_t i = 0; i < nK; ++i) {\n    int64_t v = order[i];"),
    ("NaN race scores compete", "if (std::isnan(r)) continue;", ";"),
    ("top-k set left unsorted", "std::sort(order.begin(), order.begin() + nK, before);", ";"),
    ("greedy rows keep the nucleus", "if (greedy || p <= 0.0f) {", "if (p <= 0.0f) {"),
    ("EOS token does not finish its row", "if (idx[b] == eos) finished[b] = 1;", ";"),
    ("finished rows counted as left", "if (!finished[b]) ++left;", "++left;"),
    ("seen bits row stride off by one", "bits[b * W + v / 32] >> (v % 32)", "bits[b * (W - 1) + v / 32] >> (v % 32)"),
    ("draw takes the next word", "const uint32_t w = c[v & 3];", "const uint32_t w = c[(v + 1) & 3];"),
]


def _run_pins_against(name: str, old: str, new: str) -> tuple[str, int, str]:
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant '{name}': its text occurs {src.count(old)} times in the oracle"
    with tempfile.TemporaryDirectory(prefix="kps_mut_") as tmp:
        shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(tmp, "oracle"),
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
        with open(os.path.join(tmp, "oracle", "kps_oracle.cpp"), "w") as f:
            f.write(src.replace(old, new))
        shutil.copytree(os.path.join(ROOT, "decode_token_sampling_gb300"), os.path.join(tmp, "decode_token_sampling_gb300"),
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
        tdir = os.path.join(tmp, "tests")
        os.makedirs(tdir)
        for fn in ("conftest.py", "golden_io.py", "test_oracle_pins.py"):
            shutil.copy(os.path.join(ROOT, "tests", fn), tdir)
        shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tdir, "golden"))
        env = dict(os.environ, PYTHONPATH=tmp)
        proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                               os.path.join(tdir, "test_oracle_pins.py")],
                              cwd=tmp, env=env, capture_output=True, text=True, timeout=600)
        return name, proc.returncode, proc.stdout[-600:]


def test_every_mutant_fails_a_pin():
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda m: _run_pins_against(*m), MUTANTS))
    survivors = [(name, tail) for name, rc, tail in results if rc == 0]
    # pytest exits 1 when a test fails; anything else (e.g. a mutant that does not build)
    # is not a caught mistake either
    broken = [(name, rc, tail) for name, rc, tail in results if rc not in (0, 1)]
    assert not broken, f"mutants whose pin run did not complete: {broken}"
    assert not survivors, f"mutants that pass every pin: {[n for n, _ in survivors]}"


def test_unmutated_oracle_passes_the_pins_in_a_copy():
    """The harness itself: the copied, unmodified oracle passes (so a failing mutant fails
    because of its mutation)."""
    name, rc, tail = _run_pins_against("none", "extern \"C\" {", "extern \"C\" {")
    assert rc == 0, tail
