"""The error budget of the GPU's weights and race quotients, at its bound (CPU).

The kernels decide the top-p boundary and the race winner in fp32 arithmetic
whose every factor has a bounded relative error (error_budget.py; the GPU test
test_weight_error.py measures each factor over its whole input domain).  If
every element's mass carries a relative error of at most e, the kernel's
top-p count can differ from the exact rule's only where the exact prefix mass
at the boundary lies within 2 (1 - p) e / (1 - e) of p * S (relative), and its
race winner only where the two best scores lie within 2 e / (1 - e) of each
other.  These tests check that both bands lie inside the near-tie band of the
parity rule (1e-6), for every p, and that the top-p band is exact (attained,
and not exceeded) on a flat row of 151936 tokens: with the worst perturbation
of every mass (up on one side of the boundary, down on the other), the count
can change just below the band and cannot just above it.
"""

import numpy as np
import pytest

import oracle
from error_budget import (NEAR, mass_error_topk, mass_error_wide, race_error_topk, race_error_wide,
                          race_flip_band, topp_flip_band)
from decode_token_sampling_gb300.workloads import SamplingInputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("kind", ["wide", "topk"])
def test_bands_inside_the_near_tie_band(kind):
    em = mass_error_wide() if kind == "wide" else mass_error_topk()
    er = race_error_wide() if kind == "wide" else race_error_topk()
    for p in np.linspace(0.0, 1.0, 101)[1:-1]:
        assert topp_flip_band(em, p) < NEAR, (p, topp_flip_band(em, p))
    assert topp_flip_band(em, 1e-9) < NEAR
    assert race_flip_band(er) < NEAR, race_flip_band(er)


def _flat_row(V=151936, seed=4):
    """One row like the full-vocabulary nucleus workload: N(0, 0.5) fp32 logits, top-k off,
    temperature 1."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 0.5, (1, V)).astype(np.float32)
    return SamplingInputs(name="flat", dtype="f32", B=1, V=V, logits=x, top_k=np.zeros(1, np.int32),
                          top_p=np.full(1, 0.9, np.float32), temperature=np.ones(1, np.float32),
                          q=None, eps=1e-20, need_logits=False)


def _count_can_change(c_before, c_at, S, p, e):
    """Whether masses each perturbed by a factor in [1 - e, 1 + e] can move the top-p count
    away from the exact count n (c_before = mass of the first n - 1 elements, c_at = of the
    first n): fewer kept if the first n - 1 can reach p * S (all of them up, the rest
    down); more kept if the first n can fall short of it (them down, the rest up)."""
    fewer = (1 - p) * c_before * (1 + e) - p * (S - c_before) * (1 - e) >= 0
    more = (1 - p) * c_at * (1 - e) - p * (S - c_at) * (1 + e) < 0
    return fewer or more


@pytest.mark.parametrize("n", [300, 3000, 12000, 40000])
def test_topp_band_is_exact_on_a_flat_row(n):
    """p swept over the 81 floats nearest c_n / S (the mass of the first n elements of the order
    over the total): at each, the oracle's count and boundary gap against what masses off by the
    budget's e could do.  The count can change exactly when the gap is inside the band."""
    inp = _flat_row()
    t = oracle.row_terms(inp, 0)
    assert t["nK"] == inp.V and not t["greedy"]
    c = np.concatenate([[0.0], np.cumsum(t["e"])])
    S = t["S"]
    e = mass_error_wide()
    ps = [np.float32(c[n] / S)]
    for direction in (np.float32(-1.0), np.float32(2.0)):
        q = ps[0]
        for _ in range(40):
            q = np.nextafter(q, direction)
            ps.append(q)
    seen = set()
    for k, p32 in enumerate(ps):
        p = float(p32)
        inp.top_p[0] = p32
        ref = oracle.sample(inp, need_logits=False)
        kept = int(ref["kept"][0])
        gap = float(ref["topp_gap"][0])
        can = _count_can_change(c[kept - 1], c[kept], S, p, e)
        band = topp_flip_band(e, p)
        if gap > 1.01 * band:
            assert not can, (k, gap, band)
        if gap < 0.99 * band:
            assert can, (k, gap, band)
        if can:
            assert gap < NEAR, (k, gap)
        seen.add(can)
    assert seen == {True, False}  # the sweep crosses the band's edge


def test_race_band_is_exact():
    e = race_error_wide()
    band = race_flip_band(e)
    r1 = 1.0
    for factor, flips in ((0.99, True), (1.01, False)):
        r2 = r1 * (1 - factor * band)
        # the runner-up up by e and the best down by e
        assert (r2 * (1 + e) >= r1 * (1 - e)) == flips
