"""The near-tie validity check (parity.check_row_valid) on the CPU.

Where the oracle reports a near-tie, the GPU's row is checked against the
method's definition instead of against the oracle's choice.  These tests pin
that check: it accepts the oracle's own results on every row of random and
edge-case inputs, accepts the other side of a constructed exact tie (top-p
boundary and race), and rejects planted mistakes of each kind it exists to
catch, on rows far from any tie.
"""

import dataclasses

import numpy as np
import pytest

import oracle
from decode_token_sampling_gb300.workloads import SamplingInputs, make_random
from parity import NEAR_LOG, check_row_valid, compare


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("case", ["plain", "penalty", "special", "ties", "bf16", "greedy", "no_q"])
def test_accepts_the_oracle_on_every_row(case):
    kw = dict(plain={}, penalty=dict(penalty=1.3, n_seen=200), special=dict(special=True),
              ties=dict(ties=True), bf16=dict(dtype="bf16"), greedy={}, no_q={})[case]
    inp = make_random(24, 3001, seed=11, **kw)
    if case == "greedy":
        inp.temperature[::2] = 0.0
        inp.top_p[1::4] = 0.0
    if case == "no_q":
        inp.q = None
    ref = oracle.sample(inp, need_logits=True)
    for b in range(inp.B):
        why = check_row_valid(inp, b, int(ref["idx"][b]), ref["filtered"][b])
        assert why is None, (b, why)


def _far_row(inp, ref, gap=1e-3):
    """A row with top-p active, several kept elements and no near tie of either kind."""
    for b in range(inp.B):
        if ref["kept"][b] >= 3 and ref["topp_gap"][b] > gap and ref["race_gap"][b] > gap and 0 < inp.top_p[b] < 1 \
                and inp.temperature[b] > 0:
            return b
    raise AssertionError("no far row")


def _setup():
    inp = make_random(32, 2000, seed=5, k_range=(20, 600), k_skip_frac=0.0, p_range=(0.3, 0.9))
    ref = oracle.sample(inp, need_logits=True)
    b = _far_row(inp, ref)
    return inp, ref, b, oracle.row_terms(inp, b)


def test_rejects_planted_mistakes():
    inp, ref, b, t = _setup()
    row, idx = ref["filtered"][b], int(ref["idx"][b])
    order, n = t["order"], int(ref["kept"][b])
    x = t["x"]

    def check(r, i):
        return check_row_valid(inp, b, i, r, t)

    assert check(row, idx) is None
    # a hole in the prefix: drop the second element, keep the (n+1)-th instead
    r = row.copy()
    r[order[1]] = -np.inf
    r[order[n]] = x[order[n]]
    assert "prefix" in check(r, idx if idx != order[1] else int(order[0]))
    # one element short of the top-p target
    r = row.copy()
    r[order[n - 1]] = -np.inf
    i = idx if idx != order[n - 1] else int(order[0])
    assert "short" in check(r, i)
    # one element past the target
    r = row.copy()
    r[order[n]] = x[order[n]]
    assert "above" in check(r, idx)
    # a kept value altered
    r = row.copy()
    r[order[0]] = x[order[0]] * (1 + 1e-3) + 1e-3
    assert "values" in check(r, idx)
    # a token outside the kept set
    assert "not kept" in check(row, int(order[n]))
    # the runner-up of the race
    kept = order[:n]
    with np.errstate(divide="ignore"):
        scores = t["e"][:n] / (inp.q[b, kept].astype(np.float64) + inp.eps)
    second = int(kept[np.argsort(-scores)[1]])
    assert "below the best" in check(row, second)
    assert "out of range" in check(row, inp.V)


def test_rejects_wrong_counts_on_greedy_and_topp_off_rows():
    inp, ref, b, t = _setup()
    inp2 = dataclasses.replace(inp, temperature=inp.temperature.copy(), top_p=inp.top_p.copy())
    inp2.temperature[b] = 0.0  # greedy: exactly pi's first
    t2 = oracle.row_terms(inp2, b)
    r = np.full(inp.V, -np.inf, np.float32)
    r[t2["order"][:2]] = t2["x"][t2["order"][:2]]
    assert "greedy" in check_row_valid(inp2, b, int(t2["order"][0]), r, t2)
    inp2.temperature[b] = inp.temperature[b]
    inp2.top_p[b] = 1.0  # top-p off: the whole top-k set
    t3 = oracle.row_terms(inp2, b)
    r = np.full(inp.V, -np.inf, np.float32)
    r[t3["order"][:-1]] = t3["x"][t3["order"][:-1]]
    assert "top-p off" in check_row_valid(inp2, b, int(t3["order"][0]), r, t3)


def _tied_row():
    """V=8, all logits 0, top-k off, p=0.5: every weight is 1, S=8, p*S=4 exactly, so the
    oracle keeps 4 (the 5th element's exclusive mass 4 is not below 4) and keeping 5 is on
    the boundary.  q equal on tokens 0 and 3, larger elsewhere: the race ties 0 and 3."""
    V = 8
    q = np.full((1, V), 2.0, np.float32)
    q[0, 0] = q[0, 3] = 1.0
    return SamplingInputs(name="tied", dtype="f32", B=1, V=V, logits=np.zeros((1, V), np.float32),
                          top_k=np.array([0], np.int32), top_p=np.array([0.5], np.float32),
                          temperature=np.array([1.0], np.float32), q=q, eps=1e-20, need_logits=True)


def test_accepts_the_other_side_of_an_exact_tie():
    inp = _tied_row()
    ref = oracle.sample(inp, need_logits=True)
    assert ref["kept"][0] == 4 and ref["idx"][0] == 0
    assert ref["topp_gap"][0] == 0.0 and ref["race_gap"][0] == 0.0
    five = np.zeros(inp.V, np.float32)
    five[5:] = -np.inf
    assert check_row_valid(inp, 0, 3, five) is None  # boundary element kept, other tied token chosen
    three = np.zeros(inp.V, np.float32)
    three[3:] = -np.inf
    assert "short" in check_row_valid(inp, 0, 0, three)
    assert "below the best" in check_row_valid(inp, 0, 1, ref["filtered"][0])


def test_compare_accepts_a_valid_near_tie_and_logs_it():
    inp = _tied_row()
    ref = oracle.sample(inp, need_logits=True)
    five = np.zeros((1, inp.V), np.float32)
    five[0, 5:] = -np.inf
    n0 = len(NEAR_LOG)
    assert compare(inp, ref, np.array([3]), five, "tied") == [0]
    assert NEAR_LOG[n0][1:] == ("tied", 1, 1, 1)
    with pytest.raises(AssertionError, match="near-tie row invalid"):
        compare(inp, ref, np.array([1]), five, "tied, runner-up")
