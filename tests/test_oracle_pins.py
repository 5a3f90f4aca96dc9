"""Pins for the CPU oracle: the pages' worked examples, brute force on tiny rows,
invariants the method must satisfy, and the race's sampling distribution.

None of these re-types the oracle's own code: the brute-force reference below
uses rank counting and subset enumeration instead of sorting + cumsum, and the
race is checked statistically against the categorical distribution it must
sample from.
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from golden_io import floats, read_pairs

NEG_INF = float("-inf")


def run1(logits, top_k=0, top_p=1.0, temperature=1.0, q=None, seen=None, penalty=None,
         need_logits=True, dtype="f32"):
    """Oracle on a single row given as a Python list."""
    x = np.asarray([logits], dtype=np.float32)
    V = x.shape[1]
    q = np.ones((1, V), np.float32) if q is None else np.asarray([q], np.float32)
    kw = {}
    if seen is not None:
        kw = dict(seen_indptr=np.array([0, len(seen)], np.int32), seen_ids=np.array(seen, np.int32),
                  penalty=np.array([penalty], np.float32))
    return oracle.sample_arrays(x, dtype, [top_k], [top_p], [temperature], q, 1e-20, need_logits, **kw)


# ----------------------------------------------------------------------------------------------
# Worked examples printed on the pages (tests/golden/*.txt, each with its citation)
# ----------------------------------------------------------------------------------------------

def test_golden_topk_example():
    d = dict(read_pairs("topk_worked_example.txt"))
    logits = floats(d["logits"])
    r = run1(logits, top_k=int(d["top_k"]))
    np.testing.assert_array_equal(r["filtered"][0], np.array(floats(d["filtered"]), np.float32))
    assert r["kept"][0] == 3
    assert r["idx"][0] == 1  # q == 1: the race picks the most probable kept token (5.0)


def test_golden_topp_example():
    d = dict(read_pairs("topp_worked_example.txt"))
    probs = floats(d["sorted_probs"])
    # place the tokens in a scrambled vocabulary order; logits = log(prob) (any shift)
    perm = [3, 0, 4, 1, 2]
    logits = [0.0] * 5
    for rank, v in enumerate(perm):
        logits[v] = math.log(probs[rank]) + 1.5
    r = run1(logits, top_k=0, top_p=float(d["top_p"]))
    kept = int(d["kept"])
    assert r["kept"][0] == kept
    finite = np.isfinite(r["filtered"][0])
    assert sorted(np.nonzero(finite)[0].tolist()) == sorted(perm[:kept])


def test_golden_penalty_example():
    pairs = read_pairs("penalty_worked_example.txt")
    pen = float(pairs[0][1])
    cases = [(float(pairs[i][1]), float(pairs[i + 1][1]), int(pairs[i + 2][1])) for i in range(1, len(pairs), 3)]
    scores = [c[0] for c in cases] + [0.75]  # last token is never seen
    # token 0 listed twice: the penalty is applied once per distinct id
    r = run1(scores, top_k=0, top_p=1.0, seen=[0, 1, 0, 1], penalty=pen)
    out = r["filtered"][0]
    for v, (_, want, dec) in enumerate(cases):
        assert round(float(out[v]), dec) == pytest.approx(want, abs=0.5 * 10 ** -dec)
    assert out[2] == np.float32(0.75)


def test_golden_temperature_scaled_logits():
    pairs = read_pairs("temperature_scaled_logits.txt")
    logits = floats(pairs[0][1])
    for i in range(1, len(pairs), 2):
        T = float(pairs[i][1])
        want = floats(pairs[i + 1][1])
        r = run1(logits, top_k=0, top_p=1.0, temperature=T)
        np.testing.assert_array_equal(r["filtered"][0], np.array(want, np.float32))


# ----------------------------------------------------------------------------------------------
# Brute force on tiny rows (independent formulation)
# ----------------------------------------------------------------------------------------------

def brute_row(x32, k, p, T, q, eps, seen, pen):
    """Reference for one tiny row: rank counting for top-k, subset enumeration for top-p."""
    x = [np.float32(v) for v in x32]
    V = len(x)
    x = [np.float32(NEG_INF) if np.isnan(v) else v for v in x]
    if seen is not None and pen > 0:
        for v in sorted(set(i for i in seen if 0 <= i < V)):
            x[v] = np.float32(x[v] / np.float32(pen)) if x[v] > 0 else np.float32(x[v] * np.float32(pen))
    greedy = not (T > 0) or math.isinf(T)
    if not greedy:
        x = [np.float32(v / np.float32(T)) for v in x]
    xf = [float(v) for v in x]

    def precedes(u, v):  # u comes before v in the order (value desc, index asc)
        return xf[u] > xf[v] or (xf[u] == xf[v] and u < v)

    rank = [sum(precedes(u, v) for u in range(V)) for v in range(V)]
    topk_on = 1 <= k <= min(V, 1024)
    K = [v for v in range(V) if (rank[v] < k if topk_on else True)]
    first = min(K, key=lambda v: rank[v])
    M = xf[first]
    e = {v: (1.0 if xf[v] == M else math.exp(xf[v] - M)) for v in K}
    S = sum(e.values())
    if greedy or p <= 0:
        m = 1
    elif p < 1:
        target = p * S
        m = None
        for size in range(1, len(K) + 1):
            if any(sum(e[v] for v in U) >= target for U in itertools.combinations(K, size)):
                m = size
                break
    else:
        m = len(K)
    P = sorted(K, key=lambda v: rank[v])[:m]
    SP = sum(e[v] for v in P)
    best, rb = None, None
    for v in sorted(P):
        r = (e[v] / SP) / (float(q[v]) + float(np.float32(eps)))
        if math.isnan(r):
            continue
        if best is None or r > rb:
            best, rb = v, r
    if best is None:
        best = first
    return best, set(P), x


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny_rows(seed):
    rng = np.random.default_rng(1000 + seed)
    n_rows = 150
    for _ in range(n_rows):
        V = int(rng.integers(1, 10))
        mode = rng.integers(0, 4)
        if mode == 0:
            x = rng.normal(0, 2, V)
        elif mode == 1:  # heavy ties
            x = rng.integers(-2, 3, V).astype(float)
        elif mode == 2:  # specials
            x = rng.normal(0, 2, V)
            x[rng.random(V) < 0.2] = np.nan
            x[rng.random(V) < 0.2] = -np.inf
        else:
            x = np.full(V, 0.5)
        x = x.astype(np.float32)
        k = int(rng.choice([0, -1, 1, 2, 3, V, V + 1, 1025]))
        p = float(np.float32(rng.choice([0.0, -0.5, 0.3, 0.6, 0.9, 0.999, 1.0, 1.5])))
        T = float(np.float32(rng.choice([1.0, 0.7, 1.3, 0.0, -1.0])))
        q = rng.exponential(1.0, V).astype(np.float32)
        if rng.random() < 0.25:  # NaN draws: their race scores take no part
            q[rng.random(V) < 0.4] = np.nan
        seen = rng.integers(-1, V + 1, 4).tolist() if rng.random() < 0.5 else None
        pen = 1.3
        r = oracle.sample_arrays(x[None], "f32", [k], [p], [T], q[None], 1e-20, True,
                                 *( (np.array([0, len(seen)], np.int32), np.array(seen, np.int32),
                                     np.array([pen], np.float32)) if seen is not None else (None, None, None)))
        if r["topp_gap"][0] < 1e-9 or r["race_gap"][0] < 1e-9:
            continue  # a decision within rounding of a tie; not a pin
        want_idx, want_P, xt = brute_row(x, k, p, T, q, 1e-20, seen, pen)
        # -inf values can be kept too (they carry zero mass and print as -inf): compare the
        # kept count and the set of kept finite values
        got_finite = set(np.nonzero(np.isfinite(r["filtered"][0]))[0].tolist())
        assert r["kept"][0] == len(want_P), (x, k, p, T)
        assert {v for v in want_P if np.isfinite(xt[v])} == got_finite
        assert r["idx"][0] == want_idx, (x, k, p, T, q)
        for v in want_P:
            if np.isfinite(xt[v]):
                assert r["filtered"][0][v] == xt[v]


def test_nan_draws_take_no_part_in_the_race():
    """A NaN draw makes its token's race score NaN, and NaN scores are ignored: the best
    of the others wins, and with every score NaN the first token of the order is chosen
    (the reading of the race's argmax for NaN scores).  Expected values from brute_row."""
    x = np.array([3.0, 2.0, 1.0, 0.0], np.float32)
    nan = np.float32(np.nan)
    cases = [[nan, 1.0, 1.0, 1.0], [1.0, nan, 0.01, 1.0], [nan, nan, nan, nan], [nan, nan, nan, 0.5]]
    for q in cases:
        q = np.array(q, np.float32)
        r = run1(x.tolist(), top_k=0, top_p=1.0, temperature=1.0, q=q.tolist())
        want, _, _ = brute_row(x, 0, 1.0, 1.0, q, 1e-20, None, 0.0)
        assert r["idx"][0] == want, (q, r["idx"][0], want)
    assert [run1(x.tolist(), q=c)["idx"][0] for c in cases] == [1, 2, 0, 3]


# ----------------------------------------------------------------------------------------------
# Invariants
# ----------------------------------------------------------------------------------------------

def _rows(seed, B=40, V=300, **kw):
    from decode_token_sampling_gb300.workloads import make_random
    return make_random(B, V, seed=seed, **kw)


def _order_first(x):
    """Index of the first element in the order (value desc, index asc)."""
    m = np.max(x)
    return int(np.nonzero(x == m)[0][0])


def _transformed(inp):
    """Penalty + temperature applied with numpy float32 IEEE ops (no selection)."""
    r = oracle.sample_arrays(inp.logits, inp.dtype, np.zeros(inp.B, np.int32), np.ones(inp.B, np.float32),
                             inp.temperature, inp.q, inp.eps, True, inp.seen_indptr, inp.seen_ids, inp.penalty)
    return r["filtered"]


def test_kept_set_is_prefix_of_order():
    inp = _rows(1, penalty=1.2, n_seen=20)
    r = oracle.sample(inp)
    x = _transformed(inp)
    for b in range(inp.B):
        f = r["filtered"][b]
        kept = np.nonzero(f != NEG_INF)[0]
        if len(kept) == 0:
            continue
        order = sorted(range(inp.V), key=lambda v: (-x[b][v], v))
        prefix = set(order[: r["kept"][b]])
        assert set(kept.tolist()) <= prefix
        assert r["idx"][b] in prefix


def test_k1_and_p0_give_argmax():
    inp = _rows(2)
    x = _transformed(inp)
    for variant in ("k1", "p0", "pneg", "ptiny"):
        k = inp.top_k.copy()
        p = inp.top_p.copy()
        if variant == "k1":
            k[:] = 1
        elif variant == "p0":
            p[:] = 0.0
        elif variant == "pneg":
            p[:] = -1.0
        else:
            k[:] = 0
            p[:] = 1e-12
        r = oracle.sample_arrays(inp.logits, "f32", k, p, inp.temperature, inp.q)
        for b in range(inp.B):
            assert r["idx"][b] == _order_first(x[b])
            assert r["kept"][b] == 1


def test_skipped_stages_are_identity():
    inp = _rows(3, penalty=1.1, n_seen=10)
    x = _transformed(inp)
    for k in (0, -1, 1025, inp.V + 7):
        r = oracle.sample_arrays(inp.logits, "f32", np.full(inp.B, k, np.int32), np.ones(inp.B, np.float32),
                                 inp.temperature, inp.q, 1e-20, True, inp.seen_indptr, inp.seen_ids, inp.penalty)
        np.testing.assert_array_equal(r["filtered"], x)
        assert (r["kept"] == inp.V).all()
    r = oracle.sample_arrays(inp.logits, "f32", np.zeros(inp.B, np.int32), np.full(inp.B, np.nan, np.float32),
                             inp.temperature, inp.q)
    assert (r["kept"] == inp.V).all()


def test_penalty_one_is_identity():
    inp = _rows(4, penalty=1.0, n_seen=50)
    a = oracle.sample(inp)
    b = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, inp.q)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["filtered"], b["filtered"])


def test_nonpositive_penalty_is_skipped():
    inp = _rows(5, penalty=-2.0, n_seen=50)
    a = oracle.sample(inp)
    b = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, inp.q)
    np.testing.assert_array_equal(a["filtered"], b["filtered"])


def test_unit_q_picks_argmax_of_filtered():
    inp = _rows(6)
    q1 = np.ones_like(inp.q)
    r = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, q1)
    for b in range(inp.B):
        assert r["idx"][b] == _order_first(r["filtered"][b])


def test_greedy_temperature_rows():
    x = np.array([[0.5, 3.0, 3.0, -1.0, 2.9]], np.float32)
    for T in (0.0, -1.0, float("nan"), float("inf")):
        r = oracle.sample_arrays(x, "f32", [0], [0.9], [T], np.full((1, 5), 0.01, np.float32))
        assert r["idx"][0] == 1 and r["kept"][0] == 1
        assert r["filtered"][0][1] == np.float32(3.0)  # no division on a greedy row


def test_nan_logits_are_minus_inf():
    x = np.array([[np.nan, 1.0, np.nan, 0.0]], np.float32)
    r = oracle.sample_arrays(x, "f32", [0], [1.0], [1.0], np.ones((1, 4), np.float32))
    assert r["filtered"][0][0] == NEG_INF and r["filtered"][0][2] == NEG_INF
    assert r["idx"][0] == 1


def test_bf16_is_widened_exactly():
    from decode_token_sampling_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits
    rng = np.random.default_rng(7)
    x = rng.normal(0, 3, (3, 257)).astype(np.float32)
    h = f32_to_bf16_bits(x)
    k = np.array([5, 0, 300], np.int32)
    p = np.array([0.9, 0.8, 1.0], np.float32)
    t = np.array([0.7, 1.0, 1.3], np.float32)
    q = rng.exponential(1, (3, 257)).astype(np.float32)
    a = oracle.sample_arrays(h, "bf16", k, p, t, q)
    b = oracle.sample_arrays(bf16_bits_to_f32(h), "f32", k, p, t, q)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["filtered"], b["filtered"])


def test_race_samples_the_kept_distribution():
    """With q ~ Exp(1), argmax of p_i / q_i is distributed as p (a standard fact about
    exponential races); chi-square over 1e5 draws on an 8-token row."""
    V, N = 8, 100_000
    logits = np.array([1.2, -0.3, 0.8, 2.0, 0.1, -1.0, 1.9, 0.5], np.float32)
    rng = np.random.default_rng(12345)
    q = rng.exponential(1.0, (N, V)).astype(np.float32)
    x = np.repeat(logits[None], N, axis=0)
    k, p, T = 6, 0.95, 0.9
    r = oracle.sample_arrays(x, "f32", np.full(N, k, np.int32), np.full(N, p, np.float32),
                             np.full(N, T, np.float32), q, 1e-20, False)
    xt = (logits / np.float32(T)).astype(np.float64)
    order = sorted(range(V), key=lambda v: (-xt[v], v))
    K = order[:k]
    w = np.exp(xt[K] - xt[K].max())
    w /= w.sum()
    cum = np.cumsum(w)
    m = int(np.searchsorted(cum, p) + 1)  # shortest prefix whose mass reaches p
    P = K[:m]
    pw = w[:m] / w[:m].sum()
    counts = np.array([(r["idx"] == v).sum() for v in P])
    assert counts.sum() == N  # nothing outside the kept set is ever chosen
    expected = pw * N
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    dof = len(P) - 1
    # 99.9% quantile of chi-square with dof <= 5 is below 20.6
    assert chi2 < 20.6, (chi2, counts, expected)


def test_deterministic():
    inp = _rows(8, penalty=1.1, n_seen=30)
    a = oracle.sample(inp)
    b = oracle.sample(inp)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["filtered"], b["filtered"])


def test_rejects_bad_arguments():
    x = np.zeros((1, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.sample_arrays(x, "f16", [0], [1.0], [1.0], np.ones((1, 4), np.float32))


def test_topp_exact_boundary_stops_at_reaching_mass():
    """All-equal rows where p*S is hit exactly by a prefix: the shortest prefix whose
    mass reaches top_p is kept, nothing more (exact in binary: masses are 1.0 each)."""
    for V, p, want in ((4, 0.5, 2), (8, 0.25, 2), (8, 0.75, 6), (8, 0.125, 1), (16, 0.5, 8)):
        r = run1([0.25] * V, top_k=0, top_p=p)
        assert r["kept"][0] == want, (V, p)
        assert sorted(np.nonzero(np.isfinite(r["filtered"][0]))[0].tolist()) == list(range(want))


def test_topk_above_1024_is_skipped_even_when_below_V():
    inp = _rows(9, B=4, V=2000)
    x = _transformed(inp)
    for k in (1025, 1500, 2000):
        r = oracle.sample_arrays(inp.logits, "f32", np.full(inp.B, k, np.int32), np.ones(inp.B, np.float32),
                                 inp.temperature, inp.q)
        np.testing.assert_array_equal(r["filtered"], x)
    r = oracle.sample_arrays(inp.logits, "f32", np.full(inp.B, 1024, np.int32), np.ones(inp.B, np.float32),
                             inp.temperature, inp.q)
    assert (r["kept"] == 1024).all()


def test_race_exact_tie_takes_lower_index():
    # tokens 1 and 3 have equal logits and equal q: equal race scores
    x = [1.0, 3.0, 0.5, 3.0, -2.0]
    q = [5.0, 0.25, 9.0, 0.25, 9.0]
    r = run1(x, top_k=0, top_p=1.0, q=q)
    assert r["idx"][0] == 1
    # mirror the vocabulary: the winner is again the lower index of the tied pair
    r = run1(x[::-1], top_k=0, top_p=1.0, q=q[::-1])
    assert r["idx"][0] == 1


def test_sampling_off_takes_the_first_of_the_order():
    """q absent (sampling off): the argmax of the filtered row, the lowest index among equal
    maxima [NPU scenario table, Sample disabled; MM10 greedy mode]; the kept set and the
    filtered row are those of a sampled call."""
    inp = _rows(6)
    x = _transformed(inp)
    off = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, None)
    on = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, inp.q)
    for b in range(inp.B):
        assert off["idx"][b] == _order_first(x[b])
        assert off["kept"][b] == on["kept"][b]
        assert np.array_equal(off["filtered"][b], on["filtered"][b])
        assert math.isinf(off["race_gap"][b])
    # equal maxima: the lower index
    r = oracle.sample_arrays(np.array([[3.0, 5.0, 5.0, -1.0]], np.float32), "f32", [0], [0.99], [1.0], None)
    assert r["idx"][0] == 1


# ----------------------------------------------------------------------------------------------
# Generated Exp(1) draws (a seeded call races with these instead of a supplied q)
# ----------------------------------------------------------------------------------------------

def test_philox_known_answers():
    """The generator reproduces the published Philox4x32-10 known-answer vectors."""
    pairs = read_pairs("philox4x32_10_kat.txt")
    hexes = lambda s: [int(t, 16) for t in s.split()]
    n = 0
    for i in range(0, len(pairs), 3):
        (kc, c), (kk, k), (ko, o) = pairs[i:i + 3]
        assert (kc, kk, ko) == ("counter", "key", "out")
        assert oracle.philox4x32_10(hexes(c), hexes(k)) == hexes(o)
        n += 1
    assert n == 3


def test_exp_draws_follow_their_definition():
    """Each draw is -log(u) of its own Philox word: counter (v/4, row, step), word v mod 4."""
    seed, step = 0x0123456789ABCDEF, 7
    q = oracle.exp_draws(3, 10, seed, step)
    for b in range(3):
        for v in range(10):
            w = oracle.philox4x32_10([v // 4, b, step & 0xFFFFFFFF, step >> 32],
                                     [seed & 0xFFFFFFFF, seed >> 32])[v % 4]
            u = (2 * (w >> 9) + 1) / 2.0**24
            assert q[b, v] == np.float32(-math.log(u))
    # a different step or seed gives different draws
    assert not np.array_equal(q, oracle.exp_draws(3, 10, seed, step + 1))
    assert not np.array_equal(q, oracle.exp_draws(3, 10, seed + 1, step))


def test_exp_draws_are_exp1():
    """Kolmogorov-Smirnov distance to the Exp(1) distribution, mean and variance, and no
    correlation between neighbouring tokens or rows, over 10^6 draws."""
    q = oracle.exp_draws(100, 10000, seed=2024, step=3).astype(np.float64)
    x = np.sort(q.ravel())
    n = x.size
    cdf = 1.0 - np.exp(-x)
    ks = max(np.max(np.arange(1, n + 1) / n - cdf), np.max(cdf - np.arange(0, n) / n))
    assert ks < 1.95 / math.sqrt(n)  # about the 0.1% critical value
    assert abs(x.mean() - 1.0) < 5e-3 and abs(x.var() - 1.0) < 1e-2
    assert abs(np.corrcoef(q[:, :-1].ravel(), q[:, 1:].ravel())[0, 1]) < 5e-3
    assert abs(np.corrcoef(q[:-1].ravel(), q[1:].ravel())[0, 1]) < 5e-3


def test_eos_epilogue_follows_the_generate_loop():
    """MiniMind's generate loop: a finished sequence emits eos, a sequence that emits eos is
    finished, and the loop may stop when none is left."""
    idx = np.array([5, 2, 7, 2, 9], np.int64)
    fin = np.array([0, 0, 1, 0, 1], np.uint8)
    left = oracle.eos_epilogue(idx, fin, 2)
    assert idx.tolist() == [5, 2, 2, 2, 2]
    assert fin.tolist() == [0, 1, 1, 1, 1]
    assert left == 1
    idx = np.array([2, 2], np.int64)
    fin = np.zeros(2, np.uint8)
    assert oracle.eos_epilogue(idx, fin, 2) == 0 and fin.tolist() == [1, 1]


# ----------------------------------------------------------------------------------------------
# The seen set kept as bits across decode steps (MiniMind ch.10: the repetition penalty runs
# over the unique ids of the sequence so far; the generate loop appends each step's token)
# ----------------------------------------------------------------------------------------------

def _bits_of(sets, V, junk_rng=None):
    """Bit matrix of Python id sets (plus, when junk_rng is given, random bits above V)."""
    W = (V + 31) // 32
    bits = np.zeros((len(sets), W), np.uint32)
    for b, s in enumerate(sets):
        for v in s:
            bits[b, v // 32] |= np.uint32(1 << (v % 32))
        if junk_rng is not None and V % 32:
            bits[b, W - 1] |= np.uint32(int(junk_rng.integers(1, 2**32)) & ~((1 << (V % 32)) - 1) & 0xFFFFFFFF)
    return bits


def test_seen_ids_from_bits_lists_each_set_once():
    rng = np.random.default_rng(77)
    V = 70  # three words; bits 70..95 of the last one are not tokens
    sets = [set(), {0}, {69}, set(int(v) for v in rng.integers(0, V, 40)), set(range(V))]
    bits = _bits_of(sets, V, junk_rng=rng)
    indptr, ids = oracle.seen_ids_from_bits(bits, V)
    assert indptr[0] == 0 and indptr.shape == (len(sets) + 1,)
    for b, s in enumerate(sets):
        assert ids[indptr[b]:indptr[b + 1]].tolist() == sorted(s)


def test_seen_append_adds_the_token_only():
    V = 70
    sets = [{1, 2}, set(), {40}, {5}, {6}]
    bits = _bits_of(sets, V)
    idx = np.array([3, 69, 40, -1, V], np.int64)  # in range, top token, already seen, outside x2
    oracle.seen_append(bits, idx, V)
    indptr, ids = oracle.seen_ids_from_bits(bits, V)
    want = [{1, 2, 3}, {69}, {40}, {5}, {6}]
    for b, s in enumerate(want):
        assert ids[indptr[b]:indptr[b + 1]].tolist() == sorted(s)


def test_penalty_over_bits_equals_penalty_over_the_id_list():
    """The penalty depends on the set alone: a list with duplicates and out-of-range ids and the
    bit form of its distinct in-range ids give the same result."""
    rng = np.random.default_rng(78)
    B, V = 6, 300
    x = rng.normal(0, 2, (B, V)).astype(np.float32)
    lists = [list(rng.integers(-5, V + 5, 60)) + [7, 7, 7] for _ in range(B)]
    indptr = np.cumsum([0] + [len(l) for l in lists]).astype(np.int32)
    ids = np.concatenate(lists).astype(np.int32)
    pen = np.full(B, 1.3, np.float32)
    kw = dict(top_k=np.array([0, 5, 50, 0, 1, 1025], np.int32), top_p=np.array([1.0, 0.9, 0.7, 0.5, 1.0, 0.95],
              np.float32), temperature=np.array([1.0, 0.8, 1.2, 0.7, 1.0, 0.9], np.float32))
    q = oracle.exp_draws(B, V, 5, 0)
    a = oracle.sample_arrays(x, "f32", kw["top_k"], kw["top_p"], kw["temperature"], q, 1e-20, True, indptr, ids, pen)
    bits = _bits_of([set(int(v) for v in l if 0 <= v < V) for l in lists], V, junk_rng=rng)
    ip2, ids2 = oracle.seen_ids_from_bits(bits, V)
    b = oracle.sample_arrays(x, "f32", kw["top_k"], kw["top_p"], kw["temperature"], q, 1e-20, True, ip2, ids2, pen)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["filtered"], b["filtered"])


def test_incremental_bits_follow_the_generate_loop():
    """Three decode steps: the bits grown by seen_append give the penalty over the unique ids
    of the growing sequence (prompt ids plus every emitted token), built here from a list."""
    rng = np.random.default_rng(79)
    B, V = 5, 200
    seqs = [list(int(v) for v in rng.integers(0, V, 8)) for _ in range(B)]
    bits = _bits_of([set(s) for s in seqs], V)
    pen = np.full(B, 1.5, np.float32)
    top_k = np.array([0, 20, 3, 0, 50], np.int32)
    top_p = np.array([0.9, 1.0, 0.8, 1.0, 0.6], np.float32)
    T = np.ones(B, np.float32)
    for step in range(3):
        x = rng.normal(0, 1, (B, V)).astype(np.float32)
        q = oracle.exp_draws(B, V, 11, step)
        indptr = np.cumsum([0] + [len(s) for s in seqs]).astype(np.int32)
        ref = oracle.sample_arrays(x, "f32", top_k, top_p, T, q, 1e-20, True, indptr,
                                   np.concatenate(seqs).astype(np.int32), pen)
        ip2, ids2 = oracle.seen_ids_from_bits(bits, V)
        got = oracle.sample_arrays(x, "f32", top_k, top_p, T, q, 1e-20, True, ip2, ids2, pen)
        np.testing.assert_array_equal(ref["idx"], got["idx"])
        np.testing.assert_array_equal(ref["filtered"], got["filtered"])
        for b in range(B):
            seqs[b].append(int(ref["idx"][b]))
        oracle.seen_append(bits, got["idx"], V)
    ip3, ids3 = oracle.seen_ids_from_bits(bits, V)
    for b in range(B):
        assert ids3[ip3[b]:ip3[b + 1]].tolist() == sorted(set(seqs[b]))
