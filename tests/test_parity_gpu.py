"""GPU path vs the CPU oracle, element by element, through the C ABI.

Covers the five named workloads at full size (the B=256, V=151936 one in the
same launch configuration the benchmark times), ragged and tiny vocabularies
that span several CTAs with ragged tails, heavy ties, NaN/-inf logits,
penalties with duplicate and out-of-range ids, and the per-row edge cases of
every stage (top-k out of range, top-p <= 0 / >= 1 / NaN, temperature <= 0 /
NaN / inf).
"""

import dataclasses

import numpy as np
import pytest

import oracle
from decode_token_sampling_gb300.workloads import WORKLOADS, make_random, make_workload
from parity import NEAR, check_row_valid, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_token_sampling_gb300 import build
    build.build()
    oracle.build()


@pytest.fixture(params=["cluster", "row", "row_exact", "auto"])
def kernel(request):
    """Runs the test under each kernel policy: the cluster kernel alone, the row kernel
    alone (it only takes aligned rows; other shapes fall back to the cluster kernel),
    the row kernel with its exact whole-row selection forced on every row (the path a
    missed sample or an overflowing band takes), and the automatic choice by batch size."""
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy({"cluster": kps.KERNEL_CLUSTER, "row": kps.KERNEL_ROW,
                           "row_exact": kps.KERNEL_ROW_EXACT, "auto": kps.KERNEL_AUTO}[request.param])
    yield request.param
    kps.set_kernel_policy(kps.KERNEL_AUTO)


@pytest.mark.parametrize("name", WORKLOADS)
def test_named_workloads(name, kernel):
    inp = make_workload(name)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"{name} [{kernel}]")
    if not inp.need_logits:  # also check the filtered output of the same workload
        ref = oracle.sample(inp, need_logits=True)
        gi, gf = run_gpu(inp, need_logits=True)
        compare(inp, ref, gi, gf, f"{name}+logits [{kernel}]")


@pytest.mark.parametrize("V", [1, 2, 7, 31, 33, 1023, 1025, 4099, 8191, 8192, 40000, 40960])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_vocab(V, dtype, kernel):
    inp = make_random(6, V, seed=V, dtype=dtype, penalty=1.3, n_seen=min(3 * V, 200))
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"V={V} {dtype}")


@pytest.mark.parametrize("V", [64, 5000, 70001, 70000])
def test_ties_and_specials(V, kernel):
    inp = make_random(12, V, seed=7 + V, ties=True, special=True, penalty=1.5, n_seen=50)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"ties V={V}")


@pytest.mark.parametrize("V", [3000, 20000])
def test_all_equal_rows_split_ties_by_index(V, kernel):
    inp = make_random(8, V, seed=11)
    inp.logits[:] = 0.5
    inp.top_k[:] = [1, 2, 17, 1024, 0, 0, 700, V][:8]
    inp.top_p[:] = [1.0, 0.5, 1.0, 0.25, 0.5, 0.125, 0.99, 1.0]
    inp.temperature[:] = 1.0
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, "all-equal")


@pytest.mark.parametrize("V", [3001, 3000, 12288])
def test_edge_parameters(V, kernel):
    B = 16
    inp = make_random(B, V, seed=99, penalty=1.2, n_seen=40)
    inp.top_k[:] = [0, -1, 1, 1024, 1025, V, V + 7, 5, 50, 1, 0, 3, 2, 1000, 7, 9]
    inp.top_p[:] = [0.0, -1.0, np.nan, 1.0, 1.5, 1e-7, 0.999999, 0.5, 0.9, 0.3, 0.95, 0.0, 1.0, 0.7, np.nan, 0.8]
    inp.temperature[:] = [1.0, 0.0, -1.0, np.nan, np.inf, 0.5, 2.0, 1e-3, 1e3, 1.0, 0.7, 1.0, 0.9, 1.1, 1.0, 1.0]
    inp.penalty[:] = [1.2, 0.0, -1.0, np.nan, 1.0, 1.2, 1.2, 2.0, 0.5, 1.2, 1.2, 1.2, 1.2, 1.2, 1.2, 1.2]
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"edge params V={V}")


@pytest.mark.parametrize("V", [2048, 10240])
def test_q_edge_values(V, kernel):
    inp = make_random(6, V, seed=5)
    inp.q[0, :] = 0.0
    inp.q[1, ::2] = np.inf
    inp.q[2, :] = 1.0
    inp.q[3, 100:200] = np.nan
    inp.q[4, :] = 1e-30
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"q edges V={V}")


def test_zero_rows_is_noop():
    import torch
    import decode_token_sampling_gb300 as kps
    dev = "cuda:0"
    z = torch.empty(0, 100, device=dev)
    idx, f = kps.sample(z, torch.empty(0, dtype=torch.int32, device=dev), torch.empty(0, device=dev),
                        torch.empty(0, device=dev), torch.empty(0, 100, device=dev))
    torch.cuda.synchronize()
    assert idx.numel() == 0 and f is None


def test_status_word_clean_after_runs():
    import torch
    import decode_token_sampling_gb300 as kps
    inp = make_random(4, 5000, seed=3)
    ws = kps.new_workspace(inp.B, inp.V)
    run_gpu(inp, workspace=ws)
    assert kps.last_device_status(ws) == 0


def test_side_stream_and_repeat_determinism():
    import torch
    inp = make_workload("small_mixed")
    s = torch.cuda.Stream()
    a = run_gpu(inp, stream=s)
    b = run_gpu(inp)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("B", [1, 3, 64, 200, 600])
def test_batch_sizes_and_row_walk(B, kernel):
    """Persistent grids walk several rows per CTA / cluster when B exceeds the resident slots."""
    inp = make_random(B, 16384, seed=40 + B, penalty=1.2, n_seen=100)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"B={B} [{kernel}]")


PREC_BYTES = 32896  # one pre-pass record (bin sums, race words, the maximum and H)


@pytest.mark.parametrize("name", ["batch256_penalty", "flat_nucleus"])
@pytest.mark.parametrize("records", [0, 3])
def test_row_kernel_with_few_pre_pass_records(name, records):
    """A workspace with room for no (or only 3) pre-pass records: the top-p-only rows beyond
    them run their own pass A inside the row kernel.  Same results as the oracle."""
    import torch
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_workload(name)
        ref = oracle.sample(inp)
        ws = torch.zeros(256 + records * PREC_BYTES, dtype=torch.uint8, device="cuda:0")
        gi, gf = run_gpu(inp, workspace=ws)
        compare(inp, ref, gi, gf, f"{name} [{records} records]")
        assert kps.last_device_status(ws) == 0
        assert int(ws[256:].count_nonzero().item()) == 0
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


@pytest.mark.parametrize("name", ["batch256_penalty", "flat_nucleus"])
def test_pre_pass_leaves_its_records_zeroed(name):
    """The row kernel clears every pre-pass record it reads: several calls on one workspace
    give the oracle's results and leave everything past the status word zero."""
    import torch
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_workload(name)
        ref = oracle.sample(inp)
        ws = kps.new_workspace(inp.B, inp.V, torch.float32, "cuda:0")
        assert ws.numel() >= 256 + PREC_BYTES * min(inp.B, 1024)
        for _ in range(3):
            gi, gf = run_gpu(inp, workspace=ws)
            compare(inp, ref, gi, gf, f"{name} [reused workspace]")
        assert kps.last_device_status(ws) == 0
        assert int(ws[256:].count_nonzero().item()) == 0
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pre_pass_with_many_top_p_rows(dtype):
    """More rows than the grid has clusters, most of them top-p-only (so their pass A runs in
    the pre-pass, several chunks to a row), with penalties, a vocabulary that is no multiple
    of a tile (rows still start on 16-byte boundaries, as the row kernel needs) and some
    top-k rows between them."""
    import torch
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_random(400, 12296, seed=41, dtype=dtype, k_range=(1, 64), k_skip_frac=0.8,
                          p_range=(0.3, 0.999), penalty=1.3, n_seen=40)
        ref = oracle.sample(inp)
        ws = kps.new_workspace(inp.B, inp.V, torch.bfloat16 if dtype == "bf16" else torch.float32, "cuda:0")
        for _ in range(2):
            gi, gf = run_gpu(inp, workspace=ws)
            compare(inp, ref, gi, gf, f"many top-p rows {dtype}")
        assert kps.last_launch_count() == 2
        assert kps.last_device_status(ws) == 0
        assert int(ws[256:].count_nonzero().item()) == 0
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


@pytest.mark.parametrize("case", ["special", "spike", "huge"])
def test_pre_pass_records_on_odd_rows(case):
    """Top-p-only rows whose pre-pass record cannot be used as it stands: NaN and -inf logits
    (special), a maximum the sample misses by far more than the headroom (spike: the row
    redoes its pass A), and logits too large for the 1/32 grid (huge: the exact whole-row
    selection).  Results match the oracle and every record is left zeroed."""
    import torch
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_random(320, 8200, seed=77, k_range=(1, 64), k_skip_frac=0.7, p_range=(0.5, 0.99),
                          special=(case == "special"))
        if case == "spike":
            for b in range(0, inp.B, 3):
                inp.logits[b, (b * 977) % inp.V] = 60.0  # far above the rest, rarely in the sample
        if case == "huge":
            inp.logits[::2] *= 3.0e5
        ref = oracle.sample(inp)
        ws = kps.new_workspace(inp.B, inp.V, torch.float32, "cuda:0")
        for _ in range(2):
            gi, gf = run_gpu(inp, workspace=ws)
            compare(inp, ref, gi, gf, f"odd rows {case}")
        assert kps.last_launch_count() == 2
        assert kps.last_device_status(ws) == 0
        assert int(ws[256:].count_nonzero().item()) == 0
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


@pytest.mark.parametrize("name", ["small_mixed", "batch256_penalty", "flat_nucleus", "single_row_long"])
def test_sampling_off(name, kernel):
    """q absent: every row's index is the first element of its kept set's order (the
    oracle's reading of sampling off); the filtered row is unchanged."""
    inp = make_workload(name)
    inp.q = None
    inp.need_logits = True
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"{name} [sampling off]")


def test_sampling_off_edge_rows():
    """Sampling off on rows with NaN/-inf logits, ties, penalties and edge parameters."""
    inp = make_random(24, 5003, seed=91, ties=True, special=True, penalty=1.5, n_seen=50)
    inp.q = None
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, "edge rows [sampling off]")


@pytest.mark.parametrize("name", WORKLOADS)
def test_generated_draws(name, kernel):
    """kps_sample_seeded: the race with the library's own Philox4x32-10 Exp(1) draws matches
    the oracle racing with the same draws (generated on the CPU from their definition)."""
    seed, step = 0x5EED0000 + WORKLOADS.index(name), 11
    inp = make_workload(name)
    inp.q = oracle.exp_draws(inp.B, inp.V, seed, step)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp, seed=seed, step=step)
    compare(inp, ref, gi, gf, f"{name} [generated draws]",
            rerun=lambda: run_gpu(inp, need_logits=True, seed=seed, step=step))


def test_generated_draws_edge_rows():
    """Generated draws on rows with NaN/-inf logits, ties, penalties and edge parameters, and
    another step of the same seed."""
    inp = make_random(24, 5004, seed=93, ties=True, special=True, penalty=1.5, n_seen=50)
    for step in (0, 2**40 + 3):
        inp.q = oracle.exp_draws(inp.B, inp.V, 77, step)
        ref = oracle.sample(inp)
        gi, gf = run_gpu(inp, seed=77, step=step)
        compare(inp, ref, gi, gf, f"edge rows [generated draws, step {step}]",
                rerun=lambda: run_gpu(inp, need_logits=True, seed=77, step=step))


@pytest.mark.parametrize("draws", ["supplied", "generated"])
def test_eos_epilogue(kernel, draws):
    """kps_sample_step's end-of-sequence epilogue: finished rows emit eos, rows that emit it
    become finished, and the unfinished rows are counted, as the oracle's epilogue does."""
    import torch
    import decode_token_sampling_gb300 as kps
    inp = make_workload("batch256_penalty", rows=range(0, 256, 3))
    seed = 4242
    if draws == "generated":
        inp.q = oracle.exp_draws(inp.B, inp.V, seed, 3)
    ref = oracle.sample(inp)
    rng = np.random.default_rng(5)
    fin0 = (rng.random(inp.B) < 0.3).astype(np.uint8)
    eos = int(ref["idx"][np.nonzero(fin0 == 0)[0][0]])  # an unfinished row emits eos
    ref_idx, ref_fin = ref["idx"].copy(), fin0.copy()
    left = oracle.eos_epilogue(ref_idx, ref_fin, eos)
    dev = "cuda:0"
    fin = torch.from_numpy(fin0.copy()).to(dev)
    unf = torch.full((1,), -5, dtype=torch.int32, device=dev)
    kw = dict(seen_indptr=torch.from_numpy(inp.seen_indptr).to(dev), seen_ids=torch.from_numpy(inp.seen_ids).to(dev),
              penalty=torch.from_numpy(inp.penalty).to(dev))
    idx, filt = kps.sample(torch.from_numpy(inp.logits).to(dev), torch.from_numpy(inp.top_k).to(dev),
                           torch.from_numpy(inp.top_p).to(dev), torch.from_numpy(inp.temperature).to(dev),
                           torch.from_numpy(inp.q).to(dev) if draws == "supplied" else None,
                           seed=seed if draws == "generated" else None, step=3, eps=inp.eps, need_logits=True,
                           finished=fin, eos_id=eos, unfinished=unf, **kw)
    torch.cuda.synchronize()
    got, gf = idx.cpu().numpy(), filt.cpu().numpy()
    # an unfinished row where the GPU chose another token must sit at a near-tie and be valid
    # by the definition; the expected epilogue then starts from the GPU's choice in that row
    near = (ref["race_gap"] < NEAR) | (ref["topp_gap"] < NEAR)
    pre = ref["idx"].copy()
    for b in np.nonzero((fin0 == 0) & (got != pre))[0]:
        assert near[b], f"row {b}: gpu {got[b]}, oracle {pre[b]}, away from any tie"
        why = check_row_valid(inp, b, int(got[b]), gf[b])
        assert why is None, (b, why)
        pre[b] = got[b]
    exp_idx, exp_fin = pre.copy(), fin0.copy()
    exp_left = oracle.eos_epilogue(exp_idx, exp_fin, eos)
    assert np.array_equal(got, exp_idx)
    assert np.array_equal(fin.cpu().numpy(), exp_fin)
    assert int(unf.item()) == exp_left
    assert (got[fin0 == 1] == eos).all()
    assert left == exp_left or near.any()  # the oracle's own count differs only through a tie


def _bits_from_ids(inp, rng=None):
    """The workload's seen lists as a uint32 bit matrix [B, ceil(V/32)] (input side: set the
    bit of every in-range id; with rng, random bits above V in the last word as well)."""
    V = inp.V
    W = (V + 31) // 32
    bits = np.zeros((inp.B, W), np.uint32)
    for b in range(inp.B):
        ids = inp.seen_ids[inp.seen_indptr[b]:inp.seen_indptr[b + 1]]
        ids = ids[(ids >= 0) & (ids < V)].astype(np.int64)
        np.bitwise_or.at(bits[b], ids >> 5, (np.uint32(1) << (ids & 31).astype(np.uint32)))
        if rng is not None and V % 32:
            bits[b, W - 1] |= np.uint32(int(rng.integers(1, 2**32)) & ~((1 << (V % 32)) - 1) & 0xFFFFFFFF)
    return bits


def _run_bits(inp, bits, update, dev="cuda:0", **extra):
    import torch
    import decode_token_sampling_gb300 as kps
    from parity import to_dev
    if inp.dtype == "bf16":
        logits = to_dev(inp.logits.view(np.int16), dev).view(torch.bfloat16)
    else:
        logits = to_dev(inp.logits, dev)
    tb = to_dev(bits.view(np.int32), dev)
    idx, filt = kps.sample(logits, to_dev(inp.top_k, dev), to_dev(inp.top_p, dev), to_dev(inp.temperature, dev),
                           to_dev(inp.q, dev) if "seed" not in extra else None, eps=inp.eps,
                           need_logits=inp.need_logits, penalty=to_dev(inp.penalty, dev), seen_bits=tb,
                           update_seen=update, **extra)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (filt.cpu().numpy() if filt is not None else None), tb.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("name", ["batch256_penalty", "single_row_long"])
@pytest.mark.parametrize("update", [False, True])
def test_seen_bits_match_the_id_lists(name, update, kernel):
    """The seen set given as bits (with junk above V) gives the oracle's result over the id
    list; with the update the emitted token's bit, and only it, is set afterwards."""
    inp = make_workload(name)
    ref = oracle.sample(inp)
    bits0 = _bits_from_ids(inp, np.random.default_rng(9))
    gi, gf, after = _run_bits(inp, bits0.copy(), update)
    compare(inp, ref, gi, gf, f"{name} bits [{kernel}]")
    want = bits0.copy()
    if update:
        oracle.seen_append(want, gi.astype(np.int64), inp.V)
    np.testing.assert_array_equal(after, want)


@pytest.mark.parametrize("V", [7, 33, 1025, 4092, 4099, 8188, 40000, 40960])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_seen_bits_ragged_vocab(V, dtype, kernel):
    """Chunk starts that are not multiples of 32 (the cluster kernel's shifted words) and
    ragged last words (4092 and 8188: whole 16-byte groups of words, the last word part
    tokens and part padding)."""
    inp = make_random(6, V, seed=V + 1, dtype=dtype, penalty=1.3, n_seen=min(3 * V, 200))
    ref = oracle.sample(inp)
    bits0 = _bits_from_ids(inp, np.random.default_rng(V))
    gi, gf, after = _run_bits(inp, bits0.copy(), True)
    compare(inp, ref, gi, gf, f"V={V} {dtype} bits")
    want = bits0.copy()
    oracle.seen_append(want, gi.astype(np.int64), V)
    np.testing.assert_array_equal(after, want)


def test_seen_bits_across_decode_steps(kernel):
    """Four decode steps on the device: generated draws, the end-of-sequence epilogue and the
    seen bits updated in place, against the oracle's loop over growing id lists.  Rows at a
    near-tie (wide top-p rows whose boundary mass gap is below 1e-6 of S) may choose otherwise:
    there the GPU's row must be valid by the definition, and both loops carry its token on."""
    import torch
    import decode_token_sampling_gb300 as kps
    from parity import NEAR, to_dev
    dev = "cuda:0"
    inp = make_workload("batch256_penalty", rows=range(0, 256, 4))
    B, V = inp.B, inp.V
    seqs = [list(inp.seen_ids[inp.seen_indptr[b]:inp.seen_indptr[b + 1]]) for b in range(B)]
    bits = to_dev(_bits_from_ids(inp).view(np.int32), dev)
    fin = torch.zeros(B, dtype=torch.uint8, device=dev)
    fin_ref = np.zeros(B, np.uint8)
    unf = torch.zeros(1, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(31)
    seed = 99
    eos = None
    for step in range(4):
        x = (inp.logits + rng.normal(0, 0.5, inp.logits.shape)).astype(np.float32)
        indptr = np.cumsum([0] + [len(s) for s in seqs]).astype(np.int32)
        ids = np.concatenate(seqs).astype(np.int32)
        q = oracle.exp_draws(B, V, seed, step)
        ref = oracle.sample_arrays(x, "f32", inp.top_k, inp.top_p, inp.temperature, q, inp.eps, True,
                                   indptr, ids, inp.penalty)
        if eos is None:
            eos = int(ref["idx"][1])  # some row emits eos at the first step
        idx, filt = kps.sample(to_dev(x, dev), to_dev(inp.top_k, dev), to_dev(inp.top_p, dev),
                               to_dev(inp.temperature, dev), None, seed=seed, step=step, eps=inp.eps,
                               need_logits=True, penalty=to_dev(inp.penalty, dev), seen_bits=bits,
                               update_seen=True, finished=fin, eos_id=eos, unfinished=unf)
        torch.cuda.synchronize()
        got = idx.cpu().numpy()
        gf = filt.cpu().numpy()
        near = (ref["race_gap"] < NEAR) | (ref["topp_gap"] < NEAR)
        chosen = ref["idx"].copy()
        step_inp = dataclasses.replace(inp, logits=x, seen_indptr=indptr, seen_ids=ids, q=q)
        for b in np.nonzero((fin_ref == 0) & (got != chosen))[0]:
            assert near[b], (step, b, "away from any tie")
            why = check_row_valid(step_inp, b, int(got[b]), gf[b])
            assert why is None, (step, b, why)
            chosen[b] = got[b]
        left = oracle.eos_epilogue(chosen, fin_ref, eos)
        np.testing.assert_array_equal(got, chosen)
        np.testing.assert_array_equal(fin.cpu().numpy(), fin_ref)
        assert int(unf.item()) == left
        for b in range(B):
            seqs[b].append(int(chosen[b]))
    indptr, ids = oracle.seen_ids_from_bits(bits.cpu().numpy().view(np.uint32), V)
    for b in range(B):
        assert ids[indptr[b]:indptr[b + 1]].tolist() == sorted(set(int(v) for v in seqs[b] if 0 <= v < V))


def test_seen_bits_tracked_without_penalty(kernel):
    """Seen bits with no penalty array: the step samples as without a penalty and still
    appends each row's token to the bits."""
    import torch
    import decode_token_sampling_gb300 as kps
    from parity import to_dev
    inp = make_random(70, 12296, seed=12, penalty=1.5, n_seen=100)
    ref = oracle.sample_arrays(inp.logits, "f32", inp.top_k, inp.top_p, inp.temperature, inp.q, inp.eps, True)
    bits0 = _bits_from_ids(inp)
    tb = to_dev(bits0.view(np.int32), "cuda:0")
    idx, filt = kps.sample(to_dev(inp.logits, "cuda:0"), to_dev(inp.top_k, "cuda:0"), to_dev(inp.top_p, "cuda:0"),
                           to_dev(inp.temperature, "cuda:0"), to_dev(inp.q, "cuda:0"), eps=inp.eps, need_logits=True,
                           seen_bits=tb, update_seen=True)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    compare(inp, ref, gi, filt.cpu().numpy(), "bits without penalty")
    want = bits0.copy()
    oracle.seen_append(want, gi.astype(np.int64), inp.V)
    np.testing.assert_array_equal(tb.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_largest_vocabulary_and_one_past_it(dtype):
    """At the largest vocabulary the library takes (one row spread over the widest cluster)
    the rows match the oracle; a vocabulary past it is refused on the host, before any launch."""
    import torch
    import decode_token_sampling_gb300 as kps
    code = 1 if dtype == "bf16" else 0
    vmax = int(kps.load_library().kps_max_vocab(code))
    assert vmax >= 262144
    inp = make_random(2, vmax, seed=77, dtype=dtype, penalty=1.2, n_seen=300)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    compare(inp, ref, gi, gf, f"V={vmax} {dtype}")
    big = make_random(2, vmax + 8, seed=78, dtype=dtype)
    with pytest.raises(kps.KpsError) as e:
        run_gpu(big)
    assert e.value.code == 2  # KPS_ERR_UNSUPPORTED


def test_row_kernel_at_its_largest_vocabulary():
    """V = 262144 fp32 over 64 rows: the row kernel's largest row (its seen bitmap fills the
    shared-memory slot it has)."""
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_random(64, 262144, seed=79, penalty=1.2, n_seen=300, need_logits=True)
        ref = oracle.sample(inp)
        gi, gf = run_gpu(inp)
        assert kps.last_kernel() == "kps_row_kernel"
        compare(inp, ref, gi, gf, "row kernel V=262144")
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


def test_more_work_units_than_the_item_list_holds():
    """80000 rows of 16 tokens: more units per cluster than the row kernel's item list holds,
    so every CTA takes rows on its own, round-robin."""
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        inp = make_random(80000, 16, seed=80, penalty=1.2, n_seen=8, need_logits=True)
        ref = oracle.sample(inp)
        gi, gf = run_gpu(inp)
        assert kps.last_kernel() == "kps_row_kernel"
        compare(inp, ref, gi, gf, "B=80000 V=16")
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)


def test_cluster_size_follows_the_batch():
    """The launch shapes are cached per (device, dtype, V) only; the cluster kernel's width
    still follows each call's batch size.  Calls at B=40, then B=1, then B=40 again launch the
    cluster size kps_query_launch reports for their own B, and match the oracle: on a
    262144-token bf16 vocabulary (the widest clusters) and on a 65536-token one, where the
    single row gets a wider cluster than a batch of 40."""
    import torch
    import decode_token_sampling_gb300 as kps
    kps.set_kernel_policy(kps.KERNEL_AUTO)
    for V in (262144, 65536):
        for B in (40, 1, 40):
            inp = make_random(B, V, seed=90 + B, dtype="bf16", k_range=(1, 200), p_range=(0.5, 0.95))
            ref = oracle.sample(inp)
            gi, gf = run_gpu(inp)
            compare(inp, ref, gi, gf, f"B={B} V={V}")
            assert kps.last_kernel() == "kps_sample_kernel"
            want = kps.query_launch(B, V, torch.bfloat16)["cluster_size"]
            assert kps.last_cluster_size() == want, (V, B, kps.last_cluster_size(), want)
    assert kps.query_launch(1, 65536, torch.bfloat16)["cluster_size"] > kps.query_launch(40, 65536, torch.bfloat16)["cluster_size"]

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["plain", "ties", "big_k", "no_logits"])
def test_shared_topk_rows(dtype, case):
    """Batches with at most one row per cluster of the row kernel: both CTAs of a cluster
    stream one top-k row against the same sampled threshold and rank 0 merges their
    candidate segments (a merge that would overflow a segment sends the row to the exact
    whole-row select: the tied case).  Against the oracle, with filtered logits."""
    import decode_token_sampling_gb300 as kps
    kw = dict(plain=dict(k_range=(1, 1024)), ties=dict(ties=True, k_range=(500, 1024)),
              big_k=dict(k_range=(1000, 1024), p_range=(0.9, 1.0)), no_logits=dict(need_logits=False))[case]
    inp = make_random(100, 50000, seed=61 + len(case), dtype=dtype, penalty=1.2, n_seen=300, **kw)
    ref = oracle.sample(inp)
    kps.set_kernel_policy(kps.KERNEL_ROW)
    try:
        gi, gf = run_gpu(inp)
        assert kps.last_kernel() == "kps_row_kernel"
        assert kps.last_cluster_size() == 2
    finally:
        kps.set_kernel_policy(kps.KERNEL_AUTO)
    compare(inp, ref, gi, gf, f"shared top-k rows {case} {dtype}")


def _spiky_rows(dtype, seed):
    """Rows of m spikes over a background far below them, with k and m set so that the
    number of top-k candidates a cluster collects lands on both sides of 256 (the
    gathered-candidate paths of the cluster kernel and the histogram searches), tied spike
    values, and top-p cuts that fall inside the spikes.  Half of each row's seen ids are
    spike positions, so the penalty reorders them."""
    from decode_token_sampling_gb300.workloads import f32_to_bf16_bits
    rows = [  # (m spikes, k, p, tied values)
        (10, 1, 0.9, None), (200, 50, 0.9, None), (256, 200, 0.5, None), (257, 256, 0.95, None),
        (300, 100, 0.7, (6.0, 6.5, 7.0)), (600, 255, 0.3, None), (600, 300, 0.99, None), (40, 20, 0.6, (7.0,)),
    ]
    B, V = len(rows), 65536
    inp = make_random(B, V, seed=seed, dtype="f32", penalty=1.3, n_seen=64)
    rng = np.random.Generator(np.random.PCG64([0x5EED0100, seed, 7]))
    x = rng.normal(-20.0, 0.5, (B, V)).astype(np.float32)
    for b, (m, k, p, tied) in enumerate(rows):
        pos = rng.choice(V, m, replace=False)
        x[b, pos] = rng.choice(np.array(tied, np.float32), m) if tied else rng.normal(5.0, 1.0, m).astype(np.float32)
        h = min(32, m // 2)
        inp.seen_ids[b * 64:b * 64 + h] = pos[:h]
        inp.top_k[b], inp.top_p[b], inp.temperature[b] = k, p, 0.8
    inp.logits = f32_to_bf16_bits(x) if dtype == "bf16" else x
    inp.dtype = dtype
    inp.name = f"spiky_B{B}_V{V}"
    return inp


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spiky_rows_around_the_candidate_gather(dtype, kernel):
    """Top-k rows whose candidates number from a handful to several hundred: with at most
    256 in the cluster, rank 0 gathers them and ranks them pairwise for the k-th and the
    top-p cut; above that, the histogram searches run (and rank 0 still cuts top-p over
    the gathered survivors when k <= 256).  Against the oracle, with filtered logits."""
    import decode_token_sampling_gb300 as kps
    inp = _spiky_rows(dtype, seed=171)
    ref = oracle.sample(inp)
    gi, gf = run_gpu(inp)
    if kernel == "cluster":
        assert kps.last_kernel() == "kps_sample_kernel"
    compare(inp, ref, gi, gf, f"spiky rows {dtype}")
