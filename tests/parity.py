"""Helpers for GPU-vs-oracle parity tests (the oracle decides what is right).

Agreement rule: chosen indices and the kept set (positions of non -inf
filtered logits) must be identical, and kept values equal within 1e-6
relative, except in rows where the oracle reports a near-tie: the two best
race scores, or the top-p boundary cumsum and p*S, within 1e-6 relative.
Those rows are checked for validity against the definition instead
(check_row_valid): the GPU's kept set is a prefix of the order pi whose mass
meets the top-p rule within 1e-6, and its chosen token wins the race over
that kept set within 1e-6.  Every compare() call records how many rows it
found near a tie and how many of them it accepted on validity; the test
session prints the counts per test at its end.
"""

from __future__ import annotations

import numpy as np

NEAR = 1e-6

# (test, label, rows compared, near-tie rows, near-tie rows accepted on validity) per compare()
NEAR_LOG: list = []


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_gpu(inp, dev="cuda:0", need_logits=None, workspace=None, stream=None, seed=None, step=0):
    import torch
    import decode_token_sampling_gb300 as kps

    nl = inp.need_logits if need_logits is None else need_logits
    if inp.dtype == "bf16":
        logits = to_dev(inp.logits.view(np.int16), dev).view(torch.bfloat16)
    else:
        logits = to_dev(inp.logits, dev)
    kw = {}
    if inp.seen_indptr is not None:
        kw = dict(seen_indptr=to_dev(inp.seen_indptr, dev), seen_ids=to_dev(inp.seen_ids, dev),
                  penalty=to_dev(inp.penalty, dev))
    idx, filt = kps.sample(logits, to_dev(inp.top_k, dev), to_dev(inp.top_p, dev), to_dev(inp.temperature, dev),
                           to_dev(inp.q, dev) if (inp.q is not None and seed is None) else None, eps=inp.eps,
                           seed=seed, step=step, need_logits=nl, workspace=workspace, stream=stream,
                           **kw)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (filt.cpu().numpy() if filt is not None else None)


def check_row_valid(inp, b: int, got_idx: int, got_row, terms=None):
    """Checks one GPU result row against the method's definition where the oracle reports a
    near-tie, so that the oracle's own choice need not be matched.  Returns None if valid,
    else what is wrong.  got_row is the GPU's filtered row (float32 [V]; its kept set is
    where it is not -inf).  With x the transformed row, pi the order and e the weights of the
    oracle's row terms, p = top_p[b] and S the top-k mass:
      * the kept set is the first n elements of pi, 1 <= n <= nK (greedy or p <= 0: n = 1;
        p >= 1 or NaN: every element of the top-k set);
      * top-p: with c_i the mass of the first i elements and t = p * S, c_n >= t - 1e-6 S and
        c_(n-1) <= t + 1e-6 S, and every element where the GPU and the oracle's rule disagree
        has its exclusive mass c_i within 1e-6 t of t;
      * kept values equal x within 1e-6 relative;
      * the chosen token is kept; with draws q its race score e_v / (q_v + eps) is within
        1e-6 relative of the best score over the kept set; without draws it is pi's first.
    Elements whose transformed value is -inf are invisible in the filtered row; they sit at
    the end of pi with zero weight (or the row is all -inf), so n counts the visible ones."""
    t = terms if terms is not None else __import__("oracle").row_terms(inp, b)
    x, order, e, S, nK = t["x"], t["order"], t["e"], t["S"], t["nK"]
    V = inp.V
    if not (0 <= got_idx < V):
        return "index out of range"
    kept = got_row != -np.inf
    n = int(kept.sum())
    finite = order[x[order] != -np.inf]  # visible part of the top-k set, in pi order
    if finite.size == 0:  # every value -inf: nothing visible; the race runs over pi's elements
        if n:
            return "kept values in an all -inf row"
        keep_ids = order
    else:
        if not (1 <= n <= finite.size):
            return f"kept count {n} outside [1, {finite.size}]"
        if not np.array_equal(np.sort(np.nonzero(kept)[0]), np.sort(finite[:n])):
            return "kept set is not a prefix of the order"
        p = float(inp.top_p[b])
        if t["greedy"] or p <= 0.0:
            if n != 1:
                return f"greedy / p <= 0 row keeps {n}"
        elif not (p < 1.0):  # p >= 1 or NaN: top-p off
            if n != finite.size:
                return f"top-p off but {n} of {finite.size} kept"
        else:
            c = np.concatenate([[0.0], np.cumsum(e)])  # c[i]: mass of the first i elements
            target = p * S
            if c[n] < target - NEAR * S:
                return f"kept mass {c[n]!r} short of p*S {target!r}"
            if c[n - 1] > target + NEAR * S:
                return f"mass before the last kept {c[n - 1]!r} above p*S {target!r}"
            n_or = int(np.searchsorted(c[1:], target, side="left")) + 1  # the rule's count
            n_or = min(n_or, nK)
            for i in range(min(n, n_or), max(n, n_or)):
                if i < finite.size and abs(c[i] - target) > NEAR * target:
                    return f"element {int(order[i])} at position {i} decided away from the boundary"
        gv, xv = got_row[kept], x[kept]
        if not np.all((gv == xv) | (np.abs(gv - xv) <= NEAR * np.abs(xv))):
            return "kept values differ from the transformed row"
        keep_ids = finite[:n]
        if not kept[got_idx]:
            return "chosen token not kept"
    if inp.q is None:
        return None if got_idx == int(order[0]) else f"sampling off: chose {got_idx}, pi's first is {int(order[0])}"
    ew = np.zeros(V, np.float64)
    ew[order] = e
    with np.errstate(divide="ignore", invalid="ignore"):
        r = ew[keep_ids] / (inp.q[b, keep_ids].astype(np.float64) + float(inp.eps))
    ok = ~np.isnan(r)
    if not ok.any():
        return None if got_idx == int(order[0]) else "all race scores NaN but not pi's first chosen"
    best = r[ok].max()
    pos = np.nonzero(keep_ids == got_idx)[0]
    if pos.size == 0:
        return "chosen token outside the kept set"
    rg = r[pos[0]]
    if np.isnan(rg):
        return "chosen token has a NaN race score"
    if not (rg == best or rg >= best * (1.0 - NEAR)):
        return f"chosen token's race score {rg!r} below the best {best!r}"
    return None


def compare(inp, ref, got_idx, got_filt, label="", rerun=None):
    """Asserts parity; returns the list of near-tie rows that were accepted on validity.
    rerun: a callable that repeats the GPU call with need_logits=True and returns (idx,
    filtered); used when got_filt is None and a near-tie row differs (default: run_gpu)."""
    import os
    near = (ref["race_gap"] < NEAR) | (ref["topp_gap"] < NEAR)
    accepted = []
    bad = []
    pending = []
    for b in range(inp.B):
        idx_ok = got_idx[b] == ref["idx"][b]
        f_ok = True
        if got_filt is not None:
            g, r = got_filt[b], ref["filtered"][b]
            gk, rk = g != -np.inf, r != -np.inf
            if not np.array_equal(gk, rk):
                f_ok = False
            else:
                gv, rv = g[gk], r[rk]
                f_ok = bool(np.all((gv == rv) | (np.abs(gv - rv) <= NEAR * np.abs(rv))))
        if idx_ok and f_ok:
            continue
        if near[b]:
            pending.append(b)
            continue
        bad.append((b, f"idx gpu={got_idx[b]} oracle={ref['idx'][b]} filtered_ok={f_ok} kept={ref['kept'][b]}"))
    if pending:
        filt = got_filt
        if filt is None:
            ri, filt = (rerun or (lambda: run_gpu(inp, need_logits=True)))()
            for b in pending:
                if ri[b] != got_idx[b]:
                    bad.append((b, f"choice changed with need_logits: {got_idx[b]} then {ri[b]}"))
        for b in pending:
            why = check_row_valid(inp, b, int(got_idx[b]), filt[b])
            if why is None:
                accepted.append(b)
            else:
                bad.append((b, f"near-tie row invalid: {why}"))
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    NEAR_LOG.append((test, label, int(inp.B), int(near.sum()), len(accepted)))
    assert not bad, f"[{label}] parity failures (row, what): {bad[:10]} (of {len(bad)})"
    return accepted
