"""Helpers for GPU-vs-oracle parity tests (the oracle decides what is right).

Agreement rule: chosen indices and the kept set (positions of non -inf
filtered logits) must be identical, and kept values equal within 1e-6
relative, except in rows where the oracle reports a near-tie: the two best
race scores, or the top-p boundary cumsum and p*S, within 1e-6 relative.
Those rows are logged and checked for validity only (the GPU's choice lies
in its own kept set, and its kept set differs from the oracle's only at the
boundary of the order).
"""

from __future__ import annotations

import numpy as np

NEAR = 1e-6


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


def compare(inp, ref, got_idx, got_filt, label=""):
    """Asserts parity; returns the list of near-tie rows that were accepted."""
    near = (ref["race_gap"] < NEAR) | (ref["topp_gap"] < NEAR)
    accepted = []
    bad = []
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
            if not (0 <= got_idx[b] < inp.V):
                bad.append((b, "index out of range"))
            elif got_filt is not None and got_filt[b][got_idx[b]] == -np.inf and ref["filtered"][b][got_idx[b]] != -np.inf:
                bad.append((b, "chosen token not kept"))
            else:
                accepted.append(b)
            continue
        bad.append((b, f"idx gpu={got_idx[b]} oracle={ref['idx'][b]} filtered_ok={f_ok} kept={ref['kept'][b]}"))
    if accepted:
        print(f"[{label}] near-tie rows accepted: {accepted}")
    assert not bad, f"[{label}] parity failures (row, what): {bad[:10]} (of {len(bad)})"
    return accepted
