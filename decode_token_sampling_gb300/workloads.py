"""Seeded synthetic inputs for the sampling step.

This module only draws random numbers and lays them out; it holds none of the
sampling arithmetic, so the CPU oracle and the CUDA path can both consume its
output without sharing any of the method's code.

Five workloads, named by what they are:

  small_mixed      B=4,   V=32000,  fp32, N(0,2) logits + 5 spikes of +8 per row,
                   top_k [50, 1, 1024, 0], top_p [0.85, 1.0, 0.9, 0.5], T=0.85,
                   no penalty, filtered logits requested.
  bf16_zipf        B=64,  V=128256, bf16, N(0,3) + Zipf rank bonus,
                   top_k ~ U[1,1024], top_p ~ U[0.7,0.99], T=0.7, no penalty.
  batch256_penalty B=256, V=151936, fp32, N(0,2.5) + Zipf rank bonus,
                   top_k ~ U[1,1024] with 10% out of range (0, -1, 1025, V+7),
                   top_p ~ U[0.5,1.0], T ~ U[0.5,1.2], penalty 1.1 over 512
                   seen ids per row, filtered logits requested.
  flat_nucleus     B=128, V=151936, fp32, flat N(0,0.5), top_k = 0 (skip),
                   top_p ~ U[0.95,0.999], T=1.0, no penalty.
  single_row_long  B=1,   V=262144, bf16, N(0,2) + Zipf rank bonus, top_k=50,
                   top_p=0.85, T=0.85, penalty 1.05 over 2048 seen ids.

All draw q ~ Exp(1) (fp32) and eps = 1e-20.

Zipf rank bonus: a seeded per-row permutation pi_b of the vocabulary; the
token at rank r (1-based) gets +10 / sqrt(r).  Seen ids: half uniform over
the vocabulary, half drawn from the 2048 best-ranked tokens of pi_b (so the
penalty changes which tokens survive), duplicates allowed.

Every row is generated from its own stream seeded by (workload seed, row), so
any subset of rows can be regenerated without the rest.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

WORKLOADS = ("small_mixed", "bf16_zipf", "batch256_penalty", "flat_nucleus", "single_row_long")

_SEED_BASE = 0x5EED0000


@dataclasses.dataclass
class SamplingInputs:
    """Host-side inputs of one sampling step (numpy arrays, row-major)."""

    name: str
    dtype: str  # "f32" or "bf16"
    B: int
    V: int
    logits: np.ndarray  # float32 [B,V] or uint16 [B,V] (bf16 bit patterns)
    top_k: np.ndarray  # int32 [B]
    top_p: np.ndarray  # float32 [B]
    temperature: np.ndarray  # float32 [B]
    q: np.ndarray  # float32 [B,V]
    eps: float
    need_logits: bool
    seen_indptr: Optional[np.ndarray] = None  # int32 [B+1]
    seen_ids: Optional[np.ndarray] = None  # int32 [nnz]
    penalty: Optional[np.ndarray] = None  # float32 [B]

    @property
    def has_penalty(self) -> bool:
        return self.seen_indptr is not None

    def metric_bytes(self) -> int:
        """Bytes counted by the throughput metric: logits + q (+ filtered output)."""
        esize = 4 if self.dtype == "f32" else 2
        n = self.B * self.V
        return n * esize + n * 4 + (n * 4 if self.need_logits else 0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def _row_rng(wid: int, row: int, seed_offset: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([_SEED_BASE + wid + seed_offset, row]))


def _zipf_bonus(rng: np.random.Generator, V: int) -> tuple[np.ndarray, np.ndarray]:
    perm = rng.permutation(V)
    bonus = np.empty(V, dtype=np.float64)
    bonus[perm] = 10.0 / np.sqrt(np.arange(1, V + 1, dtype=np.float64))
    return bonus, perm


def _seen(rng: np.random.Generator, V: int, perm: np.ndarray, n: int) -> np.ndarray:
    half = n // 2
    uni = rng.integers(0, V, size=n - half)
    top = perm[rng.integers(0, min(2048, V), size=half)]
    ids = np.concatenate([uni, top]).astype(np.int32)
    rng.shuffle(ids)
    return ids


def make_workload(name: str, rows: Optional[Sequence[int]] = None, seed_offset: int = 0) -> SamplingInputs:
    """Build the named workload; `rows` selects a subset of its rows (in order)."""
    wid = WORKLOADS.index(name) + 1
    spec = {
        "small_mixed": dict(B=4, V=32000, dtype="f32", need_logits=True),
        "bf16_zipf": dict(B=64, V=128256, dtype="bf16", need_logits=False),
        "batch256_penalty": dict(B=256, V=151936, dtype="f32", need_logits=True),
        "flat_nucleus": dict(B=128, V=151936, dtype="f32", need_logits=False),
        "single_row_long": dict(B=1, V=262144, dtype="bf16", need_logits=False),
    }[name]
    B_full, V = spec["B"], spec["V"]
    rows = list(range(B_full)) if rows is None else [int(r) for r in rows]
    B = len(rows)
    logits32 = np.empty((B, V), dtype=np.float32)
    q = np.empty((B, V), dtype=np.float32)
    top_k = np.empty(B, dtype=np.int32)
    top_p = np.empty(B, dtype=np.float32)
    temp = np.empty(B, dtype=np.float32)
    pen = np.empty(B, dtype=np.float32)
    seen_rows: list[np.ndarray] = []
    for i, r in enumerate(rows):
        rng = _row_rng(wid, r, seed_offset)
        if name == "small_mixed":
            x = rng.normal(0.0, 2.0, V)
            x[rng.choice(V, 5, replace=False)] += 8.0
            top_k[i] = (50, 1, 1024, 0)[r % 4]
            top_p[i] = (0.85, 1.0, 0.9, 0.5)[r % 4]
            temp[i] = 0.85
        elif name == "bf16_zipf":
            bonus, _ = _zipf_bonus(rng, V)
            x = rng.normal(0.0, 3.0, V) + bonus
            top_k[i] = rng.integers(1, 1025)
            top_p[i] = rng.uniform(0.7, 0.99)
            temp[i] = 0.7
        elif name == "batch256_penalty":
            bonus, perm = _zipf_bonus(rng, V)
            x = rng.normal(0.0, 2.5, V) + bonus
            if rng.random() < 0.10:
                top_k[i] = (0, -1, 1025, V + 7)[rng.integers(0, 4)]
            else:
                top_k[i] = rng.integers(1, 1025)
            top_p[i] = rng.uniform(0.5, 1.0)
            temp[i] = rng.uniform(0.5, 1.2)
            pen[i] = 1.1
            seen_rows.append(_seen(rng, V, perm, 512))
        elif name == "flat_nucleus":
            x = rng.normal(0.0, 0.5, V)
            top_k[i] = 0
            top_p[i] = rng.uniform(0.95, 0.999)
            temp[i] = 1.0
        elif name == "single_row_long":
            bonus, perm = _zipf_bonus(rng, V)
            x = rng.normal(0.0, 2.0, V) + bonus
            top_k[i] = 50
            top_p[i] = 0.85
            temp[i] = 0.85
            pen[i] = 1.05
            seen_rows.append(_seen(rng, V, perm, 2048))
        else:  # pragma: no cover
            raise ValueError(name)
        logits32[i] = x.astype(np.float32)
        q[i] = rng.exponential(1.0, V).astype(np.float32)
    if spec["dtype"] == "bf16":
        logits = f32_to_bf16_bits(logits32)
    else:
        logits = logits32
    inp = SamplingInputs(name=name, dtype=spec["dtype"], B=B, V=V, logits=logits, top_k=top_k,
                         top_p=top_p, temperature=temp, q=q, eps=1e-20,
                         need_logits=spec["need_logits"])
    if seen_rows:
        indptr = np.zeros(B + 1, dtype=np.int32)
        indptr[1:] = np.cumsum([len(s) for s in seen_rows])
        inp.seen_indptr = indptr
        inp.seen_ids = np.concatenate(seen_rows).astype(np.int32)
        inp.penalty = pen
    return inp


def make_random(B: int, V: int, *, seed: int, dtype: str = "f32", scale: float = 2.0,
                k_range=(1, 1024), p_range=(0.5, 1.0), t_range=(0.5, 1.2),
                penalty: Optional[float] = None, n_seen: int = 0, need_logits: bool = True,
                k_skip_frac: float = 0.1, ties: bool = False,
                special: bool = False) -> SamplingInputs:
    """Generic seeded inputs for parity tests of arbitrary (including ragged) shapes.

    ties: quantise logits to a coarse grid so that many values are equal.
    special: sprinkle NaN, -inf and +inf logits and edge-case per-row parameters.
    """
    rng = np.random.Generator(np.random.PCG64([_SEED_BASE + 0x100, seed]))
    x = rng.normal(0.0, scale, (B, V))
    if ties:
        x = np.round(x * 2.0) / 2.0
    x = x.astype(np.float32)
    if special and V >= 4:
        m = rng.random((B, V))
        x[m < 0.01] = np.nan
        x[(m >= 0.01) & (m < 0.03)] = -np.inf
    top_k = rng.integers(k_range[0], k_range[1] + 1, B).astype(np.int32)
    skip = rng.random(B) < k_skip_frac
    top_k[skip] = rng.choice(np.array([0, -1, 1025, V + 7], dtype=np.int64), skip.sum()).astype(np.int32)
    top_p = rng.uniform(p_range[0], p_range[1], B).astype(np.float32)
    temp = rng.uniform(t_range[0], t_range[1], B).astype(np.float32)
    q = rng.exponential(1.0, (B, V)).astype(np.float32)
    inp = SamplingInputs(name=f"random_B{B}_V{V}", dtype=dtype, B=B, V=V,
                         logits=f32_to_bf16_bits(x) if dtype == "bf16" else x,
                         top_k=top_k, top_p=top_p, temperature=temp, q=q, eps=1e-20,
                         need_logits=need_logits)
    if penalty is not None and n_seen > 0:
        ids = rng.integers(-3, V + 3, (B, n_seen)).astype(np.int32)  # includes out-of-range ids
        inp.seen_indptr = (np.arange(B + 1, dtype=np.int64) * n_seen).astype(np.int32)
        inp.seen_ids = ids.reshape(-1)
        inp.penalty = np.full(B, penalty, dtype=np.float32)
    return inp
