"""CPU oracle for the decode-step sampling post-process — TEST INFRASTRUCTURE ONLY.

The oracle is a plain single-threaded C++ implementation (kps_oracle.cpp)
written from the method's definition.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  It shares no code with the CUDA library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kps_oracle.cpp")
_LIB = os.path.join(_HERE, "libkps_oracle.so")
_lib: Optional[ctypes.CDLL] = None

# -ffp-contract=off: every fp32 step is a single IEEE operation (no fused
# multiply-add contraction), matching the definition.
CXXFLAGS = ["-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library in-tree (seconds); returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CXXFLAGS, "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.kpso_sample.restype = ctypes.c_int
        lib.kpso_sample.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P, P,
                                    P, ctypes.c_float, ctypes.c_int, P, P, P, P, P]
        lib.kpso_eos_epilogue.restype = ctypes.c_int64
        lib.kpso_eos_epilogue.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64]
        lib.kpso_exp_draws.restype = ctypes.c_int
        lib.kpso_exp_draws.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, P]
        lib.kpso_philox4x32_10.restype = None
        lib.kpso_philox4x32_10.argtypes = [P, ctypes.c_uint32, ctypes.c_uint32]
        lib.kpso_seen_ids_from_bits.restype = ctypes.c_int64
        lib.kpso_seen_ids_from_bits.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P]
        lib.kpso_row_terms.restype = ctypes.c_int64
        lib.kpso_row_terms.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P, P, P,
                                       P, P, P, P, P, P]
        lib.kpso_seen_append.restype = None
        lib.kpso_seen_append.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def sample_arrays(logits: np.ndarray, dtype: str, top_k, top_p, temperature, q, eps: float = 1e-20,
                  need_logits: bool = True, seen_indptr=None, seen_ids=None, penalty=None) -> dict:
    """Run the oracle on host arrays.  logits: float32 [B,V] or uint16 bf16 bits [B,V]."""
    lib = _load()
    if dtype == "f32":
        logits = np.ascontiguousarray(logits, dtype=np.float32)
    elif dtype == "bf16":
        logits = np.ascontiguousarray(logits, dtype=np.uint16)
    else:
        raise ValueError(dtype)
    B, V = logits.shape
    top_k = np.ascontiguousarray(top_k, dtype=np.int32)
    top_p = np.ascontiguousarray(top_p, dtype=np.float32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    if q is not None:  # None: sampling off (greedy)
        q = np.ascontiguousarray(q, dtype=np.float32)
        assert q.shape == (B, V)
    assert top_k.shape == (B,) and top_p.shape == (B,) and temperature.shape == (B,)
    if seen_indptr is not None:
        seen_indptr = np.ascontiguousarray(seen_indptr, dtype=np.int32)
        seen_ids = np.ascontiguousarray(seen_ids, dtype=np.int32)
        penalty = np.ascontiguousarray(penalty, dtype=np.float32)
    out_idx = np.empty(B, dtype=np.int64)
    out = np.empty((B, V), dtype=np.float32) if need_logits else None
    kept = np.empty(B, dtype=np.int64)
    race_gap = np.empty(B, dtype=np.float64)
    topp_gap = np.empty(B, dtype=np.float64)
    rc = lib.kpso_sample(_ptr(logits), 0 if dtype == "f32" else 1, B, V, _ptr(top_k), _ptr(top_p),
                         _ptr(temperature), _ptr(seen_indptr), _ptr(seen_ids), _ptr(penalty), _ptr(q),
                         float(eps), 1 if need_logits else 0, _ptr(out_idx), _ptr(out), _ptr(kept),
                         _ptr(race_gap), _ptr(topp_gap))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return dict(idx=out_idx, filtered=out, kept=kept, race_gap=race_gap, topp_gap=topp_gap)


def sample(inp, need_logits: Optional[bool] = None) -> dict:
    """Run the oracle on a workloads.SamplingInputs."""
    nl = inp.need_logits if need_logits is None else need_logits
    return sample_arrays(inp.logits, inp.dtype, inp.top_k, inp.top_p, inp.temperature, inp.q, inp.eps,
                         nl, inp.seen_indptr, inp.seen_ids, inp.penalty)


def row_terms(inp, b: int) -> dict:
    """The terms of row b of a workloads.SamplingInputs before top-p: the transformed row x
    (float32 [V]: NaN -> -inf, penalty, temperature), the first nK elements of the order pi
    (int64), their softmax weights e (float64, e = exp(x - max)), their sum S, and whether
    the row is greedy.  For checking a result at a near-tie against the definition."""
    lib = _load()
    logits = np.ascontiguousarray(inp.logits, dtype=np.float32 if inp.dtype == "f32" else np.uint16)
    B, V = logits.shape
    top_k = np.ascontiguousarray(inp.top_k, dtype=np.int32)
    temperature = np.ascontiguousarray(inp.temperature, dtype=np.float32)
    indptr = ids = pen = None
    if inp.seen_indptr is not None:
        indptr = np.ascontiguousarray(inp.seen_indptr, dtype=np.int32)
        ids = np.ascontiguousarray(inp.seen_ids, dtype=np.int32)
        pen = np.ascontiguousarray(inp.penalty, dtype=np.float32)
    x = np.empty(V, np.float32)
    order = np.empty(V, np.int64)
    e = np.empty(V, np.float64)
    S = np.zeros(1, np.float64)
    greedy = np.zeros(1, np.int32)
    nK = lib.kpso_row_terms(_ptr(logits), 0 if inp.dtype == "f32" else 1, B, V, int(b), _ptr(top_k),
                            _ptr(temperature), _ptr(indptr), _ptr(ids), _ptr(pen), _ptr(x), _ptr(order), _ptr(e),
                            _ptr(S), _ptr(greedy))
    if nK < 1:
        raise ValueError(f"oracle rejected its arguments (code {nK})")
    return dict(x=x, order=order[:nK].copy(), e=e[:nK].copy(), S=float(S[0]), nK=int(nK), greedy=bool(greedy[0]))


def exp_draws(B: int, V: int, seed: int, step: int = 0) -> np.ndarray:
    """The generated Exp(1) draws q[B, V] of a seeded call (Philox4x32-10, see kps_oracle.cpp)."""
    q = np.empty((B, V), dtype=np.float32)
    if _load().kpso_exp_draws(B, V, seed & (2**64 - 1), step & (2**64 - 1), _ptr(q)) != 0:
        raise ValueError("bad sizes")
    return q


def philox4x32_10(counter, key) -> list:
    """One Philox4x32-10 block: four 32-bit counter words and two key words in, four words out."""
    c = np.array(counter, dtype=np.uint32)
    _load().kpso_philox4x32_10(c.ctypes.data_as(ctypes.c_void_p), int(key[0]), int(key[1]))
    return [int(x) for x in c]


def eos_epilogue(idx: np.ndarray, finished: np.ndarray, eos: int) -> int:
    """The end-of-sequence epilogue on host arrays (int64 idx, uint8 finished, both updated
    in place); returns the rows left unfinished."""
    assert idx.dtype == np.int64 and finished.dtype == np.uint8 and idx.shape == finished.shape
    return int(_load().kpso_eos_epilogue(_ptr(idx), _ptr(finished), int(eos), idx.size))


def seen_ids_from_bits(bits: np.ndarray, V: int):
    """The seen sets of a uint32 bit matrix [B, ceil(V/32)] as CSR (indptr int32 [B+1],
    ids int32 [nnz], each row's ids distinct and ascending)."""
    bits = np.ascontiguousarray(bits).view(np.uint32)
    B = bits.shape[0]
    assert bits.shape == (B, (V + 31) // 32)
    indptr = np.zeros(B + 1, np.int32)
    lib = _load()
    n = int(lib.kpso_seen_ids_from_bits(_ptr(bits), B, V, _ptr(indptr), None))
    ids = np.zeros(max(n, 1), np.int32)
    lib.kpso_seen_ids_from_bits(_ptr(bits), B, V, _ptr(indptr), _ptr(ids))
    return indptr, ids[:n]


def seen_append(bits: np.ndarray, idx: np.ndarray, V: int) -> None:
    """Sets the bit of each row's token idx[b] (int64, ignored outside [0, V)) in place."""
    assert bits.dtype in (np.uint32, np.int32) and bits.flags.c_contiguous and idx.dtype == np.int64
    assert bits.shape == (idx.size, (V + 31) // 32)
    _load().kpso_seen_append(_ptr(bits), _ptr(idx), idx.size, V)

