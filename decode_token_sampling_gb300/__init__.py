"""GB300-native decode-step token sampling (penalty -> temperature -> top-k -> top-p
-> exponential race) over a [batch, vocab] logits matrix.

The work runs in hand-written sm_103a CUDA kernels behind the C ABI declared in
include/kps.h (libkps.so, built in-tree).  This module only marshals torch
tensors into that ABI; there is no fallback of any kind: if the library is
missing or the tensors are not on a CUDA device, calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkps.so")

KPS_F32, KPS_BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size", 3: "workspace missing, misaligned or too small",
          4: "CUDA error", 5: "device wait timed out"}


class KpsError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, 'unknown status')} (code {code})")
        self.code = code


_lib: Optional[ctypes.CDLL] = None


class StepOpts(ctypes.Structure):
    """kps_step_opts (include/kps.h)."""
    _fields_ = [("q", ctypes.c_void_p), ("generate", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("step", ctypes.c_uint64), ("finished", ctypes.c_void_p), ("eos_id", ctypes.c_int64),
                ("unfinished", ctypes.c_void_p), ("seen_bits", ctypes.c_void_p), ("update_seen", ctypes.c_int),
                ("kernel_policy", ctypes.c_int)]


def load_library() -> ctypes.CDLL:
    """Load libkps.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -m decode_token_sampling_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.kps_workspace_size.restype = ctypes.c_size_t
    lib.kps_workspace_size.argtypes = [I64, I64, I32]
    lib.kps_max_vocab.restype = I64
    lib.kps_max_vocab.argtypes = [I32]
    lib.kps_sample.restype = I32
    lib.kps_sample.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, P, F32, I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_last_device_status.restype = I32
    lib.kps_last_device_status.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.kps_status_string.restype = ctypes.c_char_p
    lib.kps_status_string.argtypes = [I32]
    lib.kps_sample_seeded.restype = I32
    lib.kps_sample_seeded.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_float, I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_sample_step.restype = I32
    lib.kps_sample_step.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, ctypes.POINTER(StepOpts), ctypes.c_float,
                                    I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_last_kernel.restype = I32
    lib.kps_last_kernel.argtypes = []
    lib.kps_last_launch_count.restype = I32
    lib.kps_last_launch_count.argtypes = []
    lib.kps_last_cluster_size.restype = I32
    lib.kps_last_cluster_size.argtypes = []
    lib.kps_query_launch.restype = I32
    lib.kps_query_launch.argtypes = [I64, I64, I32, ctypes.POINTER(I32), ctypes.POINTER(I64),
                                     ctypes.POINTER(ctypes.c_size_t)]
    _lib = lib
    return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KPS_F32
    if t.dtype == torch.bfloat16:
        return KPS_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, shape: Tuple[int, ...], device) -> None:
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, logits on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(B: int, V: int, dtype: torch.dtype = torch.float32) -> int:
    code = KPS_BF16 if dtype == torch.bfloat16 else KPS_F32
    return int(load_library().kps_workspace_size(B, V, code))


def new_workspace(B: int, V: int, dtype: torch.dtype = torch.float32, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer (uint8) of the size kps_sample needs."""
    n = max(workspace_size(B, V, dtype), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


KERNEL_AUTO, KERNEL_CLUSTER, KERNEL_ROW, KERNEL_ROW_EXACT = 0, 1, 2, 3

_local = threading.local()


def set_kernel_policy(policy: int) -> None:
    """This thread's default kernel choice for sample() calls that pass no `kernel`:
    KERNEL_AUTO, KERNEL_CLUSTER, KERNEL_ROW or KERNEL_ROW_EXACT (kps_step_opts.kernel_policy in
    include/kps.h).  The library itself keeps no choice: it goes with each call."""
    if policy not in (KERNEL_AUTO, KERNEL_CLUSTER, KERNEL_ROW, KERNEL_ROW_EXACT):
        raise ValueError(f"unknown kernel policy {policy}")
    _local.policy = int(policy)


def get_kernel_policy() -> int:
    return getattr(_local, "policy", KERNEL_AUTO)


KERNEL_NAMES = {1: "kps_sample_kernel", 2: "kps_row_kernel"}


def last_kernel() -> str:
    """Name of the kernel this thread's most recent launching sample() call used ("" if none)."""
    return KERNEL_NAMES.get(int(load_library().kps_last_kernel()), "")


def last_launch_count() -> int:
    """Kernels this thread's most recent launching sample() call queued (2: pre-pass + row kernel)."""
    return int(load_library().kps_last_launch_count())


def last_cluster_size() -> int:
    """CTAs per cluster of the kernel this thread's most recent launching sample() call used."""
    return int(load_library().kps_last_cluster_size())


def query_launch(B: int, V: int, dtype: torch.dtype = torch.float32) -> dict:
    lib = load_library()
    cs, nc, sm = ctypes.c_int(0), ctypes.c_int64(0), ctypes.c_size_t(0)
    code = KPS_BF16 if dtype == torch.bfloat16 else KPS_F32
    st = lib.kps_query_launch(B, V, code, ctypes.byref(cs), ctypes.byref(nc), ctypes.byref(sm))
    if st != 0:
        raise KpsError(st, "kps_query_launch")
    return dict(cluster_size=cs.value, chunk_elems=nc.value, smem_bytes=sm.value)


def sample(logits: torch.Tensor, top_k: torch.Tensor, top_p: torch.Tensor, temperature: torch.Tensor,
           q: Optional[torch.Tensor], *, seen_indptr: Optional[torch.Tensor] = None, seen_ids: Optional[torch.Tensor] = None,
           penalty: Optional[torch.Tensor] = None, eps: float = 1e-20, need_logits: bool = False,
           out_idx: Optional[torch.Tensor] = None, out_filtered: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
           seed: Optional[int] = None, step: int = 0, finished: Optional[torch.Tensor] = None,
           eos_id: int = 0, unfinished: Optional[torch.Tensor] = None, seen_bits: Optional[torch.Tensor] = None,
           update_seen: bool = False, kernel: Optional[int] = None):
    """One fused sampling step on the GPU (asynchronous on `stream`).

    q: the race's Exp(1) draws [B, V] fp32, or None to sample off (each row's index is
    the first element of its kept set's order: the argmax of the filtered row).
    seed: race with draws generated from (seed, step) instead (q must then be None;
    kps_sample_seeded in include/kps.h defines them).
    finished (uint8 [B], updated in place), eos_id, unfinished (int32 [1]): the
    end-of-sequence epilogue of kps_sample_step.
    seen_bits (int32 [B, ceil(V/32)], bit v % 32 of word v // 32 = token v seen): the
    seen set in place of seen_indptr/seen_ids; update_seen sets each row's emitted
    token in it after the step (kps_sample_step).
    kernel: the kernel policy of this call (KERNEL_*; default: this thread's
    set_kernel_policy choice, else automatic).
    Returns (out_idx int64[B], out_filtered float32[B,V] or None).
    """
    lib = load_library()
    if logits.dim() != 2:
        raise ValueError("logits must be [B, V]")
    B, V = logits.shape
    dev = logits.device
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    dt = _dtype_code(logits)
    _check(logits, "logits", logits.dtype, (B, V), dev)
    _check(top_k, "top_k", torch.int32, (B,), dev)
    _check(top_p, "top_p", torch.float32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    if q is not None:
        if seed is not None:
            raise ValueError("pass q or seed, not both")
        _check(q, "q", torch.float32, (B, V), dev)
    if seen_indptr is not None:
        _check(seen_indptr, "seen_indptr", torch.int32, (B + 1,), dev)
        if seen_ids is None or penalty is None:
            raise ValueError("seen_indptr, seen_ids and penalty go together")
        _check(seen_ids, "seen_ids", torch.int32, tuple(seen_ids.shape), dev)
        _check(penalty, "penalty", torch.float32, (B,), dev)
    if seen_bits is not None:
        if seen_indptr is not None or seen_ids is not None:
            raise ValueError("pass seen_bits or seen_indptr/seen_ids, not both")
        _check(seen_bits, "seen_bits", torch.int32, (B, (V + 31) // 32), dev)
        if penalty is not None:
            _check(penalty, "penalty", torch.float32, (B,), dev)
    elif update_seen:
        raise ValueError("update_seen needs seen_bits")
    if out_idx is None:
        out_idx = torch.empty(B, dtype=torch.int64, device=dev)
    _check(out_idx, "out_idx", torch.int64, (B,), dev)
    if need_logits:
        if out_filtered is None:
            out_filtered = torch.empty(B, V, dtype=torch.float32, device=dev)
        _check(out_filtered, "out_filtered", torch.float32, (B, V), dev)
    else:
        out_filtered = None
    if workspace is None:
        workspace = new_workspace(B, V, logits.dtype, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    policy = get_kernel_policy() if kernel is None else int(kernel)
    step_call = finished is not None or seen_bits is not None or policy != KERNEL_AUTO
    if step_call:
        if finished is not None:
            _check(finished, "finished", torch.uint8, (B,), dev)
            if unfinished is not None:
                _check(unfinished, "unfinished", torch.int32, (1,), dev)
        elif unfinished is not None:
            raise ValueError("unfinished needs finished")
        opts = StepOpts(_ptr(q) if seed is None else None, 0 if seed is None else 1,
                        0 if seed is None else int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(finished),
                        int(eos_id), _ptr(unfinished), _ptr(seen_bits), 1 if update_seen else 0, policy)
        st = lib.kps_sample_step(_ptr(logits), dt, B, V, _ptr(top_k), _ptr(top_p), _ptr(temperature),
                                 _ptr(seen_indptr), _ptr(seen_ids), _ptr(penalty), ctypes.byref(opts), float(eps),
                                 1 if need_logits else 0, _ptr(out_idx), _ptr(out_filtered), _ptr(workspace),
                                 workspace.numel(), ctypes.c_void_p(s.cuda_stream))
    elif seed is not None:
        st = lib.kps_sample_seeded(_ptr(logits), dt, B, V, _ptr(top_k), _ptr(top_p), _ptr(temperature),
                                   _ptr(seen_indptr), _ptr(seen_ids), _ptr(penalty), int(seed) & (2**64 - 1),
                                   int(step) & (2**64 - 1), float(eps), 1 if need_logits else 0, _ptr(out_idx),
                                   _ptr(out_filtered), _ptr(workspace), workspace.numel(),
                                   ctypes.c_void_p(s.cuda_stream))
    else:
        st = lib.kps_sample(_ptr(logits), dt, B, V, _ptr(top_k), _ptr(top_p), _ptr(temperature),
                            _ptr(seen_indptr), _ptr(seen_ids), _ptr(penalty), _ptr(q), float(eps),
                            1 if need_logits else 0, _ptr(out_idx), _ptr(out_filtered), _ptr(workspace),
                            workspace.numel(), ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise KpsError(st, "kps_sample_step" if step_call else
                       "kps_sample_seeded" if seed is not None else "kps_sample")
    return out_idx, out_filtered


def last_device_status(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Reads and clears the device status word (0 = ok, 5 = a bounded wait ran out)."""
    lib = load_library()
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    out = ctypes.c_int(0)
    st = lib.kps_last_device_status(_ptr(workspace), ctypes.c_void_p(s.cuda_stream), ctypes.byref(out))
    if st != 0:
        raise KpsError(st, "kps_last_device_status")
    return out.value
