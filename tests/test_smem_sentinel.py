"""The kernels against the oracle in a debug build whose shared memory starts as a NaN
pattern (GPU).

The library built with -DKPS_DEBUG_SENTINEL fills every word of each block's dynamic
shared memory with 0x7FBADBAD before the kernel runs.  A read of a shared word that no
thread of the launch wrote (a missing barrier, a stale count, an uninitialised slot) then
returns that pattern instead of a previous launch's plausible leftovers, and shows up as a
parity failure.  The cases cover both kernels and every row class: top-k rows alone and
shared by a cluster's CTAs, top-p-only rows with and without the pre-pass records, keep-all
and one-element rows, ties, NaN/inf, penalties, filtered output on and off.
"""

import ctypes

import numpy as np
import pytest

import oracle
from decode_token_sampling_gb300.workloads import make_random, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_token_sampling_gb300 import build
    oracle.build()
    lib = ctypes.CDLL(build.build_sentinel())
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.kps_sample_step.restype = I32
    lib.kps_sample_step.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, P, F32, I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_workspace_size.restype = ctypes.c_size_t
    lib.kps_workspace_size.argtypes = [I64, I64, I32]
    lib.kps_last_device_status.restype = I32
    lib.kps_last_device_status.argtypes = [P, P, ctypes.POINTER(I32)]
    return lib


def _run(lib, inp, policy, need_logits):
    import torch
    from decode_token_sampling_gb300 import StepOpts
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    logits = d(inp.logits) if inp.dtype == "f32" else d(inp.logits.view(np.int16))
    t = [d(inp.top_k), d(inp.top_p), d(inp.temperature)]
    pen = [d(inp.seen_indptr), d(inp.seen_ids), d(inp.penalty)] if inp.seen_indptr is not None else [None] * 3
    q = d(inp.q)
    dt = 0 if inp.dtype == "f32" else 1
    ws = torch.zeros(max(256, lib.kps_workspace_size(inp.B, inp.V, dt)), dtype=torch.uint8, device="cuda")
    idx = torch.full((inp.B,), -1, dtype=torch.int64, device="cuda")
    filt = torch.empty(inp.B, inp.V, dtype=torch.float32, device="cuda") if need_logits else None
    ptr = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
    opts = StepOpts(ptr(q), 0, 0, 0, None, 0, None, None, 0, policy)
    stream = torch.cuda.current_stream()
    rc = lib.kps_sample_step(ptr(logits), dt, inp.B, inp.V, *[ptr(x) for x in t], *[ptr(x) for x in pen],
                             ctypes.byref(opts), ctypes.c_float(inp.eps), 1 if need_logits else 0, ptr(idx), ptr(filt),
                             ptr(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    st = ctypes.c_int(-1)
    assert lib.kps_last_device_status(ptr(ws), ctypes.c_void_p(stream.cuda_stream), ctypes.byref(st)) == 0
    assert st.value == 0
    return idx.cpu().numpy(), (filt.cpu().numpy() if filt is not None else None)


CASES = {
    "batch256_penalty": lambda: make_workload("batch256_penalty", rows=range(0, 256, 2)),
    "batch256_full": lambda: make_workload("batch256_penalty"),
    "flat_rows": lambda: make_workload("flat_nucleus", rows=range(0, 128, 4)),
    "bf16_zipf": lambda: make_workload("bf16_zipf"),
    "small_mixed": lambda: make_workload("small_mixed"),
    "ragged_specials": lambda: make_random(40, 20011, seed=5, special=True, ties=True, penalty=1.3, n_seen=100),
    "keep_all_short": lambda: make_random(70, 4096, seed=6, dtype="bf16", k_skip_frac=0.5),
    "single_long": lambda: make_random(2, 262144, seed=7, dtype="bf16", k_range=(1, 200)),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("policy", [0, 1, 2, 3])
def test_sentinel_build_matches_oracle(lib, case, policy):
    from parity import compare
    inp = CASES[case]()
    ref = oracle.sample(inp, need_logits=True)
    gi, gf = _run(lib, inp, policy, True)
    compare(inp, ref, gi, gf, f"sentinel {case} policy {policy}")
    gi2, _ = _run(lib, inp, policy, False)
    compare(inp, ref, gi2, None, f"sentinel {case} policy {policy} no logits",
            rerun=lambda: _run(lib, inp, policy, True))
