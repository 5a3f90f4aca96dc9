"""The cluster kernel's bounded copy wait, made to run out (GPU).

A test build of the library (compiled with KPS_TEST_SPIN_CYCLES) is called
with the cluster kernel forced (kps_sample_step, kernel policy 1); it sends each
CTA's first copy wait to a barrier that no copy ever completes, bounded by a
few thousand cycles: the wait gives up, the CTA records KPS_ERR_TIMEOUT in the
workspace status word, gives the real copy its full bound, finds it landed and
finishes the row.  Nothing traps or hangs: the call's results still match the
oracle, kps_last_device_status reports the timeout (and clears it), and a
normal call of the product library afterwards on the same context and
workspace reports 0.
"""

import ctypes

import numpy as np
import pytest

import oracle
from decode_token_sampling_gb300.workloads import make_random

pytestmark = pytest.mark.gpu

KPS_ERR_TIMEOUT = 5


def _bind(path):
    lib = ctypes.CDLL(path)
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.kps_sample.restype = I32
    lib.kps_sample.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, P, F32, I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_last_device_status.restype = I32
    lib.kps_last_device_status.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.kps_sample_step.restype = I32
    lib.kps_sample_step.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, P, F32, I32, P, P, P, ctypes.c_size_t, P]
    lib.kps_last_kernel.restype = I32
    return lib


@pytest.fixture(scope="module")
def libs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_token_sampling_gb300 import build
    oracle.build()
    return _bind(build.build_spin_test()), _bind(build.build())


def _call(lib, inp, ws, stream):
    import torch
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t = [d(inp.logits), d(inp.top_k), d(inp.top_p), d(inp.temperature), d(inp.seen_indptr), d(inp.seen_ids),
         d(inp.penalty), d(inp.q)]
    idx = torch.full((inp.B,), -1, dtype=torch.int64, device="cuda")
    filt = torch.empty(inp.B, inp.V, dtype=torch.float32, device="cuda")
    p = [ctypes.c_void_p(x.data_ptr()) for x in t]
    from decode_token_sampling_gb300 import KERNEL_CLUSTER, StepOpts
    opts = StepOpts(p[7], 0, 0, 0, None, 0, None, None, 0, KERNEL_CLUSTER)
    rc = lib.kps_sample_step(p[0], 0, inp.B, inp.V, p[1], p[2], p[3], p[4], p[5], p[6], ctypes.byref(opts),
                             ctypes.c_float(inp.eps), 1, ctypes.c_void_p(idx.data_ptr()),
                             ctypes.c_void_p(filt.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                             ctypes.c_void_p(stream.cuda_stream))
    return rc, idx, filt


def _status(lib, ws, stream):
    out = ctypes.c_int(-1)
    assert lib.kps_last_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream.cuda_stream),
                                      ctypes.byref(out)) == 0
    return out.value


# (B, V): one row per cluster; more rows than clusters (each CTA issues its next copies after
# the recovered timeout); a long vocabulary on wide clusters
@pytest.mark.parametrize("B,V", [(4, 20480), (700, 20480), (3, 131072)])
def test_copy_wait_times_out_and_recovers(libs, B, V):
    import torch
    from parity import compare
    spin, prod = libs
    stream = torch.cuda.current_stream()
    inp = make_random(B, V, seed=B, penalty=1.2, n_seen=64, need_logits=True)
    ref = oracle.sample(inp)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")

    rc, idx, filt = _call(spin, inp, ws, stream)
    assert rc == 0
    assert spin.kps_last_kernel() == 1  # the cluster kernel, the one with the copy wait
    torch.cuda.synchronize()
    assert _status(spin, ws, stream) == KPS_ERR_TIMEOUT
    compare(inp, ref, idx.cpu().numpy(), filt.cpu().numpy(), f"timed-out wait B={B} V={V}")
    assert _status(spin, ws, stream) == 0  # read and cleared

    rc, idx, filt = _call(prod, inp, ws, stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert _status(prod, ws, stream) == 0
    compare(inp, ref, idx.cpu().numpy(), filt.cpu().numpy(), f"normal call after it B={B} V={V}")
