"""The no-allocation entry point (kps_sample_noalloc) against kps_sample.

kps_sample_noalloc serves callers that cannot allocate device memory (an
allocator that owns the whole GPU, an allocation-free real-time path): it
takes no workspace and keeps its scratch in a fixed array inside the library.
This test calls both entry points through the C ABI on the same inputs and
checks that they agree, on two calls in a row (the second call finds the
first call's contents in the shared scratch).  The file is named so pytest
collects it last.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_token_sampling_gb300 import build
    build.build()
    import decode_token_sampling_gb300 as kps
    lib = kps.load_library()
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.kps_sample_noalloc.restype = I32
    lib.kps_sample_noalloc.argtypes = [P, I32, I64, I64, P, P, P, P, P, P, P, F32, I32, P, P, P]
    return lib


def _inputs(seed, B=8, V=20011):
    import torch
    from decode_token_sampling_gb300.workloads import make_random
    inp = make_random(B, V, seed=seed, penalty=1.2, n_seen=300, need_logits=True)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return inp, dict(logits=d(inp.logits), top_k=d(inp.top_k), top_p=d(inp.top_p), temperature=d(inp.temperature),
                     indptr=d(inp.seen_indptr), ids=d(inp.seen_ids), penalty=d(inp.penalty), q=d(inp.q))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


# (B, V, kernel): a small batch of unaligned rows takes the cluster kernel; a batch of at
# least 64 rows of a vocabulary that is a multiple of 4 takes the row kernel, whose
# workspace here is the 256-byte status word alone (no records).
CASES = [(8, 20011, 1), (96, 20480, 2)]


@pytest.mark.parametrize("B,V,kernel", CASES)
def test_noalloc_matches_kps_sample_twice(lib, B, V, kernel):
    import torch
    stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream)
    for call, seed in enumerate((21, 22)):
        inp, t = _inputs(seed, B, V)
        B, V = inp.B, inp.V
        ref_idx = torch.empty(B, dtype=torch.int64, device="cuda")
        ref_f = torch.empty(B, V, dtype=torch.float32, device="cuda")
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        args = [_ptr(t["logits"]), 0, B, V, _ptr(t["top_k"]), _ptr(t["top_p"]), _ptr(t["temperature"]),
                _ptr(t["indptr"]), _ptr(t["ids"]), _ptr(t["penalty"]), _ptr(t["q"]), ctypes.c_float(inp.eps), 1]
        assert lib.kps_sample(*args, _ptr(ref_idx), _ptr(ref_f), _ptr(ws), ws.numel(), s) == 0
        got_idx = torch.full((B,), -1, dtype=torch.int64, device="cuda")
        got_f = torch.zeros(B, V, dtype=torch.float32, device="cuda")
        assert lib.kps_sample_noalloc(*args, _ptr(got_idx), _ptr(got_f), s) == 0, f"call {call}"
        assert lib.kps_last_kernel() == kernel, f"call {call}: kernel {lib.kps_last_kernel()}"
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got_idx.cpu().numpy(), ref_idx.cpu().numpy())
        g, r = got_f.cpu().numpy(), ref_f.cpu().numpy()
        np.testing.assert_array_equal(g == -np.inf, r == -np.inf)
        fin = r != -np.inf
        np.testing.assert_allclose(g[fin], r[fin], rtol=1e-6, atol=0)


def test_noalloc_rejects_bad_arguments_on_host(lib):
    """Every argument is checked before the shared array is touched: a call without logits,
    or asking for filtered logits without a buffer for them, or with a negative eps, is
    rejected with KPS_ERR_INVALID_ARG."""
    fake = ctypes.c_void_p(1 << 20)
    base = [fake, 0, 4, 100, fake, fake, fake, None, None, None, fake, ctypes.c_float(1e-20), 0, fake, None, None]
    no_logits = list(base)
    no_logits[0] = None
    assert lib.kps_sample_noalloc(*no_logits) == 1
    no_out = list(base)
    no_out[12] = 1  # need_logits without out_filtered
    assert lib.kps_sample_noalloc(*no_out) == 1
    neg_eps = list(base)
    neg_eps[11] = ctypes.c_float(-1.0)
    assert lib.kps_sample_noalloc(*neg_eps) == 1


def test_noalloc_rejects_bad_sizes_on_host(lib):
    fake = ctypes.c_void_p(1 << 20)
    bad_v = [fake, 0, 4, 0, fake, fake, fake, None, None, None, fake, ctypes.c_float(1e-20), 0, fake, None, None]
    assert lib.kps_sample_noalloc(*bad_v) == 1
    bad_dt = [fake, 9, 4, 100, fake, fake, fake, None, None, None, fake, ctypes.c_float(1e-20), 0, fake, None, None]
    assert lib.kps_sample_noalloc(*bad_dt) == 1
