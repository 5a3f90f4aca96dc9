"""CPU-side checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments on the host before touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_token_sampling_gb300 import build
    build.build()
    import decode_token_sampling_gb300 as kps
    return kps.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kps.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kps_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "kps_sample" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size(lib):
    # the status word, plus one 32896-byte pre-pass record per row (top-p-only rows of a
    # vocabulary past 4096) for up to 1024 rows
    assert lib.kps_workspace_size(256, 151936, 0) == 256 + 256 * 32896
    assert lib.kps_workspace_size(4000, 151936, 1) == 256 + 1024 * 32896
    assert lib.kps_workspace_size(64, 4096, 0) == 256
    assert lib.kps_workspace_size(0, 151936, 0) == 256
    assert lib.kps_workspace_size(-1, 10, 0) == 0
    assert lib.kps_workspace_size(1, 0, 0) == 0
    assert lib.kps_workspace_size(1, 10, 7) == 0


def test_status_strings(lib):
    for code in range(6):
        assert lib.kps_status_string(code)


def _gpu_present() -> bool:
    import torch
    return torch.cuda.is_available()


def _call(lib, **over):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the host checks run first
    args = dict(logits=fake, dt=0, B=4, V=100, top_k=fake, top_p=fake, temperature=fake, seen_indptr=None,
                seen_ids=None, penalty=None, q=fake, eps=1e-20, need_logits=0, out_idx=fake, out_filtered=None,
                workspace=ctypes.c_void_p(1 << 20), workspace_bytes=256, stream=None)
    args.update(over)
    return lib.kps_sample(*args.values())


def test_host_validation_without_gpu(lib):
    assert _call(lib, dt=5) == 1
    assert _call(lib, V=0) == 1
    assert _call(lib, B=-1) == 1
    assert _call(lib, eps=-1.0) == 1
    assert _call(lib, eps=float("nan")) == 1
    assert _call(lib, eps=float("inf")) == 1
    assert _call(lib, workspace=None) == 3
    assert _call(lib, workspace=ctypes.c_void_p((1 << 20) + 8)) == 3
    assert _call(lib, workspace_bytes=8) == 3
    assert _call(lib, B=0) == 0  # valid no-op, nothing launched
    assert _call(lib, logits=None) == 1
    if not _gpu_present():  # a valid call would launch on the fake pointers
        assert _call(lib, q=None) not in (1, 3)  # sampling off: valid (fails only for want of a GPU)
    assert _call(lib, out_idx=None) == 1
    assert _call(lib, need_logits=1, out_filtered=None) == 1


def test_no_silent_cpu_path(lib):
    """Valid arguments on a machine without a GPU must fail with a CUDA error, never compute."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib) == 4


def test_step_options_are_checked_without_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)
    lib.kps_sample_step.restype = ctypes.c_int
    args = [fake, 0, 4, 100, fake, fake, fake, None, None, None, None, ctypes.c_float(1e-20), 0, fake, None,
            ctypes.c_void_p(1 << 20), ctypes.c_size_t(256), None]
    assert lib.kps_sample_step(*args) == 1  # no options

    from decode_token_sampling_gb300 import StepOpts
    o = StepOpts(None, 0, 0, 0, None, 2, fake)  # a count without flags
    args[10] = ctypes.byref(o)
    assert lib.kps_sample_step(*args) == 1



def test_seen_bit_options_are_checked_without_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)
    lib.kps_sample_step.restype = ctypes.c_int
    from decode_token_sampling_gb300 import StepOpts
    args = [fake, 0, 4, 100, fake, fake, fake, None, None, fake, None, ctypes.c_float(1e-20), 0, fake, None,
            ctypes.c_void_p(1 << 20), ctypes.c_size_t(256), None]
    # the bit form and the id list together
    o = StepOpts(None, 0, 0, 0, None, 0, None, fake, 0)
    args[10] = ctypes.byref(o)
    args[7], args[8] = fake, fake
    assert lib.kps_sample_step(*args) == 1
    args[7], args[8] = None, fake
    assert lib.kps_sample_step(*args) == 1
    args[7], args[8] = None, None
    # a misaligned bit matrix
    o2 = StepOpts(None, 0, 0, 0, None, 0, None, ctypes.c_void_p((1 << 20) + 2), 0)
    args[10] = ctypes.byref(o2)
    assert lib.kps_sample_step(*args) == 1
    # an update without bits
    o3 = StepOpts(None, 0, 0, 0, None, 0, None, None, 1)
    args[10] = ctypes.byref(o3)
    assert lib.kps_sample_step(*args) == 1
    # a valid call with bits (and the update) reaches the GPU step: a CUDA error without one
    # (never run where a GPU would launch on the fake pointers)
    if not _gpu_present():
        o4 = StepOpts(None, 0, 0, 0, None, 0, None, fake, 1)
        args[10] = ctypes.byref(o4)
        assert lib.kps_sample_step(*args) not in (1, 3)


def test_kernel_policy_is_per_call_and_checked(lib):
    """The kernel choice travels with each call (kps_step_opts.kernel_policy): the library
    exports no process-wide setter, and an unknown policy is rejected on the host."""
    from decode_token_sampling_gb300 import StepOpts
    assert not hasattr(lib, "kps_set_kernel_policy")
    fake = ctypes.c_void_p(1 << 20)
    opts = StepOpts(fake, 0, 0, 0, None, 0, None, None, 0, 7)
    args = [fake, 0, 4, 100, fake, fake, fake, None, None, None, ctypes.byref(opts), ctypes.c_float(1e-20), 0, fake,
            None, fake, 4096, None]
    assert lib.kps_sample_step(*args) == 1
    opts.kernel_policy = -1
    assert lib.kps_sample_step(*args) == 1


def test_step_opts_layout_matches_the_header(tmp_path):
    """The binding's kps_step_opts has the header's field offsets and size (checked by
    compiling a C program against include/kps.h)."""
    import shutil
    import subprocess
    from decode_token_sampling_gb300 import StepOpts
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = "/usr/local/cuda/include"
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    fields = [name for name, _ in StepOpts._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "kps.h"\nint main(void) {\n'
                   + "".join(f'  printf("%zu\\n", offsetof(kps_step_opts, {f}));\n' for f in fields)
                   + '  printf("%zu\\n", sizeof(kps_step_opts));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [getattr(StepOpts, f).offset for f in fields] + [ctypes.sizeof(StepOpts)]
    assert got == want
