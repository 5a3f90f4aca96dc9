"""Each factor of the kernels' weights and race quotients within its error budget (GPU).

Builds tests/weight_error_scan.cu against the kernels' own header
(kps_weights.cuh) and checks the largest relative error it measures over each
factor's input domain against the constants of error_budget.py, from which the
top-p and race near-tie bands are derived (test_error_budget.py).
"""

import json
import os
import subprocess
import tempfile

import pytest

import error_budget as eb

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def measured():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_token_sampling_gb300 import build
    with tempfile.TemporaryDirectory(prefix="kps_wscan_") as tmp:
        exe = os.path.join(tmp, "weight_error_scan")
        subprocess.check_call([build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "decode_token_sampling_gb300", "csrc"),
                               "-o", exe, os.path.join(HERE, "weight_error_scan.cu")])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    return json.loads(out.stdout)


def test_w24_weight(measured):
    assert measured["w24"] <= eb.EPS_W24


def test_exp_bin_table(measured):
    assert measured["exp_bin"] <= eb.EPS_EXP_BIN


def test_rcp_approx(measured):
    assert measured["rcp"] <= eb.EPS_RCP


def test_softmax_weight(measured):
    assert measured["softmax_weight_grid"] <= eb.EPS_EXPF
    assert measured["softmax_weight_pairs"] <= eb.EPS_SOFTMAX_WEIGHT
