"""Shared helpers for the tests (no method arithmetic here)."""

import os

import numpy as np
import pytest
import torch

BF16_TOL = 5e-3   # max per-head relative L2 error, bf16 inputs / fp32 accumulate
F32_TOL = 1e-5    # max per-head relative L2 error, float32 workloads
# Bias gradient of the mimicry loss with bf16 inputs.  db = sum_t dL/dh_t over
# every token cancels heavily (|sum| is a small fraction of sum |dL/dh_t|), so
# the bf16 rounding of the features (2^-9 relative, entering a_ij, the
# dPhi = G phi contraction and dL/dh = dPhi_+ e^h - dPhi_- e^-h) is amplified
# in db more than in dW or the forward outputs.  tests/test_error_budget.py
# shows it with the fp64 oracle: rounding only the features to bf16 moves db
# by more than BF16_TOL on the 14-query-head GQA inputs (5.5e-3) while dW
# stays inside it.  Bound: twice BF16_TOL.
DB_TOL_BF16 = 1e-2

# Every relative error computed by rel_l2_per_head, with the test that asked
# for it; conftest.py prints the largest per test at the end of the run (and
# writes them to $HH_ERROR_REPORT as JSON when that is set).
MEASURED = []


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2_per_head(a, r, lead=2):
    """Max over the leading ``lead`` axes of ||a - r|| / ||r|| (flattened rest)."""
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert a.shape == r.shape, (a.shape, r.shape)
    m = int(np.prod(a.shape[:lead]))
    a = a.reshape(m, -1)
    r = r.reshape(m, -1)
    num = np.linalg.norm(a - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    den = np.where(den == 0, 1.0, den)
    val = float(np.max(num / den)) if m else 0.0
    MEASURED.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], val))
    return val


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip("needs an sm_103 GPU")


def lib_or_build():
    """The loaded library; builds it first when missing."""
    from softmax_mimicking_feature_gb300 import _abi, build
    import os
    if not os.path.exists(_abi.lib_path()):
        build.build()
    return _abi.lib()
