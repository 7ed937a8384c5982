"""hh_linattn_fwd_causal_noalloc: the prefill for callers that cannot allocate.

Callers such as plugin interfaces that only receive input/output buffers, or
serving loops that forbid device allocation after start-up, cannot provide
the prefill's workspace.  This entry point keeps that scratch in a fixed
device array inside the library.  The test calls it through the C ABI, twice
in a row on different inputs, and checks each result against the ordinary
entry point (which is given a freshly allocated workspace) within the usual
bf16 tolerance.  The first call loads the array; the test checks that the
second call leaves the device's free memory unchanged, i.e. allocates
nothing.  It also checks that a problem needing more scratch than the array
holds is refused before anything runs.
"""

import ctypes

import numpy as np
import pytest
import torch

import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import _abi
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, f64, need_gpu, rel_l2_per_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(fm, q, k, v, y, S, z, status):
    B, H, n, d = q.shape
    s = fm.struct()
    return _abi.lib().hh_linattn_fwd_causal_noalloc(
        ctypes.byref(s), _abi.HH_BF16, _p(q), _p(k), _p(v), B, H, n, 64, _p(y), _p(S), _p(z),
        _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_the_allocating_entry_point_twice():
    w = wl.WORKLOADS["llama2_prefill_1x32x4096_d128"].with_(B=1, H=8, n=1500)
    fm_inputs = [wl.make_inputs(w, seed=s, device="cuda") for s in (71, 72)]
    for call, x in enumerate(fm_inputs):
        fm = hh.FeatureMap("hedgehog", w.d, x["W"], x["b"])
        segs, _ = hh.fwd_plan(fm, torch.bfloat16, w.B, w.H, w.n, 64)
        assert segs > 1, "the case must use the scratch"
        y = torch.empty_like(x["q"])
        S = torch.empty(w.B, w.H, 2 * w.d, w.d, dtype=torch.float32, device="cuda")
        z = torch.empty(w.B, w.H, 2 * w.d, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(fm, x["q"], x["k"], x["v"], y, S, z, status) == _abi.HH_OK
        torch.cuda.synchronize()
        if call > 0:
            # the array was loaded by the first call; this one allocates nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        y_ref, S_ref, z_ref = hh.linattn_fwd_causal(fm, x["q"], x["k"], x["v"], chunk=64,
                                                    return_state=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_l2_per_head(f64(y), f64(y_ref)) <= BF16_TOL
        assert rel_l2_per_head(f64(S), f64(S_ref)) <= BF16_TOL
        assert rel_l2_per_head(f64(z), f64(z_ref)) <= BF16_TOL


def test_noalloc_refuses_problems_beyond_its_scratch(monkeypatch):
    # 63 segments of 32 heads at d = 128 need ~266 MB of scratch (> 16 MiB)
    monkeypatch.setenv("HH_PREFILL_SEGMENTS", "64")
    w = wl.WORKLOADS["llama2_prefill_1x32x4096_d128"].with_(B=1, H=32, n=8192)
    x = wl.make_inputs(w, seed=73, device="cuda")
    fm = hh.FeatureMap("hedgehog", w.d, x["W"], x["b"])
    assert hh.fwd_workspace_bytes(fm, torch.bfloat16, 1, 32, 8192, 64) > 16 << 20
    y = torch.full_like(x["q"], 3.0)
    rc = _noalloc(fm, x["q"], x["k"], x["v"], y, None, None, None)
    torch.cuda.synchronize()
    assert rc == _abi.HH_ERR_WORKSPACE
    assert bool((y == 3.0).all())  # nothing ran
