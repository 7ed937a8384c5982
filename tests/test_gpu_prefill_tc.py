"""Tensor-core prefill specifics: sequence segmentation, state export across
segments, and the bounded-wait status report.  Parity is against the fp64
oracle (max per-head relative L2 <= 5e-3)."""

import os

import numpy as np
import pytest
import torch

import oracle as O
import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, f64, need_gpu, rel_l2_per_head

pytestmark = pytest.mark.gpu

CASES = {
    "gpt2_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=3, n=1000)),
    "llama_d128": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=700)),
    "taylor_d16": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=2, n=900)),
}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


@pytest.fixture
def env(monkeypatch):
    return monkeypatch


def _setup(case, seed):
    name, kw = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = (hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"]) if w.kind == "hedgehog"
          else hh.FeatureMap("taylor2", w.d))
    return w, x, xd, fm


def _phi(w, x, t, h, bi=0):
    a = f64(x[t])[bi, h]
    if w.kind == "hedgehog":
        return O.hedgehog_feature_map(a, f64(x["W"])[h], f64(x["b"])[h])
    return O.taylor2_feature_map(a)


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("segments", [1, 2, 3, 7])
def test_segment_count_does_not_change_the_result(case, segments, env):
    env.setenv("HH_PREFILL_SEGMENTS", str(segments))
    w, x, xd, fm = _setup(case, seed=31)
    P, launches = hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n, 64)
    assert P == min(segments, (w.n + 127) // 128) or P <= segments
    # state pass and output pass, plus the scan for more than two segments or
    # for a state pass split into pieces (the Taylor default)
    assert launches in ((1,) if P == 1 else ((2, 3) if P == 2 else (3,)))
    y, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], chunk=64, return_state=True)
    torch.cuda.synchronize()
    W = None if x["W"] is None else f64(x["W"])
    b = None if x["b"] is None else f64(x["b"])
    y_ref = O.fwd_causal(w.kind, f64(x["q"]), f64(x["k"]), f64(x["v"]), W, b)
    assert rel_l2_per_head(f64(y), y_ref) <= BF16_TOL
    dp = O.taylor2_feature_dim(w.d) if w.kind == "taylor2" else 2 * w.d
    for h in range(w.H):
        pk = _phi(w, x, "k", h)
        S_ref, z_ref = pk.T @ f64(x["v"])[0, h], pk.sum(0)
        Sg, zg = f64(S)[0, h], f64(z)[0, h]
        assert np.linalg.norm(Sg[:dp] - S_ref) <= BF16_TOL * np.linalg.norm(S_ref)
        assert np.linalg.norm(zg[:dp] - z_ref) <= BF16_TOL * np.linalg.norm(z_ref)
        assert np.all(Sg[dp:] == 0) and np.all(zg[dp:] == 0)


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("pieces", [1, 2, 5])
def test_state_pass_pieces_do_not_change_the_result(case, pieces, env):
    # each segment's state summed by up to `pieces` CTAs (at most one per
    # tile) and the pieces added up by the scan: the same result
    env.setenv("HH_PREFILL_SEGMENTS", "3")
    env.setenv("HH_STATE_PIECES", str(pieces))
    w, x, xd, fm = _setup(case, seed=32)
    P, launches = hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n, 64)
    assert P == 3 and launches == 3
    y, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], return_state=True)
    torch.cuda.synchronize()
    W = None if x["W"] is None else f64(x["W"])
    b = None if x["b"] is None else f64(x["b"])
    y_ref = O.fwd_causal(w.kind, f64(x["q"]), f64(x["k"]), f64(x["v"]), W, b)
    assert rel_l2_per_head(f64(y), y_ref) <= BF16_TOL
    for h in range(w.H):
        pk = _phi(w, x, "k", h)
        S_ref = pk.T @ f64(x["v"])[0, h]
        dp = pk.shape[1]
        Sg = f64(S)[0, h]
        assert np.linalg.norm(Sg[:dp] - S_ref) <= BF16_TOL * np.linalg.norm(S_ref)


def test_state_pass_empty_pieces(env):
    # 15 tiles in 3 segments of 5, each summed in 4 pieces of at most 2 tiles:
    # 2 + 2 + 1 + an empty piece (zeros) per segment
    env.setenv("HH_PREFILL_SEGMENTS", "3")
    env.setenv("HH_STATE_PIECES", "4")
    w = wl.WORKLOADS["taylor2_prefill_4x8x8192_d16"].with_(B=1, H=2, n=15 * 128)
    x = wl.make_inputs(w, seed=33)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("taylor2", w.d)
    assert hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n, 64) == (3, 3)
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"])
    torch.cuda.synchronize()
    y_ref = O.fwd_causal("taylor2", f64(x["q"]), f64(x["k"]), f64(x["v"]), None, None)
    assert rel_l2_per_head(f64(y), y_ref) <= BF16_TOL


def test_plan_splits_long_sequences():
    w, x, xd, fm = _setup("llama_d128", seed=1)
    P, launches = hh.fwd_plan(fm, torch.bfloat16, 1, 32, 4096, 64)
    assert P > 1 and launches == (2 if P == 2 else 3)
    need = hh.fwd_workspace_bytes(fm, torch.bfloat16, 1, 32, 4096, 64)
    assert need >= 32 * (P - 1) * (256 * 128 + 256) * 4


def test_bounded_wait_reports_timeout_and_still_completes(env):
    # a zero soft limit makes every wait that is not satisfied at once report
    env.setenv("HH_WAIT_SOFT_LIMIT_NS", "0")
    w, x, xd, fm = _setup("llama_d128", seed=2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6  # HH_ERR_TIMEOUT
    W, b = f64(x["W"]), f64(x["b"])
    y_ref = O.fwd_causal("hedgehog", f64(x["q"]), f64(x["k"]), f64(x["v"]), W, b)
    assert rel_l2_per_head(f64(y), y_ref) <= BF16_TOL
    # with the default limit nothing is reported
    env.delenv("HH_WAIT_SOFT_LIMIT_NS")
    status.zero_()
    hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_constant_values_give_constant_output():
    w, x, xd, fm = _setup("gpt2_d64", seed=3)
    v = torch.full_like(xd["v"], 0.75)
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], v)
    torch.cuda.synchronize()
    assert float((y.float() - 0.75).abs().max()) <= 0.75 * 2 ** -8


def test_first_row_equals_first_value():
    for case in CASES:
        w, x, xd, fm = _setup(case, seed=4)
        y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"])
        torch.cuda.synchronize()
        np.testing.assert_allclose(f64(y)[:, :, 0], f64(x["v"])[:, :, 0], rtol=2 ** -7, atol=1e-6)

