"""GPU parity of the mimicry-loss gradient w.r.t. the Hedgehog map.

hh_mimicry_loss_grad is compared with the oracle's fp64 chain rule
(loss_grad_causal), itself pinned to finite differences of the loss.  The
sizes span several 32-token tiles and a ragged tail.  Tolerances are the
per-head relative L2 bounds of the forward path: 1e-5 for float32 and 5e-3
for bf16 inputs, whose features are rounded to bf16 before the fp32 sums;
the bias gradient of bf16 inputs has the bound DB_TOL_BF16 (tests/_util.py)."""

import numpy as np
import pytest
import torch

import oracle as O
import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, DB_TOL_BF16, F32_TOL, f64, need_gpu, rel_l2_per_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


CASES = {
    "f32_d64": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=2, n=190)),
    "bf16_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=3, n=300)),
    "bf16_d128": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=3, n=389)),
    # a last tile of more than 64 rows, and nine query tiles (45 stored g tiles)
    "bf16_d128_tail100": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=356)),
    "bf16_d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=1100)),
    "bf16_n1": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1)),
    "f32_n33": ("hedgehog_f32_1x1x256_d64", dict(B=1, H=1, n=33)),
}


def _tol(w):
    return F32_TOL if w.dtype == "f32" else BF16_TOL


def _check(got, ref, tol):
    for i, (g, r) in enumerate(zip(got, ref)):
        if r is None:
            assert g is None
            continue
        err = rel_l2_per_head(f64(g), r, lead=1)
        # dW at tol; db (odd positions) of bf16 inputs at its own bound
        assert err <= (tol if (i % 2 == 0 or tol == F32_TOL) else DB_TOL_BF16), err


@pytest.mark.parametrize("case", sorted(CASES))
def test_loss_grad_shared_map(case):
    name, kw = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=31)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"])
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), f64(x["b"]))
    _check(got, ref, _tol(w))


@pytest.mark.parametrize("case", ["bf16_d64", "bf16_d128", "bf16_d128_tail100"])
def test_loss_grad_minimal_workspace(case):
    # with the minimal workspace both sides form g (no stored tiles): the
    # oracle's result, and the stored-tile path's up to rounding
    name, kw = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=37)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"])
    full = hh.loss_grad_workspace_bytes(fm, w.torch_dtype, w.B, w.H, w.n)
    small = hh.loss_grad_workspace_bytes(fm, w.torch_dtype, w.B, w.H, w.n, minimal=True)
    assert 0 < small < full
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"], workspace=ws)
    fast = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), f64(x["b"]))
    _check(got, ref, _tol(w))
    _check(got, [None if t is None else f64(t) for t in fast], _tol(w))
    with pytest.raises(RuntimeError):
        hh.mimicry_loss_grad(fm, xd["q"], xd["k"], workspace=ws[: small - 256])


@pytest.mark.parametrize("case", ["f32_d64", "bf16_d64", "bf16_d128"])
def test_loss_grad_separate_maps(case):
    name, kw = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=41)
    x2 = wl.make_inputs(w, seed=42)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"], x2["W"].cuda(), x2["b"].cuda())
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), f64(x["b"]),
                             f64(x2["W"]), f64(x2["b"]))
    _check(got, ref, _tol(w))


def test_loss_grad_empty_is_zero():
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"].with_(B=1, H=2, n=4)
    x = wl.make_inputs(w, seed=1)
    fm = hh.FeatureMap("hedgehog", w.d, x["W"].cuda(), x["b"].cuda())
    q0 = torch.empty(1, 2, 0, w.d, dtype=torch.bfloat16, device="cuda")
    dW, db, dWk, dbk = hh.mimicry_loss_grad(fm, q0, q0)
    torch.cuda.synchronize()
    assert dWk is None and dbk is None
    assert torch.all(dW == 0) and torch.all(db == 0)


def test_loss_grad_taylor_unsupported():
    q = torch.zeros(1, 1, 8, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hh.HHError):
        hh.mimicry_loss_grad(hh.FeatureMap("taylor2", 16), q, q)


def test_loss_grad_descends_the_loss():
    """A small step against the gradient lowers the kernel's own loss."""
    w = wl.WORKLOADS["hedgehog_f32_1x1x256_d64"].with_(B=1, H=2, n=160)
    x = wl.make_inputs(w, seed=51)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"])
    dW, db, _, _ = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    L0 = f64(hh.mimicry_loss(fm, xd["q"], xd["k"])[0]).sum()
    g2 = (dW.double().square().sum() + db.double().square().sum()).item()
    eta = 1e-4 * L0 / g2   # small enough for the first-order term to dominate
    fm2 = hh.FeatureMap("hedgehog", w.d, (xd["W"] - eta * dW).contiguous(),
                        (xd["b"] - eta * db).contiguous())
    L1 = f64(hh.mimicry_loss(fm2, xd["q"], xd["k"])[0]).sum()
    drop = L0 - L1
    # first order: the loss falls by eta * |grad|^2
    np.testing.assert_allclose(drop, eta * g2, rtol=0.05)
