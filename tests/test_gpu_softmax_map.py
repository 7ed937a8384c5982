"""GPU parity of the softmax-over-features map and of the per-row statistics.

The map ("The Hedgehog MLP Feature Map", Choice 4 / Eq. 5, negation block
normalised the same way, no bias) runs through every call that takes a
Hedgehog map: feature map, prefill (one- and multi-segment, shared and
separate key maps, float32), state export + decode, loss.  hh_mimicry_stats
(CE, KL, H(p), H(w)) is checked for every map kind, and the loss gradient
through the map's softmax Jacobian (dW only: no bias) against the oracle.  Reference: the fp64
oracle on the same (bf16-rounded) inputs; tolerances as elsewhere: per-head
relative L2 <= 5e-3 (bf16 inputs) or 1e-5 (float32)."""

import numpy as np
import pytest
import torch

import oracle as O
import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, F32_TOL, f64, need_gpu, rel_l2_per_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


CASES = {
    "d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=3, n=300)),
    "d128": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=3, n=389)),
    "d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=2000)),
    "d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=2100)),
    "f32_d64": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=2, n=190)),
    "d64_n1": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1)),
}


def _setup(case, seed):
    name, kw = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"])
    return w, x, xd, fm


def _tol(w):
    return F32_TOL if w.dtype == "f32" else BF16_TOL


@pytest.mark.parametrize("case", ["d64", "d128", "f32_d64"])
@pytest.mark.parametrize("is_key", [0, 1])
def test_softmax_feature_map(case, is_key):
    w, x, xd, fm = _setup(case, 3)
    t = "k" if is_key else "q"
    phi = hh.feature_map(fm, xd[t], is_key=bool(is_key))
    torch.cuda.synchronize()
    ref = np.empty(tuple(x[t].shape[:3]) + (2 * w.d,))
    for h in range(w.H):
        ref[:, h] = O.hedgehog_softmax_feature_map(f64(x[t])[:, h], f64(x["W"])[h])
    assert rel_l2_per_head(f64(phi), ref) <= _tol(w)


@pytest.mark.parametrize("case", sorted(CASES))
def test_softmax_map_prefill(case):
    w, x, xd, fm = _setup(case, 11)
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"])
    torch.cuda.synchronize()
    ref = O.fwd_causal("hedgehog_softmax", f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["W"]))
    assert rel_l2_per_head(f64(y), ref) <= _tol(w)
    if case.endswith("_long"):
        segs, _ = hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n)
        assert segs > 1   # the segment-state kernels ran too


@pytest.mark.parametrize("case", ["d64", "d128"])
def test_softmax_map_separate_key_map(case):
    w, x, xd, _ = _setup(case, 21)
    Wk = wl.make_inputs(w, seed=22)["W"]
    fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"], None, Wk.cuda(), None)
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"])
    torch.cuda.synchronize()
    ref = np.empty(f64(x["v"]).shape)
    for bi in range(w.B):
        for h in range(w.H):
            pq = O.hedgehog_softmax_feature_map(f64(x["q"])[bi, h], f64(x["W"])[h])
            pk = O.hedgehog_softmax_feature_map(f64(x["k"])[bi, h], f64(Wk)[h])
            ref[bi, h] = O.linattn_quadratic(pq, pk, f64(x["v"])[bi, h])
    assert rel_l2_per_head(f64(y), ref) <= BF16_TOL


@pytest.mark.parametrize("case", ["d64", "d128_long", "f32_d64"])
def test_softmax_map_state_and_decode(case):
    w, x, xd, fm = _setup(case, 9)
    n1 = w.n - 5
    pre = [xd[t][:, :, :n1].contiguous() for t in ("q", "k", "v")]
    _, S, z = hh.linattn_fwd_causal(fm, *pre, return_state=True)
    ys = [hh.linattn_decode_step(fm, *(xd[u][:, :, t].contiguous() for u in ("q", "k", "v")), S, z)
          for t in range(n1, w.n)]
    torch.cuda.synchronize()
    ref = O.fwd_causal("hedgehog_softmax", f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["W"]))
    assert rel_l2_per_head(f64(torch.stack(ys, dim=2)), ref[:, :, n1:]) <= _tol(w)
    for bi in range(w.B):
        for h in range(w.H):
            pk = O.hedgehog_softmax_feature_map(f64(x["k"])[bi, h], f64(x["W"])[h])
            S_ref = pk.T @ f64(x["v"])[bi, h]
            z_ref = pk.sum(0)
            assert np.linalg.norm(f64(S)[bi, h] - S_ref) <= _tol(w) * np.linalg.norm(S_ref)
            assert np.linalg.norm(f64(z)[bi, h] - z_ref) <= _tol(w) * np.linalg.norm(z_ref)


@pytest.mark.parametrize("case", ["d64", "d128", "f32_d64", "d64_n1"])
def test_softmax_map_loss(case):
    w, x, xd, fm = _setup(case, 5)
    rows, head = hh.mimicry_loss(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    L, Lh = O.loss_causal("hedgehog_softmax", f64(x["q"]), f64(x["k"]), f64(x["W"]))
    assert rel_l2_per_head(f64(rows), L) <= _tol(w)
    np.testing.assert_allclose(f64(head), Lh, rtol=_tol(w), atol=1e-6)


STATS = {
    "hedgehog_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=2, n=300), "hedgehog"),
    "hedgehog_d128": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=389), "hedgehog"),
    "softmax_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=3, n=257), "hedgehog_softmax"),
    "taylor_d16": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=2, n=333), "taylor2"),
    "hedgehog_f32": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=2, n=190), "hedgehog"),
    "softmax_f32": ("hedgehog_f32_1x1x256_d64", dict(B=1, H=2, n=150), "hedgehog_softmax"),
}


@pytest.mark.parametrize("case", sorted(STATS))
def test_mimicry_stats(case):
    name, kw, kind = STATS[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=13)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    if kind == "taylor2":
        fm, W, b = hh.FeatureMap("taylor2", w.d), None, None
    elif kind == "hedgehog":
        fm, W, b = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"]), f64(x["W"]), f64(x["b"])
    else:
        fm, W, b = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"]), f64(x["W"]), None
    st = hh.mimicry_stats(fm, xd["q"], xd["k"])
    rows, _ = hh.mimicry_loss(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.stats_causal(kind, f64(x["q"]), f64(x["k"]), W, b)
    got = f64(st)
    tol = _tol(w)
    for c in (0, 2, 3):   # CE, H(p), H(w)
        assert rel_l2_per_head(got[..., c], ref[..., c]) <= tol, c
    # KL = CE - H(p) carries the absolute error of CE: bounded relative to CE
    for bi in range(w.B):
        for h in range(w.H):
            err = np.linalg.norm(got[bi, h, :, 1] - ref[bi, h, :, 1])
            assert err <= tol * np.linalg.norm(ref[bi, h, :, 0])
    assert np.all(got[..., 1] >= -1e-3)
    # the CE column is the loss kernel's own row output
    np.testing.assert_allclose(got[..., 0], f64(rows), rtol=1e-5, atol=1e-6)


def test_softmax_map_rejects_bias():
    w, x, xd, fm = _setup("d64", 1)
    with pytest.raises(hh.HHError):
        hh.feature_map(hh.FeatureMap("hedgehog_softmax", w.d, xd["W"], xd["b"]), xd["q"])


def _check_grad(got, ref, tol):
    assert got[1] is None and got[3] is None   # no bias, no db
    for g, r in ((got[0], ref[0]), (got[2], ref[2])):
        if r is None:
            assert g is None
            continue
        assert rel_l2_per_head(f64(g), r, lead=1) <= tol
        # W + u 1^T leaves the map unchanged: every row of dW sums to zero
        rs = f64(g).sum(-1)
        assert np.abs(rs).max() <= 20 * tol * np.abs(f64(g)).max()


# tensor-core gradient (bf16, d 64 / 128, several 128-row tiles and a ragged
# tail), the CUDA-core one (float32; one row), both sides of the loss
GRAD_CASES = ["d64", "d128", "d64_long", "f32_d64", "d64_n1"]


@pytest.mark.parametrize("case", GRAD_CASES)
def test_softmax_map_loss_gradient(case):
    w, x, xd, fm = _setup(case, 31)
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), None,
                             kind="hedgehog_softmax")
    _check_grad(got, ref, _tol(w))


@pytest.mark.parametrize("case", ["d64", "d128", "f32_d64"])
def test_softmax_map_loss_gradient_separate_maps(case):
    w, x, xd, _ = _setup(case, 41)
    Wk = wl.make_inputs(w, seed=42)["W"]
    fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"], None, Wk.cuda(), None)
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), None, f64(Wk), None,
                             kind="hedgehog_softmax")
    _check_grad(got, ref, _tol(w))


def test_softmax_map_gradient_descends_the_loss():
    """A small step against the gradient lowers the kernel's own loss."""
    w, x, xd, fm = _setup("f32_d64", 51)
    dW, _, _, _ = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    L0 = f64(hh.mimicry_loss(fm, xd["q"], xd["k"])[0]).sum()
    eta = 1e-4 * L0 / dW.double().square().sum().item()
    fm2 = hh.FeatureMap("hedgehog_softmax", w.d, (xd["W"] - eta * dW).contiguous())
    L1 = f64(hh.mimicry_loss(fm2, xd["q"], xd["k"])[0]).sum()
    # first-order prediction of the drop: eta |dW|^2 = 1e-4 L0
    assert 0.5e-4 * L0 < L0 - L1 < 2e-4 * L0
