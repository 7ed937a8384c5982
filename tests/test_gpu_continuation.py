"""GPU parity of the prefill continuing from a given state.

hh_linattn_fwd_causal_from_state must give, for the tokens of the call, what
the oracle's recurrence gives when started from the same state ("Complexity
Analysis": the running sums S, z carry every earlier token).  Cases cover the
single- and multi-segment tensor-core paths of every map, the float32 path,
states that did not come from a prefill, in-place state updates and n = 0.
Tolerances: per-head relative L2 <= 5e-3 (bf16 inputs), 1e-5 (float32)."""

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
    "hedgehog_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=2, n=300), "hedgehog"),
    "hedgehog_d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1800), "hedgehog"),
    "hedgehog_d128": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=3, n=389), "hedgehog"),
    "hedgehog_d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=2000), "hedgehog"),
    "taylor_d16": ("taylor2_prefill_4x8x8192_d16", dict(B=2, H=2, n=333), "taylor2"),
    "taylor_d16_long": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=2, n=2100), "taylor2"),
    "softmax_d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1500), "hedgehog_softmax"),
    "f32_d64": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=2, n=190), "hedgehog"),
}


def _setup(case, seed):
    name, kw, kind = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    if kind == "hedgehog":
        fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"])
    elif kind == "hedgehog_softmax":
        fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"])
    else:
        fm = hh.FeatureMap("taylor2", w.d)
    return w, x, xd, fm, kind


def _phi(kind, x, t, bi, h):
    a = f64(x[t])[bi, h]
    if kind == "hedgehog":
        return O.hedgehog_feature_map(a, f64(x["W"])[h], f64(x["b"])[h])
    if kind == "hedgehog_softmax":
        return O.hedgehog_softmax_feature_map(a, f64(x["W"])[h])
    return O.taylor2_feature_map(a)


def _tol(w):
    return F32_TOL if w.dtype == "f32" else BF16_TOL


@pytest.mark.parametrize("case", sorted(CASES))
def test_continuation_equals_one_prefill(case):
    w, x, xd, fm, kind = _setup(case, 17)
    n1 = (w.n * 2) // 5 + 3   # not on a tile boundary
    first = [xd[t][:, :, :n1].contiguous() for t in ("q", "k", "v")]
    rest = [xd[t][:, :, n1:].contiguous() for t in ("q", "k", "v")]
    _, S1, z1 = hh.linattn_fwd_causal(fm, *first, return_state=True)
    y2, S2, z2 = hh.linattn_fwd_causal_from_state(fm, *rest, S1, z1, return_state=True)
    S1c, z1c = S1.clone(), z1.clone()
    y3, S3, z3 = hh.linattn_fwd_causal_from_state(fm, *rest, S1c, z1c, in_place=True)
    torch.cuda.synchronize()
    tol = _tol(w)
    ref = O.fwd_causal(kind, f64(x["q"]), f64(x["k"]), f64(x["v"]),
                       None if kind == "taylor2" else f64(x["W"]),
                       f64(x["b"]) if kind == "hedgehog" else None)
    assert rel_l2_per_head(f64(y2), ref[:, :, n1:]) <= tol
    assert torch.equal(y2, y3) and torch.equal(S2, S3) and torch.equal(z2, z3)
    dp = 2 * w.d if kind != "taylor2" else O.taylor2_feature_dim(w.d)
    for bi in range(w.B):
        for h in range(w.H):
            pk = _phi(kind, x, "k", bi, h)
            S_ref = pk.T @ f64(x["v"])[bi, h]
            z_ref = pk.sum(0)
            assert np.linalg.norm(f64(S2)[bi, h, :dp] - S_ref) <= tol * np.linalg.norm(S_ref)
            assert np.linalg.norm(f64(z2)[bi, h, :dp] - z_ref) <= tol * np.linalg.norm(z_ref)


@pytest.mark.parametrize("case", ["hedgehog_d64", "hedgehog_d128_long", "taylor_d16", "f32_d64"])
def test_continuation_from_an_arbitrary_state(case):
    """A state that no prefill produced (for Taylor not even symmetric in the
    pair rows) enters exactly as the recurrence says."""
    w, x, xd, fm, kind = _setup(case, 23)
    g = np.random.default_rng(5)
    dp = fm.dim()
    S0 = g.normal(size=(w.B, w.H, dp, w.d)) * 3.0
    z0 = np.abs(g.normal(size=(w.B, w.H, dp))) * 5.0 + 1.0
    if kind == "taylor2":
        S0[:, :, 273:] = 0.0
        z0[:, :, 273:] = 0.0
        z0[:, :, 0] += 500.0   # Taylor features change sign: keep phi(q) . z away from 0
    y = hh.linattn_fwd_causal_from_state(
        fm, xd["q"], xd["k"], xd["v"], torch.tensor(S0, dtype=torch.float32, device="cuda"),
        torch.tensor(z0, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    S0r = f64(torch.tensor(S0, dtype=torch.float32))
    z0r = f64(torch.tensor(z0, dtype=torch.float32))
    ref = np.empty(f64(x["v"]).shape)
    nd = O.taylor2_feature_dim(w.d) if kind == "taylor2" else dp
    for bi in range(w.B):
        for h in range(w.H):
            pq, pk = _phi(kind, x, "q", bi, h), _phi(kind, x, "k", bi, h)
            ref[bi, h] = O.linattn_recurrent(pq, pk, f64(x["v"])[bi, h], S0r[bi, h, :nd],
                                             z0r[bi, h, :nd])[0]
    assert rel_l2_per_head(f64(y), ref) <= _tol(w)


def test_continuation_with_no_tokens_returns_the_state():
    w, x, xd, fm, _ = _setup("hedgehog_d64", 3)
    _, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], return_state=True)
    e = xd["q"][:, :, :0].contiguous()
    _, S2, z2 = hh.linattn_fwd_causal_from_state(fm, e, e, e, S, z, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(S2, S) and torch.equal(z2, z)
