"""GPU parity with grouped key/value heads (grouped-query attention).

With kv_heads = Hkv, query head h reads key/value head h / (H / Hkv); maps,
states and outputs stay per query head.  The reference is the oracle run on
k, v repeated along the head axis (head h gets copy h / G), which is what the
grouping means.  Covers prefill (one and several segments, every map, float32),
decode, continuation, the loss, the statistics and the loss gradient.
Tolerances: per-head relative L2 <= 5e-3 (bf16 inputs), 1e-5 (float32); the
bias gradient of bf16 inputs 1e-2 (see tests/_util.py)."""

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
    "hedgehog_d64_14q2kv": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=14, n=300), 2, "hedgehog"),
    "hedgehog_d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=4, n=1700), 2, "hedgehog"),
    "hedgehog_d128": ("llama2_prefill_1x32x4096_d128", dict(B=2, H=4, n=389), 2, "hedgehog"),
    "hedgehog_d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=4, n=2000), 1, "hedgehog"),
    "taylor_d16": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=4, n=333), 1, "taylor2"),
    "taylor_d16_long": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=4, n=2100), 2, "taylor2"),
    "softmax_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=4, n=257), 2, "hedgehog_softmax"),
    "f32_d64": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=4, n=190), 2, "hedgehog"),
}


def _setup(case, seed):
    name, kw, hkv, kind = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    for t in ("k", "v"):   # keep one head per group: [B, Hkv, n, d]
        x[t] = x[t][:, : hkv].contiguous()
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    if kind == "hedgehog":
        fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"], kv_heads=hkv)
    elif kind == "hedgehog_softmax":
        fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"], kv_heads=hkv)
    else:
        fm = hh.FeatureMap("taylor2", w.d, kv_heads=hkv)
    return w, x, xd, fm, kind, hkv


def _expand(a, H):
    """[B, Hkv, ...] -> [B, H, ...], query head h taking key/value head h // (H / Hkv)."""
    a = f64(a)
    return np.repeat(a, H // a.shape[1], axis=1)


def _W(kind, x):
    return None if kind == "taylor2" else f64(x["W"])


def _b(kind, x):
    return f64(x["b"]) if kind == "hedgehog" else None


def _tol(w):
    return F32_TOL if w.dtype == "f32" else BF16_TOL


@pytest.mark.parametrize("case", sorted(CASES))
def test_gqa_prefill_and_state(case):
    w, x, xd, fm, kind, hkv = _setup(case, 31)
    y, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], return_state=True)
    torch.cuda.synchronize()
    k, v = _expand(x["k"], w.H), _expand(x["v"], w.H)
    ref = O.fwd_causal(kind, f64(x["q"]), k, v, _W(kind, x), _b(kind, x))
    assert rel_l2_per_head(f64(y), ref) <= _tol(w)
    if case.endswith("_long"):
        assert hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n)[0] > 1
    dp = 2 * w.d if kind != "taylor2" else O.taylor2_feature_dim(w.d)
    for bi in range(w.B):
        for h in range(w.H):
            Wh = None if kind == "taylor2" else _W(kind, x)[h]
            bh = None if kind != "hedgehog" else _b(kind, x)[h]
            pk = O.feature_map(kind, k[bi, h], Wh, bh)
            S_ref = pk.T @ v[bi, h]
            assert np.linalg.norm(f64(S)[bi, h, :dp] - S_ref) <= _tol(w) * np.linalg.norm(S_ref)


@pytest.mark.parametrize("case", ["hedgehog_d64_14q2kv", "hedgehog_d128_long", "taylor_d16", "f32_d64"])
def test_gqa_decode_and_continuation(case):
    w, x, xd, fm, kind, hkv = _setup(case, 33)
    n1, n2 = w.n - 40, w.n - 4
    cut = lambda a, b: [xd[t][:, :, a:b].contiguous() for t in ("q", "k", "v")]
    _, S, z = hh.linattn_fwd_causal(fm, *cut(0, n1), return_state=True)
    y_mid = hh.linattn_fwd_causal_from_state(fm, *cut(n1, n2), S, z, in_place=True)[0]
    y_dec = [hh.linattn_decode_step(fm, *(xd[u][:, :, t].contiguous() for u in ("q", "k", "v")), S, z)
             for t in range(n2, w.n)]
    torch.cuda.synchronize()
    ref = O.fwd_causal(kind, f64(x["q"]), _expand(x["k"], w.H), _expand(x["v"], w.H),
                       _W(kind, x), _b(kind, x))
    assert rel_l2_per_head(f64(y_mid), ref[:, :, n1:n2]) <= _tol(w)
    assert rel_l2_per_head(f64(torch.stack(y_dec, dim=2)), ref[:, :, n2:]) <= _tol(w)


@pytest.mark.parametrize("case", ["hedgehog_d64_14q2kv", "hedgehog_d128", "taylor_d16",
                                  "softmax_d64", "f32_d64"])
def test_gqa_loss_and_stats(case):
    w, x, xd, fm, kind, hkv = _setup(case, 35)
    rows, head = hh.mimicry_loss(fm, xd["q"], xd["k"])
    st = hh.mimicry_stats(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.stats_causal(kind, f64(x["q"]), _expand(x["k"], w.H), _W(kind, x), _b(kind, x))
    assert rel_l2_per_head(f64(rows), ref[..., 0]) <= _tol(w)
    np.testing.assert_allclose(f64(head), ref[..., 0].sum(-1), rtol=_tol(w), atol=1e-6)
    for c in (0, 2, 3):
        assert rel_l2_per_head(f64(st)[..., c], ref[..., c]) <= _tol(w)


@pytest.mark.parametrize("case", ["hedgehog_d64_14q2kv", "hedgehog_d128", "softmax_d64",
                                  "f32_d64"])
@pytest.mark.parametrize("separate", [False, True])
def test_gqa_loss_gradient(case, separate):
    w, x, xd, fm, kind, hkv = _setup(case, 37)
    Wk = bk = None
    if separate:
        x2 = wl.make_inputs(w, seed=38)
        Wk = x2["W"]
        if kind == "hedgehog":
            bk = x2["b"]
            fm = hh.FeatureMap(kind, w.d, xd["W"], xd["b"], Wk.cuda(), bk.cuda(), kv_heads=hkv)
        else:
            fm = hh.FeatureMap(kind, w.d, xd["W"], None, Wk.cuda(), None, kv_heads=hkv)
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), _expand(x["k"], w.H), f64(x["W"]), _b(kind, x),
                             None if Wk is None else f64(Wk), None if bk is None else f64(bk),
                             kind=kind)
    for i, (g, r) in enumerate(zip(got, ref)):
        if r is None:
            assert g is None
            continue
        tol = _tol(w) if (i % 2 == 0 or w.dtype == "f32") else DB_TOL_BF16   # dW / db
        assert rel_l2_per_head(f64(g), r, lead=1) <= tol


def test_gqa_rejects_bad_grouping():
    w, x, xd, fm, kind, hkv = _setup("hedgehog_d128", 1)
    bad = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"], kv_heads=3)   # 4 % 3 != 0
    with pytest.raises(hh.HHError):
        hh.linattn_fwd_causal(bad, xd["q"], xd["q"], xd["q"])
