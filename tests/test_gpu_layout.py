"""GPU parity of the [B, n, H, d] input layout (HH_LAYOUT_BNHD).

The kernels read [B][n][H][d] tensors through 4-D tensor maps (and store y
with the same layout) but do the same arithmetic in the same order as for
[B][H][n][d].  So every call must return bit for bit what the [B][H][n][d]
call returns on the transposed data -- and that path is checked against the
oracle elsewhere; one case here is also checked against the oracle directly.
Cases cover one and several segments, every map, grouped key/value heads and
the float32 path."""

import numpy as np
import pytest
import torch

import oracle as O
import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, f64, need_gpu, rel_l2_per_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


CASES = {
    "hedgehog_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=3, n=300), "hedgehog", 0),
    "hedgehog_d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1700), "hedgehog", 0),
    "hedgehog_d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=2000), "hedgehog", 0),
    "hedgehog_d128_gqa": ("llama2_prefill_1x32x4096_d128", dict(B=2, H=4, n=389), "hedgehog", 2),
    "taylor_d16_long": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=2, n=2100), "taylor2", 0),
    "softmax_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=4, n=257), "hedgehog_softmax", 2),
    "f32_d64": ("hedgehog_f32_1x1x256_d64", dict(B=2, H=4, n=190), "hedgehog", 2),
}


def _maps(case, seed):
    name, kw, kind, hkv = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    if hkv:
        for t in ("k", "v"):
            x[t] = x[t][:, :hkv].contiguous()
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    args = {"hedgehog": (xd["W"], xd["b"]), "hedgehog_softmax": (xd["W"],), "taylor2": ()}[kind]
    fm = hh.FeatureMap(kind, w.d, *args, kv_heads=hkv)
    fs = hh.FeatureMap(kind, w.d, *args, kv_heads=hkv, layout="bnhd")
    sq = {t: xd[t].transpose(1, 2).contiguous() for t in ("q", "k", "v")}   # [B, n, H, d]
    return w, x, xd, sq, fm, fs, kind


@pytest.mark.parametrize("case", sorted(CASES))
def test_layout_prefill_state_and_continuation(case):
    w, x, xd, sq, fm, fs, kind = _maps(case, 41)
    y, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], return_state=True)
    ys, Ss, zs = hh.linattn_fwd_causal(fs, sq["q"], sq["k"], sq["v"], return_state=True)
    n1 = w.n // 3 + 5
    cut = lambda d, a, b, ax: [d[t].narrow(ax, a, b - a).contiguous() for t in ("q", "k", "v")]
    _, S1, z1 = hh.linattn_fwd_causal(fm, *cut(xd, 0, n1, 2), return_state=True)
    y2 = hh.linattn_fwd_causal_from_state(fm, *cut(xd, n1, w.n, 2), S1, z1)
    _, S1s, z1s = hh.linattn_fwd_causal(fs, *cut(sq, 0, n1, 1), return_state=True)
    y2s = hh.linattn_fwd_causal_from_state(fs, *cut(sq, n1, w.n, 1), S1s, z1s)
    torch.cuda.synchronize()
    assert torch.equal(ys, y.transpose(1, 2))
    assert torch.equal(Ss, S) and torch.equal(zs, z)
    assert torch.equal(y2s, y2.transpose(1, 2))


@pytest.mark.parametrize("case", ["hedgehog_d64", "hedgehog_d128_gqa", "softmax_d64", "f32_d64"])
def test_layout_loss_stats_feature_map(case):
    w, x, xd, sq, fm, fs, kind = _maps(case, 43)
    rows, head = hh.mimicry_loss(fm, xd["q"], xd["k"])
    rows_s, head_s = hh.mimicry_loss(fs, sq["q"], sq["k"])
    st = hh.mimicry_stats(fm, xd["q"], xd["k"])
    st_s = hh.mimicry_stats(fs, sq["q"], sq["k"])
    phi = hh.feature_map(fm, xd["q"])
    phi_s = hh.feature_map(fs, sq["q"])
    torch.cuda.synchronize()
    assert torch.equal(rows_s, rows) and torch.equal(head_s, head)
    assert torch.equal(st_s, st)
    assert torch.equal(phi_s, phi)


@pytest.mark.parametrize("case", ["hedgehog_d64", "hedgehog_d128_gqa", "softmax_d64", "f32_d64"])
def test_layout_loss_gradient(case):
    w, x, xd, sq, fm, fs, kind = _maps(case, 45)
    g = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    gs = hh.mimicry_loss_grad(fs, sq["q"], sq["k"])
    torch.cuda.synchronize()
    for a, b in zip(g, gs):
        assert (a is None and b is None) or torch.equal(a, b)


def test_layout_against_the_oracle():
    w, x, xd, sq, fm, fs, kind = _maps("hedgehog_d64_long", 47)
    ys = hh.linattn_fwd_causal(fs, sq["q"], sq["k"], sq["v"])
    torch.cuda.synchronize()
    ref = O.fwd_causal("hedgehog", f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["W"]), f64(x["b"]))
    assert rel_l2_per_head(f64(ys.transpose(1, 2)), ref) <= BF16_TOL
    assert hh.fwd_plan(fs, w.torch_dtype, w.B, w.H, w.n)[0] > 1
