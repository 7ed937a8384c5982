"""Parity at the full benchmark sizes, in the configuration bench.py times.

The GPT-2-shaped workload is checked on every output: the prefill with both
Hedgehog maps and the loss gradient (dW, db) with both.

Where the oracle is too slow for every output, sampled rows are computed one
by one from the definition (row i needs tokens 0..i only); the decode workload
is also checked GPU-against-GPU over all sequences: a 2048-token prefill
followed by 1024 decode steps must equal a 3072-token prefill, final state
included."""

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


def _fm(w, x):
    if w.kind == "hedgehog":
        return hh.FeatureMap("hedgehog", w.d, x["W"], x["b"])
    return hh.FeatureMap("taylor2", w.d)


def _phi(w, x, t, bi, h):
    a = f64(x[t])[bi, h]
    if w.kind == "hedgehog":
        return O.hedgehog_feature_map(a, f64(x["W"])[h], f64(x["b"])[h])
    return O.taylor2_feature_map(a)


def _sample_rows(n, k=24, seed=0):
    r = np.random.default_rng(seed)
    rows = set(r.choice(n, size=min(k, n), replace=False).tolist())
    rows |= {0, 1, 63, 64, 127, 128, n - 1}
    return sorted(i for i in rows if i < n)


def test_gpt2_prefill_all_rows():
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"]
    x = wl.make_inputs(w, seed=0)
    xd = {k: t.cuda() for k, t in x.items()}
    y = hh.linattn_fwd_causal(_fm(w, xd), xd["q"], xd["k"], xd["v"], chunk=64)
    torch.cuda.synchronize()
    ref = O.fwd_causal("hedgehog", f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["W"]), f64(x["b"]))
    assert rel_l2_per_head(f64(y), ref) <= BF16_TOL


@pytest.mark.parametrize("name", ["llama2_prefill_1x32x4096_d128", "taylor2_prefill_4x8x8192_d16"])
def test_long_prefill_sampled_rows(name):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w, seed=0)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    y = hh.linattn_fwd_causal(_fm(w, xd), xd["q"], xd["k"], xd["v"], chunk=64)
    torch.cuda.synchronize()
    yg = f64(y)
    rows = _sample_rows(w.n, seed=1)
    got, ref = [], []
    for bi in range(w.B):
        for h in range(w.H):
            pq, pk = _phi(w, x, "q", bi, h), _phi(w, x, "k", bi, h)
            ref.append(O.linattn_rows(pq, pk, f64(x["v"])[bi, h], rows))
            got.append(yg[bi, h, rows])
    assert rel_l2_per_head(np.stack(got), np.stack(ref), lead=1) <= BF16_TOL


def test_llama_loss_sampled_rows():
    w = wl.WORKLOADS["llama2_prefill_1x32x4096_d128"]
    x = wl.make_inputs(w, seed=0)
    xd = {k: t.cuda() for k, t in x.items()}
    rows_g, head = hh.mimicry_loss(_fm(w, xd), xd["q"], xd["k"])
    torch.cuda.synchronize()
    Lg = f64(rows_g)
    rows = _sample_rows(w.n, k=16, seed=2)
    got, ref = [], []
    for h in range(w.H):
        pq, pk = _phi(w, x, "q", 0, h), _phi(w, x, "k", 0, h)
        ref.append(O.mimicry_loss_rows(f64(x["q"])[0, h], f64(x["k"])[0, h], pq, pk, rows))
        got.append(Lg[0, h, rows])
    assert rel_l2_per_head(np.stack(got), np.stack(ref), lead=1) <= BF16_TOL
    # the head sums are the row sums, and every row obeys L_i >= 0 (Gibbs)
    np.testing.assert_allclose(f64(head), Lg.sum(-1), rtol=1e-5)
    assert np.all(Lg > -1e-3) and abs(Lg[0, :, 0]).max() < 1e-3


def test_gpt2_softmax_map_prefill_all_rows():
    """The softmax-over-features map at the benchmark size: the d = 64 output
    pass forms every row's offsets itself."""
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"]
    x = wl.make_inputs(w, seed=3)
    xd = {k: t.cuda() for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog_softmax", w.d, xd["W"])
    y = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"])
    torch.cuda.synchronize()
    ref = O.fwd_causal("hedgehog_softmax", f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["W"]))
    assert rel_l2_per_head(f64(y), ref) <= BF16_TOL


@pytest.mark.parametrize("kind", ["hedgehog", "hedgehog_softmax"])
def test_gpt2_loss_gradient(kind):
    """dW (and db) of the summed loss over all 96 heads of the benchmark size,
    against the oracle's chain rule; db of bf16 inputs at its own bound."""
    from tests._util import DB_TOL_BF16
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"]
    x = wl.make_inputs(w, seed=4)
    xd = {k: t.cuda() for k, t in x.items()}
    soft = kind == "hedgehog_softmax"
    fm = hh.FeatureMap(kind, w.d, xd["W"], None if soft else xd["b"])
    got = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
    torch.cuda.synchronize()
    ref = O.loss_grad_causal(f64(x["q"]), f64(x["k"]), f64(x["W"]), None if soft else f64(x["b"]),
                             kind=kind)
    assert rel_l2_per_head(f64(got[0]), ref[0], lead=1) <= BF16_TOL
    if soft:
        assert got[1] is None and ref[1] is None
    else:
        assert rel_l2_per_head(f64(got[1]), ref[1], lead=1) <= DB_TOL_BF16


def test_decode_after_prefill_equals_long_prefill():
    w = wl.WORKLOADS["llama2_decode_128x32_d128"]
    n0, steps = w.n, w.n_decode
    x = wl.make_inputs(w, seed=0, device="cuda", n=n0 + steps)
    fm = _fm(w, x)
    pre = [x[t][:, :, :n0].contiguous() for t in ("q", "k", "v")]
    _, S, z = hh.linattn_fwd_causal(fm, *pre, return_state=True)
    y_dec = torch.empty(w.B, w.H, steps, w.d, dtype=torch.bfloat16, device="cuda")
    for t in range(steps):
        y_dec[:, :, t] = hh.linattn_decode_step(
            fm, *(x[u][:, :, n0 + t].contiguous() for u in ("q", "k", "v")), S, z)
    y_full, S_full, z_full = hh.linattn_fwd_causal(fm, x["q"], x["k"], x["v"], return_state=True)
    torch.cuda.synchronize()
    assert rel_l2_per_head(f64(y_dec), f64(y_full[:, :, n0:])) <= BF16_TOL
    assert rel_l2_per_head(f64(S), f64(S_full)) <= BF16_TOL
    assert rel_l2_per_head(f64(z), f64(z_full)) <= BF16_TOL


def test_decode_subset_against_oracle():
    w = wl.WORKLOADS["llama2_decode_128x32_d128"]
    n0, steps = w.n, 64
    x = wl.make_inputs(w, seed=0, seqs=[5, 77], n=n0 + steps)
    xd = {k: t.cuda() for k, t in x.items()}
    fm = _fm(w, xd)
    _, S, z = hh.linattn_fwd_causal(fm, *(xd[t][:, :, :n0].contiguous() for t in ("q", "k", "v")),
                                    return_state=True)
    ys = [hh.linattn_decode_step(fm, *(xd[u][:, :, n0 + t].contiguous() for u in ("q", "k", "v")),
                                 S, z) for t in range(steps)]
    torch.cuda.synchronize()
    yg = f64(torch.stack(ys, dim=2))
    rows = list(range(n0, n0 + steps))
    got, ref = [], []
    for bi in range(2):
        for h in range(w.H):
            pq, pk = _phi(w, x, "q", bi, h), _phi(w, x, "k", bi, h)
            ref.append(O.linattn_rows(pq, pk, f64(x["v"])[bi, h], rows))
            got.append(yg[bi, h])
    assert rel_l2_per_head(np.stack(got), np.stack(ref), lead=1) <= BF16_TOL
