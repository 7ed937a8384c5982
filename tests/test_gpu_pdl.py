"""Programmatic dependent launch keeps every result bit-identical.

The tensor-core kernels are launched as programmatic dependents of the kernel
before them on the stream (HH_PDL=0 launches them as ordinary kernels).  Each
waits for the preceding grids before its first global access, so the results
must not change at all: the chains below (segment state -> scan -> output,
softmax-map offsets -> output, state conversion for a continuation, feature
maps -> loss -> gradient -> share sums) are run both ways and compared bit for
bit, and a CUDA graph of back-to-back calls, the way the benchmark replays
them, must reproduce the eager results."""

import pytest
import torch

import softmax_mimicking_feature_gb300 as hh
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tests._util import lib_or_build
    lib_or_build()


CASES = {
    # multi-segment prefills: state pass, scan and output pass in one call
    "hedgehog_d64_long": ("gpt2_prefill_8x12x1024_d64", dict(B=1, H=2, n=1800), "hedgehog"),
    "hedgehog_d128_long": ("llama2_prefill_1x32x4096_d128", dict(B=1, H=2, n=2000), "hedgehog"),
    "taylor_d16_long": ("taylor2_prefill_4x8x8192_d16", dict(B=1, H=2, n=2100), "taylor2"),
    "softmax_d64": ("gpt2_prefill_8x12x1024_d64", dict(B=2, H=3, n=700), "hedgehog_softmax"),
}


def _setup(case, seed):
    name, kw, kind = CASES[case]
    w = wl.WORKLOADS[name].with_(**kw)
    x = wl.make_inputs(w, seed=seed)
    xd = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    args = {"hedgehog": (xd["W"], xd["b"]), "hedgehog_softmax": (xd["W"],), "taylor2": ()}[kind]
    return w, xd, hh.FeatureMap(kind, w.d, *args)


def _prefill_and_continue(w, xd, fm):
    y, S, z = hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], return_state=True)
    n1 = w.n // 2 + 7
    cut = lambda a, b: [xd[t][:, :, a:b].contiguous() for t in ("q", "k", "v")]
    _, S1, z1 = hh.linattn_fwd_causal(fm, *cut(0, n1), return_state=True)
    y2 = hh.linattn_fwd_causal_from_state(fm, *cut(n1, w.n), S1, z1)
    return [y, S, z, y2]


@pytest.mark.parametrize("case", sorted(CASES))
def test_pdl_on_and_off_agree_bitwise(case, monkeypatch):
    w, xd, fm = _setup(case, 61)
    monkeypatch.setenv("HH_PDL", "1")
    a = _prefill_and_continue(w, xd, fm)
    monkeypatch.setenv("HH_PDL", "0")
    b = _prefill_and_continue(w, xd, fm)
    torch.cuda.synchronize()
    for ta, tb in zip(a, b):
        assert torch.equal(ta, tb)


def test_pdl_loss_and_gradient_chains_bitwise(monkeypatch):
    w = wl.WORKLOADS["llama2_prefill_1x32x4096_d128"].with_(B=1, H=2, n=700)
    x = wl.make_inputs(w, seed=63)
    xd = {k: t.cuda() for k, t in x.items()}
    fm = hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"])

    def run():
        rows, head = hh.mimicry_loss(fm, xd["q"], xd["k"])
        st = hh.mimicry_stats(fm, xd["q"], xd["k"])
        g = hh.mimicry_loss_grad(fm, xd["q"], xd["k"])
        return [rows, head, st] + [t for t in g if t is not None]

    monkeypatch.setenv("HH_PDL", "1")
    a = run()
    monkeypatch.setenv("HH_PDL", "0")
    b = run()
    torch.cuda.synchronize()
    for ta, tb in zip(a, b):
        assert torch.equal(ta, tb)


def test_pdl_graph_of_back_to_back_calls_matches_eager():
    """Consecutive calls in one CUDA graph, each output feeding nothing and each
    input distinct, replayed twice: every output equals the eager call's."""
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"].with_(B=2, H=3, n=1024)
    xs = [wl.make_inputs(w, seed=70 + i) for i in range(3)]
    xds = [{k: t.cuda() for k, t in x.items()} for x in xs]
    fms = [hh.FeatureMap("hedgehog", w.d, xd["W"], xd["b"]) for xd in xds]
    eager = [hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"]) for fm, xd in zip(fms, xds)]
    torch.cuda.synchronize()
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for fm, xd, o in zip(fms, xds, outs):   # warm-up outside the capture
            hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], y=o)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fm, xd, o in zip(fms, xds, outs):
            hh.linattn_fwd_causal(fm, xd["q"], xd["k"], xd["v"], y=o)
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o, e in zip(outs, eager):
            assert torch.equal(o, e)
