"""Seeded synthetic inputs shaped like the pages' workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path's tests and the fp64 oracle can be
fed from it.  Values are drawn in float32 on the chosen device and then cast
(round-to-nearest-even) to the workload's storage type.

Recipe (second argument of N(0, s) read as a variance where the workload
writes one, so ``W ~ N(0, 1/64)`` has standard deviation 1/8 and
``b ~ N(0, 0.01)`` has standard deviation 0.1):

* parameters come from ``Generator.manual_seed(seed)``: W [H, d, d], then
  b [H, d] when the workload has a bias, then per-head outlier dimensions
  (``randperm(d)[:n_outliers]``) when it has outliers;
* batch element ``i`` draws q, k, v [H, n, d] in that order from
  ``Generator.manual_seed(seed * 1_000_003 + 1 + i)``, so any subset of
  sequences can be regenerated without drawing the others;
* outlier dimensions of q and k (the same dimensions in both, per head) are
  multiplied by the outlier factor at every position; v is left alone.

Generating on a CUDA device uses CUDA generators with the same seeds: same
distributions, different values from the CPU draw.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_params", "make_sequences", "make_inputs"]


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "hedgehog" | "taylor2"
    dtype: str           # "f32" | "bf16"
    B: int
    H: int
    n: int
    d: int
    w_std: float = 0.0   # Hedgehog W standard deviation
    b_std: float = 0.0   # 0 -> b = 0
    qk_std: float = 1.0
    v_std: float = 1.0
    n_outliers: int = 0
    outlier_scale: float = 1.0
    chunk: int = 64
    loss: bool = False
    n_decode: int = 0    # decode workloads: steps after an n-token prefill
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # fp32 parity workload: one 64-dim head, 256 tokens, output and loss.
    "hedgehog_f32_1x1x256_d64": Workload(
        "hedgehog_f32_1x1x256_d64", "hedgehog", "f32", 1, 1, 256, 64,
        w_std=1 / 8, b_std=0.0, qk_std=0.5, v_std=0.5, loss=True),
    # GPT-2-small attention shape: 12 heads of 64, 1024-token contexts.
    "gpt2_prefill_8x12x1024_d64": Workload(
        "gpt2_prefill_8x12x1024_d64", "hedgehog", "bf16", 8, 12, 1024, 64,
        w_std=1 / 8, b_std=0.1, qk_std=0.5, v_std=0.5, chunk=64),
    # Llama-2-7B attention shape: 32 heads of 128, outlier q/k dimensions.
    "llama2_prefill_1x32x4096_d128": Workload(
        "llama2_prefill_1x32x4096_d128", "hedgehog", "bf16", 1, 32, 4096, 128,
        w_std=1 / math.sqrt(128), b_std=0.0, qk_std=0.3, v_std=1.0,
        n_outliers=4, outlier_scale=8.0, chunk=64, loss=True),
    # Degree-2 Taylor map, d' = 273 padded to 288.
    "taylor2_prefill_4x8x8192_d16": Workload(
        "taylor2_prefill_4x8x8192_d16", "taylor2", "bf16", 4, 8, 8192, 16,
        qk_std=0.25, v_std=1.0, chunk=64),
    # Recurrent decode: 2048-token prefill then 1024 single-token steps.
    "llama2_decode_128x32_d128": Workload(
        "llama2_decode_128x32_d128", "hedgehog", "bf16", 128, 32, 2048, 128,
        w_std=1 / math.sqrt(128), b_std=0.0, qk_std=0.3, v_std=0.3,
        n_decode=1024),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) % (2**63))
    return g


def make_params(w: Workload, seed: int = 0, device="cpu"):
    """Return (W [H,d,d] in the storage type, b [H,d] fp32, outlier dims [H,k])."""
    if w.kind != "hedgehog":
        dims = None
        if w.n_outliers:
            g = _gen(device, seed)
            dims = torch.stack([torch.randperm(w.d, generator=g, device=device)[: w.n_outliers]
                                for _ in range(w.H)])
        return None, None, dims
    g = _gen(device, seed)
    W = torch.randn(w.H, w.d, w.d, generator=g, device=device) * w.w_std
    if w.b_std > 0:
        b = torch.randn(w.H, w.d, generator=g, device=device) * w.b_std
    else:
        b = torch.zeros(w.H, w.d, device=device)
    dims = None
    if w.n_outliers:
        dims = torch.stack([torch.randperm(w.d, generator=g, device=device)[: w.n_outliers]
                            for _ in range(w.H)])
    return W.to(w.torch_dtype), b.float(), dims


def make_sequences(w: Workload, seqs, n: Optional[int] = None, seed: int = 0,
                   device="cpu", dims=None):
    """q, k, v [len(seqs), H, n, d] in the storage type for the listed batch elements."""
    n = w.n if n is None else n
    qs, ks, vs = [], [], []
    for i in seqs:
        g = _gen(device, seed * 1_000_003 + 1 + int(i))
        q = torch.randn(w.H, n, w.d, generator=g, device=device) * w.qk_std
        k = torch.randn(w.H, n, w.d, generator=g, device=device) * w.qk_std
        v = torch.randn(w.H, n, w.d, generator=g, device=device) * w.v_std
        if dims is not None:
            for h in range(w.H):
                idx = dims[h].to(device)
                q[h][:, idx] *= w.outlier_scale
                k[h][:, idx] *= w.outlier_scale
        qs.append(q.to(w.torch_dtype))
        ks.append(k.to(w.torch_dtype))
        vs.append(v.to(w.torch_dtype))
    return torch.stack(qs), torch.stack(ks), torch.stack(vs)


def make_inputs(w: Workload, seed: int = 0, device="cpu", seqs=None, n: Optional[int] = None):
    """All inputs of a workload as a dict: q, k, v, W, b (W, b None for Taylor)."""
    W, b, dims = make_params(w, seed, device)
    seqs = range(w.B) if seqs is None else seqs
    q, k, v = make_sequences(w, seqs, n=n, seed=seed, device=device, dims=dims)
    return {"q": q, "k": k, "v": v, "W": W, "b": b}
