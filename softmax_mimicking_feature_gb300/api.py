"""Thin PyTorch binding of the C ABI: same names, argument marshalling only.

Tensors supply device memory and streams; every step of the computation runs
in the library's CUDA kernels.  Output buffers and workspaces are allocated
here with torch (the library itself never allocates) unless passed in.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _abi

__all__ = ["FeatureMap", "fmap_dim", "feature_map", "fwd_workspace_bytes", "fwd_plan",
           "linattn_fwd_causal", "linattn_decode_step", "loss_workspace_bytes",
           "mimicry_loss", "mimicry_stats", "fwd_from_state_workspace_bytes",
           "linattn_fwd_causal_from_state", "loss_grad_workspace_bytes", "mimicry_loss_grad",
           "HHError"]

HHError = _abi.HHError

_DTYPES = {torch.float32: _abi.HH_F32, torch.bfloat16: _abi.HH_BF16}
_KINDS = {"hedgehog": _abi.HH_FMAP_HEDGEHOG, "taylor2": _abi.HH_FMAP_TAYLOR2,
          "hedgehog_softmax": _abi.HH_FMAP_HEDGEHOG_SOFTMAX}


def _dt(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16") from None


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA device tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dims(fm, t: torch.Tensor):
    """(B, H, n, d) of a q / k / v / y tensor in the map's layout."""
    if fm.layout == "bnhd":
        B, n, H, d = t.shape
    else:
        B, H, n, d = t.shape
    return B, H, n, d


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class FeatureMap:
    """A per-layer feature map: kind "hedgehog" (W [H,d,d], b [H,d]),
    "hedgehog_softmax" (W only: softmax over the d directions of each sign)
    or "taylor2"."""
    kind: str
    d: int
    Wq: Optional[torch.Tensor] = None
    bq: Optional[torch.Tensor] = None
    Wk: Optional[torch.Tensor] = None
    bk: Optional[torch.Tensor] = None
    kv_heads: int = 0    # grouped-query attention: k, v have this many heads (0: one per head)
    layout: str = "bhnd"  # q, k, v, y as [B, H, n, d] ("bhnd") or [B, n, H, d] ("bnhd")

    @property
    def kind_id(self) -> int:
        return _KINDS[self.kind]

    def struct(self) -> _abi.HHFmap:
        s = _abi.HHFmap()
        s.kind = self.kind_id
        s.d = self.d
        s.Wq = _ptr(self.Wq)
        s.bq = _ptr(self.bq)
        s.Wk = _ptr(self.Wk)
        s.bk = _ptr(self.bk)
        s.kv_heads = int(self.kv_heads)
        s.layout = {"bhnd": _abi.HH_LAYOUT_BHND, "bnhd": _abi.HH_LAYOUT_BNHD}[self.layout]
        return s

    def dim(self, padded: bool = True) -> int:
        return fmap_dim(self.kind, self.d, padded)


def fmap_dim(kind: str, d: int, padded: bool = True) -> int:
    k = _KINDS[kind]
    return int(_abi.lib().hh_fmap_dim(k, int(d), int(bool(padded))))


def feature_map(fm: FeatureMap, x: torch.Tensor, is_key: bool = False,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """phi(x) for x [B, H, n, d] -> [B, H, n, d'p] (hh_feature_map)."""
    B, H, n, d = _dims(fm, x)
    if out is None:
        out = torch.empty(B, H, n, fm.dim(), dtype=x.dtype, device=x.device)
    s = fm.struct()
    _abi.check(_abi.lib().hh_feature_map(ctypes.byref(s), _dt(x), _ptr(x), int(is_key), B, H, n,
                                         _ptr(out), _stream(stream)), "hh_feature_map")
    return out


def fwd_workspace_bytes(fm: FeatureMap, dtype: torch.dtype, B: int, H: int, n: int,
                        chunk: int = 0) -> int:
    s = fm.struct()
    return int(_abi.lib().hh_fwd_workspace_bytes(ctypes.byref(s), _DTYPES[dtype], B, H, n, chunk))


def fwd_plan(fm: FeatureMap, dtype: torch.dtype, B: int, H: int, n: int, chunk: int = 0):
    """(segments, launches) one hh_linattn_fwd_causal call uses (hh_fwd_plan)."""
    seg, lau = ctypes.c_int(0), ctypes.c_int(0)
    s = fm.struct()
    _abi.check(_abi.lib().hh_fwd_plan(ctypes.byref(s), _DTYPES[dtype], B, H, n, chunk,
                                      ctypes.byref(seg), ctypes.byref(lau)), "hh_fwd_plan")
    return seg.value, lau.value


def linattn_fwd_causal(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       chunk: int = 0, y: Optional[torch.Tensor] = None,
                       return_state: bool = False, workspace: Optional[torch.Tensor] = None,
                       dev_status: Optional[torch.Tensor] = None, stream=None):
    """Causal linear attention (hh_linattn_fwd_causal).

    Returns y, or (y, S, z) with ``return_state``: S [B,H,d'p,d] and
    z [B,H,d'p] float32 hold the state after the last token.
    """
    B, H, n, d = _dims(fm, q)
    if y is None:
        y = torch.empty_like(q)
    S = z = None
    if return_state:
        S = torch.empty(B, H, fm.dim(), d, dtype=torch.float32, device=q.device)
        z = torch.empty(B, H, fm.dim(), dtype=torch.float32, device=q.device)
    need = fwd_workspace_bytes(fm, q.dtype, B, H, n, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = fm.struct()
    _abi.check(_abi.lib().hh_linattn_fwd_causal(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), _ptr(v), B, H, n, chunk, _ptr(y), _ptr(S),
        _ptr(z), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "hh_linattn_fwd_causal")
    return (y, S, z) if return_state else y


def fwd_from_state_workspace_bytes(fm: FeatureMap, dtype: torch.dtype, B: int, H: int, n: int,
                                   chunk: int = 0) -> int:
    s = fm.struct()
    return int(_abi.lib().hh_fwd_from_state_workspace_bytes(ctypes.byref(s), _DTYPES[dtype], B, H,
                                                            n, chunk))


def linattn_fwd_causal_from_state(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor,
                                  v: torch.Tensor, S0: torch.Tensor, z0: torch.Tensor,
                                  chunk: int = 0, y: Optional[torch.Tensor] = None,
                                  return_state: bool = False, in_place: bool = False,
                                  workspace: Optional[torch.Tensor] = None,
                                  dev_status: Optional[torch.Tensor] = None, stream=None):
    """Causal linear attention continuing from state (S0, z0)
    (hh_linattn_fwd_causal_from_state).

    Returns y, or (y, S, z) with ``return_state``; ``in_place`` writes the
    final state over S0, z0 (and returns them as S, z).
    """
    B, H, n, d = _dims(fm, q)
    if y is None:
        y = torch.empty_like(q)
    S = z = None
    if in_place:
        S, z = S0, z0
    elif return_state:
        S = torch.empty_like(S0)
        z = torch.empty_like(z0)
    need = fwd_from_state_workspace_bytes(fm, q.dtype, B, H, n, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = fm.struct()
    _abi.check(_abi.lib().hh_linattn_fwd_causal_from_state(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), _ptr(v), B, H, n, chunk, _ptr(S0), _ptr(z0),
        _ptr(y), _ptr(S), _ptr(z), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "hh_linattn_fwd_causal_from_state")
    return (y, S, z) if (return_state or in_place) else y


def linattn_decode_step(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        S: torch.Tensor, z: torch.Tensor, y: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """One decode step for q, k, v [B, H, d]; updates S, z in place (hh_linattn_decode_step)."""
    B, H, d = q.shape
    if y is None:
        y = torch.empty_like(q)
    s = fm.struct()
    _abi.check(_abi.lib().hh_linattn_decode_step(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), _ptr(v), B, H, _ptr(S), _ptr(z), _ptr(y),
        _stream(stream)), "hh_linattn_decode_step")
    return y


def loss_workspace_bytes(fm: FeatureMap, dtype: torch.dtype, B: int, H: int, n: int) -> int:
    s = fm.struct()
    return int(_abi.lib().hh_loss_workspace_bytes(ctypes.byref(s), _DTYPES[dtype], B, H, n))


def mimicry_loss(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor, return_rows: bool = True,
                 workspace: Optional[torch.Tensor] = None,
                 dev_status: Optional[torch.Tensor] = None, stream=None):
    """Distillation cross-entropy (hh_mimicry_loss): returns (rows [B,H,n] or None, head_sum [B,H])."""
    B, H, n, d = _dims(fm, q)
    rows = torch.empty(B, H, n, dtype=torch.float32, device=q.device) if return_rows else None
    head = torch.empty(B, H, dtype=torch.float32, device=q.device)
    need = loss_workspace_bytes(fm, q.dtype, B, H, n)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = fm.struct()
    _abi.check(_abi.lib().hh_mimicry_loss(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), B, H, n, _ptr(rows), _ptr(head),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)), "hh_mimicry_loss")
    return rows, head


def mimicry_stats(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor,
                  workspace: Optional[torch.Tensor] = None,
                  dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-query (CE, KL, H(p), H(w)) as float32 [B, H, n, 4] (hh_mimicry_stats)."""
    B, H, n, d = _dims(fm, q)
    out = torch.empty(B, H, n, 4, dtype=torch.float32, device=q.device)
    need = loss_workspace_bytes(fm, q.dtype, B, H, n)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = fm.struct()
    _abi.check(_abi.lib().hh_mimicry_stats(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), B, H, n, _ptr(out), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(stream)), "hh_mimicry_stats")
    return out


def loss_grad_workspace_bytes(fm: FeatureMap, dtype: torch.dtype, B: int, H: int, n: int,
                              minimal: bool = False) -> int:
    """Workspace of mimicry_loss_grad (hh_loss_grad_workspace_bytes); minimal:
    the smallest it accepts (hh_loss_grad_workspace_bytes_min), which selects
    the path that stores no tiles of dL/da."""
    s = fm.struct()
    fn = (_abi.lib().hh_loss_grad_workspace_bytes_min if minimal
          else _abi.lib().hh_loss_grad_workspace_bytes)
    return int(fn(ctypes.byref(s), _DTYPES[dtype], B, H, n))


def mimicry_loss_grad(fm: FeatureMap, q: torch.Tensor, k: torch.Tensor,
                      workspace: Optional[torch.Tensor] = None,
                      dev_status: Optional[torch.Tensor] = None, stream=None):
    """Gradient of the summed distillation loss (hh_mimicry_loss_grad).

    Returns (dWq, dbq, dWk, dbk), float32, summed over the batch; dWk, dbk are
    None when the keys share the query map (both sides are then in dWq, dbq).
    The softmax map has no bias: dbq and dbk are None for it.
    """
    B, H, n, d = _dims(fm, q)
    dev = q.device
    separate = fm.Wk is not None and fm.Wk.data_ptr() != fm.Wq.data_ptr()
    bias = fm.kind != "hedgehog_softmax"
    dWq = torch.empty(H, d, d, dtype=torch.float32, device=dev)
    dbq = torch.empty(H, d, dtype=torch.float32, device=dev) if bias else None
    dWk = torch.empty_like(dWq) if separate else None
    dbk = torch.empty(H, d, dtype=torch.float32, device=dev) if separate and bias else None
    need = loss_grad_workspace_bytes(fm, q.dtype, B, H, n)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    s = fm.struct()
    _abi.check(_abi.lib().hh_mimicry_loss_grad(
        ctypes.byref(s), _dt(q), _ptr(q), _ptr(k), B, H, n, _ptr(dWq), _ptr(dbq), _ptr(dWk),
        _ptr(dbk), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "hh_mimicry_loss_grad")
    return dWq, dbq, dWk, dbk
