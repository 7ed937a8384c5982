"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments with the documented status codes
before touching a device.  No kernel is launched here."""

import ctypes
import os
import re

import pytest

from softmax_mimicking_feature_gb300 import _abi
from tests._util import lib_or_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "hh.h")).read()
    return sorted(set(re.findall(r"HH_API\s+[\w\s\*]+?\b(hh_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    return lib_or_build()


def test_exports_every_declared_symbol(L):
    names = _declared_symbols()
    assert len(names) >= 9
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(_abi.EXPORTED)


def test_status_strings(L):
    for code in range(7):
        assert L.hh_status_str(code).decode().startswith("HH_")
    assert L.hh_status_str(99) == b"HH_ERR_UNKNOWN"


def test_fmap_dim(L):
    assert L.hh_fmap_dim(0, 64, 1) == 128 and L.hh_fmap_dim(0, 128, 0) == 256
    assert L.hh_fmap_dim(1, 16, 0) == 273 and L.hh_fmap_dim(1, 16, 1) == 288
    assert L.hh_fmap_dim(1, 64, 0) == 4161          # printed on the summary page
    assert L.hh_fmap_dim(7, 16, 0) == -1 and L.hh_fmap_dim(0, 0, 0) == -1


def _fm(kind=0, d=64, Wq=64, bq=None):
    s = _abi.HHFmap()
    s.kind, s.d = kind, d
    s.Wq = Wq
    s.bq = bq
    return s


P = ctypes.c_void_p  # fake, 16-byte aligned device addresses; never dereferenced


def _fwd(L, fm, dtype=1, q=P(256), k=P(512), v=P(768), B=1, H=1, n=8, chunk=0, y=P(1024),
         S=None, z=None, ws=None, wsb=0, st=None):
    return L.hh_linattn_fwd_causal(ctypes.byref(fm), dtype, q, k, v, B, H, n, chunk, y, S, z, ws,
                                   wsb, st, None)


def test_validation_codes(L):
    fm = _fm()
    assert L.hh_linattn_fwd_causal(None, 1, P(16), P(32), P(48), 1, 1, 8, 0, P(64), None, None,
                                   None, 0, None, None) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, dtype=7) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, _fm(kind=5)) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, B=-1) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, H=0) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, n=-3) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, q=None) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, _fm(Wq=None)) == _abi.HH_ERR_INVALID_ARG
    assert _fwd(L, fm, S=P(2048)) == _abi.HH_ERR_INVALID_ARG          # S without z
    assert _fwd(L, fm, q=P(258)) == _abi.HH_ERR_ALIGNMENT
    assert _fwd(L, fm, y=P(1032)) == _abi.HH_ERR_ALIGNMENT
    assert _fwd(L, _fm(bq=P(20))) == _abi.HH_ERR_ALIGNMENT
    assert _fwd(L, _fm(d=96)) == _abi.HH_ERR_UNSUPPORTED             # bf16 Hedgehog d
    assert _fwd(L, _fm(kind=1, d=32)) == _abi.HH_ERR_UNSUPPORTED     # bf16 Taylor d
    assert _fwd(L, _fm(d=200), dtype=0) == _abi.HH_ERR_UNSUPPORTED
    assert _fwd(L, fm, chunk=48) == _abi.HH_ERR_UNSUPPORTED
    # huge sizes overflow the index space
    assert _fwd(L, fm, B=1 << 40, H=1 << 20, n=1 << 20) == _abi.HH_ERR_INVALID_ARG


def test_empty_problems_launch_nothing(L):
    fm = _fm()
    # B = 0: nothing to do, no device needed
    assert _fwd(L, fm, B=0) == _abi.HH_OK
    assert L.hh_linattn_decode_step(ctypes.byref(fm), 1, P(16), P(32), P(48), 0, 4, P(64), P(80),
                                    P(96), None) == _abi.HH_OK
    assert L.hh_feature_map(ctypes.byref(fm), 1, P(16), 0, 2, 2, 0, P(32), None) == _abi.HH_OK


def test_loss_validation(L):
    fm = _fm()
    f = lambda **kw: L.hh_mimicry_loss(
        ctypes.byref(kw.get("fm", fm)), kw.get("dtype", 1), kw.get("q", P(16)), kw.get("k", P(32)),
        kw.get("B", 1), kw.get("H", 1), kw.get("n", 8), kw.get("rows", None),
        kw.get("head", P(64)), kw.get("ws", None), kw.get("wsb", 0), None, None)
    assert f(head=None) == _abi.HH_ERR_INVALID_ARG
    assert f(k=None) == _abi.HH_ERR_INVALID_ARG
    assert f(rows=P(8)) == _abi.HH_ERR_ALIGNMENT
    need = L.hh_loss_workspace_bytes(ctypes.byref(fm), 1, 1, 1, 8)
    assert need > 0
    assert f(ws=None, wsb=0) == _abi.HH_ERR_WORKSPACE
    assert f(ws=P(4096), wsb=need - 1) == _abi.HH_ERR_WORKSPACE


def test_decode_validation(L):
    fm = _fm()
    g = lambda **kw: L.hh_linattn_decode_step(
        ctypes.byref(kw.get("fm", fm)), 1, kw.get("q", P(16)), P(32), P(48), 2, 2,
        kw.get("S", P(64)), kw.get("z", P(80)), kw.get("y", P(96)), None)
    assert g(S=None) == _abi.HH_ERR_INVALID_ARG
    assert g(z=P(84)) == _abi.HH_ERR_ALIGNMENT
    assert g(fm=_fm(d=32)) == _abi.HH_ERR_UNSUPPORTED


def test_workspace_queries_are_consistent(L):
    fm = _fm()
    assert L.hh_fwd_workspace_bytes(None, 1, 1, 1, 8, 0) == 0
    a = L.hh_loss_workspace_bytes(ctypes.byref(fm), 1, 2, 3, 100)
    b = L.hh_loss_workspace_bytes(ctypes.byref(fm), 1, 2, 3, 200)
    assert 0 < a < b and a % 256 == 0
    assert L.hh_loss_workspace_bytes(ctypes.byref(fm), 1, 2, 3, 0) == 0


def _noalloc(L, fm, q=P(256), k=P(512), v=P(768), B=1, H=32, n=1 << 20, y=P(1024), st=None):
    return L.hh_linattn_fwd_causal_noalloc(ctypes.byref(fm), 1, q, k, v, B, H, n, 0, y, None,
                                           None, st, None)


def test_noalloc_checks_arguments_before_its_size(L, monkeypatch):
    # a problem far beyond the 16 MiB scratch (63 segment states of 32 heads
    # at d = 128): bad pointers are still reported as such, not as a
    # workspace shortage
    monkeypatch.setenv("HH_PREFILL_SEGMENTS", "64")
    fm = _fm(d=128)
    assert L.hh_fwd_workspace_bytes(ctypes.byref(fm), 1, 1, 32, 1 << 20, 0) > 16 << 20
    assert _noalloc(L, fm, q=None) == _abi.HH_ERR_INVALID_ARG
    assert _noalloc(L, fm, k=P(520)) == _abi.HH_ERR_ALIGNMENT
    assert _noalloc(L, fm, st=P(1026)) == _abi.HH_ERR_ALIGNMENT
    assert _noalloc(L, _fm(d=96)) == _abi.HH_ERR_UNSUPPORTED
    assert _noalloc(L, fm, B=0) == _abi.HH_OK


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="with a device present the call would be enqueued")
def test_noalloc_without_a_supported_device_is_unsupported(L):
    # valid arguments and no sm_103 device: the device check comes before the
    # size check and before any lookup of the scratch array
    assert _noalloc(L, _fm(d=128)) == _abi.HH_ERR_UNSUPPORTED
    assert _noalloc(L, _fm(d=128), n=300) == _abi.HH_ERR_UNSUPPORTED



def test_loss_grad_workspace_sizes(L):
    # the full workspace adds the causal 128 x 128 tiles of dL/da in bf16 to
    # the minimal one (B H T (T + 1) / 2 tiles, T = ceil(n / 128), 256-byte
    # aligned); float32 (CUDA-core path) stores none
    fm = _fm(d=128)
    for B, H, n in [(1, 32, 4096), (2, 3, 389), (1, 2, 1)]:
        full = L.hh_loss_grad_workspace_bytes(ctypes.byref(fm), 1, B, H, n)
        small = L.hh_loss_grad_workspace_bytes_min(ctypes.byref(fm), 1, B, H, n)
        t = (n + 127) // 128
        g = B * H * t * (t + 1) // 2 * 128 * 128 * 2
        assert full - small == (g + 255) // 256 * 256 and small > 0
    assert (L.hh_loss_grad_workspace_bytes(ctypes.byref(fm), 0, 1, 2, 300) ==
            L.hh_loss_grad_workspace_bytes_min(ctypes.byref(fm), 0, 1, 2, 300))
    assert L.hh_loss_grad_workspace_bytes_min(ctypes.byref(fm), 1, 0, 2, 300) == 0
