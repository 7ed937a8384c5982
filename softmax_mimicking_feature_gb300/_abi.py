"""ctypes declarations of the C ABI in include/hh.h.

Loading fails loudly when the shared library has not been built: there is
no fallback implementation of any operation.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

HH_OK, HH_ERR_INVALID_ARG, HH_ERR_UNSUPPORTED, HH_ERR_ALIGNMENT = 0, 1, 2, 3
HH_ERR_WORKSPACE, HH_ERR_CUDA, HH_ERR_TIMEOUT = 4, 5, 6
HH_F32, HH_BF16 = 0, 1
HH_FMAP_HEDGEHOG, HH_FMAP_TAYLOR2, HH_FMAP_HEDGEHOG_SOFTMAX = 0, 1, 2
HH_LAYOUT_BHND, HH_LAYOUT_BNHD = 0, 1

EXPORTED = ("hh_version", "hh_status_str", "hh_fmap_dim", "hh_feature_map",
            "hh_fwd_workspace_bytes", "hh_fwd_plan", "hh_linattn_fwd_causal", "hh_linattn_decode_step",
            "hh_loss_workspace_bytes", "hh_mimicry_loss", "hh_linattn_fwd_causal_noalloc",
            "hh_loss_grad_workspace_bytes", "hh_loss_grad_workspace_bytes_min",
            "hh_mimicry_loss_grad", "hh_mimicry_stats",
            "hh_fwd_from_state_workspace_bytes", "hh_linattn_fwd_causal_from_state")


class HHFmap(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("d", ctypes.c_int32),
                ("Wq", ctypes.c_void_p), ("bq", ctypes.c_void_p),
                ("Wk", ctypes.c_void_p), ("bk", ctypes.c_void_p),
                ("kv_heads", ctypes.c_int32), ("layout", ctypes.c_int32)]


class HHError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


_lib = None
_lock = threading.Lock()

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER(HHFmap)

_SIGS = {
    "hh_version": ([], _i32),
    "hh_status_str": ([_i32], ctypes.c_char_p),
    "hh_fmap_dim": ([_i32, _i32, _i32], _i32),
    "hh_feature_map": ([_P, _i32, _vp, _i32, _i64, _i32, _i64, _vp, _vp], _i32),
    "hh_fwd_workspace_bytes": ([_P, _i32, _i64, _i32, _i64, _i32], _sz),
    "hh_fwd_plan": ([_P, _i32, _i64, _i32, _i64, _i32, _vp, _vp], _i32),
    "hh_linattn_fwd_causal": ([_P, _i32, _vp, _vp, _vp, _i64, _i32, _i64, _i32, _vp, _vp, _vp,
                               _vp, _sz, _vp, _vp], _i32),
    "hh_linattn_decode_step": ([_P, _i32, _vp, _vp, _vp, _i64, _i32, _vp, _vp, _vp, _vp], _i32),
    "hh_loss_workspace_bytes": ([_P, _i32, _i64, _i32, _i64], _sz),
    "hh_mimicry_loss": ([_P, _i32, _vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _sz, _vp, _vp], _i32),
    "hh_linattn_fwd_causal_noalloc": ([_P, _i32, _vp, _vp, _vp, _i64, _i32, _i64, _i32, _vp, _vp,
                                       _vp, _vp, _vp], _i32),
    "hh_loss_grad_workspace_bytes": ([_P, _i32, _i64, _i32, _i64], _sz),
    "hh_loss_grad_workspace_bytes_min": ([_P, _i32, _i64, _i32, _i64], _sz),
    "hh_fwd_from_state_workspace_bytes": ([_P, _i32, _i64, _i32, _i64, _i32], _sz),
    "hh_linattn_fwd_causal_from_state": ([_P, _i32, _vp, _vp, _vp, _i64, _i32, _i64, _i32, _vp,
                                          _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp], _i32),
    "hh_mimicry_stats": ([_P, _i32, _vp, _vp, _i64, _i32, _i64, _vp, _vp, _sz, _vp, _vp], _i32),
    "hh_mimicry_loss_grad": ([_P, _i32, _vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _sz,
                              _vp, _vp], _i32),
}


def lib_path() -> str:
    return os.environ.get("HH_LIBRARY", _build.LIB_PATH)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libhh.so not found at {path}: build it first "
                    "(python -m softmax_mimicking_feature_gb300.build); there is no fallback")
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def status_str(status: int) -> str:
    try:
        return lib().hh_status_str(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {status}"


def check(status: int, where: str) -> None:
    if status != HH_OK:
        raise HHError(status, where)
