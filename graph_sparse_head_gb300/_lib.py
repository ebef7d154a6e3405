"""ctypes declarations of the C ABI in include/pmha.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpmha.so")

PMHA_OK = 0
STATUS_NAMES = {
    0: "PMHA_OK", 1: "PMHA_ERR_INVALID_ARG", 2: "PMHA_ERR_INDEX_RANGE", 3: "PMHA_ERR_DUPLICATE_EDGE",
    4: "PMHA_ERR_EMPTY", 5: "PMHA_ERR_UNSUPPORTED", 6: "PMHA_ERR_WORKSPACE", 7: "PMHA_ERR_CUDA",
    8: "PMHA_ERR_TIMEOUT", 9: "PMHA_ERR_OVERFLOW",
}
PMHA_F32, PMHA_BF16 = 0, 1
PMHA_WEIGHTS_NONE, PMHA_WEIGHTS_AVG, PMHA_WEIGHTS_PER_HEAD = 0, 1, 2

# Every function the header declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class PmhaParams(ctypes.Structure):
    _fields_ = [("embed_dim", ctypes.c_int64), ("num_heads", ctypes.c_int64), ("dtype", ctypes.c_int),
                ("wq", _vp), ("wk", _vp), ("wv", _vp), ("wo", _vp),
                ("bq", _vp), ("bk", _vp), ("bv", _vp), ("bo", _vp)]


class PmhaGrads(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("wq", "wk", "wv", "wo", "bq", "bk", "bv", "bo")]


_P = ctypes.POINTER(PmhaParams)
_G = ctypes.POINTER(PmhaGrads)
_I64P = ctypes.POINTER(ctypes.c_int64)

SIGNATURES = {
    "pmha_build_csr": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, ctypes.POINTER(_vp)]),
    "pmha_graph_info": (ctypes.c_int, [_vp, _I64P, _I64P, _I64P, _I64P]),
    "pmha_graph_split_info": (ctypes.c_int, [_vp, _I64P, _I64P, _I64P]),
    "pmha_graph_export": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp]),
    "pmha_graph_destroy": (None, [_vp]),
    "pmha_forward_workspace_size": (_sz, [_vp, _P, _i64, ctypes.c_int]),
    "pmha_edge_weights_workspace_size": (_sz, [_vp, _P, _i64, ctypes.c_int]),
    "pmha_forward": (ctypes.c_int, [_vp, _P, _vp, _vp, _vp, _vp, _i64, _vp, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "pmha_forward_host_workspace_size": (_sz, [_vp, _P, _i64, ctypes.c_int]),
    "pmha_forward_host": (ctypes.c_int, [_vp, _P, _vp, _vp, _vp, _vp, _i64, _vp, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "pmha_edge_weights": (ctypes.c_int, [_vp, _P, _vp, _vp, _vp, _i64, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "pmha_forward_noalloc": (ctypes.c_int, [_vp, _P, _vp, _vp, _vp, _vp, _i64, _vp, ctypes.c_int, _vp, _vp]),
    "pmha_device_status": (ctypes.c_int, [_vp]),
    "pmha_last_error": (ctypes.c_char_p, []),
    "pmha_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "pmha_profile_read": (ctypes.c_int, [ctypes.c_int, ctypes.c_char_p, _I64P,
                                         ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    "pmha_launch_count": (ctypes.c_int64, []),
    "pmha_backward_workspace_size": (_sz, [_vp, _P, _i64]),
    "pmha_backward": (ctypes.c_int, [_vp, _P, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _G, _vp, _sz, _vp]),
    "pmha_graph_export_by_source": (ctypes.c_int, [_vp, _vp, _vp, _vp]),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libpmha.so; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "or `python graph_sparse_head_gb300/build.py` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class PmhaError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.status_name}: {message}")


def check(status: int, where: str) -> None:
    if status != PMHA_OK:
        msg = load().pmha_last_error()
        raise PmhaError(status, where, msg.decode() if msg else "")
