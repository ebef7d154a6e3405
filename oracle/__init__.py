"""fp64 CPU oracle for edge-packed multi-head attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check of the entry module
and the CPU-baseline leg of the benchmark are the only callers. The product
path never imports this package, and this package never imports the product
package. The arithmetic lives in ``pmha_oracle.c`` (plain C loops in double);
this module only compiles it with gcc and marshals numpy arrays.

Formulas follow the kpnn2 0.3.0 API reference page "PackedMultiheadAttention"
(Notes, steps 1-5; forward() Returns). See ``pmha_oracle.c`` for the
per-function citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pmha_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_EMPTY, ERR_RANGE, ERR_DUPLICATE, ERR_ARG, ERR_NOMEM = range(6)

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_validate_edges.argtypes = [_I64, _I64, _i64, _i64, _i64]
        lib.oracle_validate_edges.restype = ctypes.c_int
        lib.oracle_append_self_loops.argtypes = [_I64, _I64, _i64, _i64, _I64, _I64, _I64]
        lib.oracle_append_self_loops.restype = ctypes.c_int
        lib.oracle_csr_by_target.argtypes = [_I64, _I64, _i64, _i64, _I64, _I64, _I64]
        lib.oracle_csr_by_target.restype = ctypes.c_int
        lib.oracle_linear.argtypes = [_i64, _i64, _i64, _D, _D, _D, _D]
        lib.oracle_linear.restype = None
        lib.oracle_attend.argtypes = [_i64, _i64, _D, _i64, _D, _D, _D, _D]
        lib.oracle_attend.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [_i64] * 5 + [_D] * 11 + [_i64, _I64, _I64, _D, _D]
        lib.oracle_forward.restype = ctypes.c_int
        _U8 = ctypes.POINTER(ctypes.c_ubyte)
        lib.oracle_forward_masked.argtypes = [_i64] * 5 + [_D] * 11 + [_i64, _I64, _I64, _U8, _D, _D]
        lib.oracle_forward_masked.restype = ctypes.c_int
        lib.oracle_attend_masked.argtypes = [_i64, _i64, _D, _i64, _D, _D, _U8, _D, _D]
        lib.oracle_attend_masked.restype = ctypes.c_int
        lib.oracle_linear_backward.argtypes = [_i64, _i64, _i64, _D, _D, _D, _D, _D, _D]
        lib.oracle_linear_backward.restype = None
        lib.oracle_backward.argtypes = ([_i64] * 5 + [_D] * 11 + [_i64, _I64, _I64, _U8] + [_D] * 12)
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_average_heads.argtypes = [_i64, _i64, _D, _D]
        lib.oracle_average_heads.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64a(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _dp(a):
    return None if a is None else a.ctypes.data_as(_D)


def _ip(a):
    return a.ctypes.data_as(_I64)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def validate_edges(source_index, target_index, query_features: int, key_features: int) -> int:
    s, t = _i64a(source_index), _i64a(target_index)
    if s.ndim != 1 or t.ndim != 1 or s.shape != t.shape:
        return ERR_ARG
    return int(_load().oracle_validate_edges(_ip(s), _ip(t), s.size, query_features, key_features))


def append_self_loops(source_index, target_index, n: int):
    s, t = _i64a(source_index), _i64a(target_index)
    os_, ot = np.empty(s.size + n, np.int64), np.empty(s.size + n, np.int64)
    cnt = np.zeros(1, np.int64)
    st = _load().oracle_append_self_loops(_ip(s), _ip(t), s.size, n, _ip(os_), _ip(ot), _ip(cnt))
    if st != OK:
        raise MemoryError("oracle_append_self_loops")
    k = int(cnt[0])
    return os_[:k].copy(), ot[:k].copy()


def csr_by_target(source_index, target_index, query_features: int):
    s, t = _i64a(source_index), _i64a(target_index)
    row_ptr = np.empty(query_features + 1, np.int64)
    col = np.empty(s.size, np.int64)
    perm = np.empty(s.size, np.int64)
    st = _load().oracle_csr_by_target(_ip(s), _ip(t), s.size, query_features,
                                      _ip(row_ptr), _ip(col), _ip(perm))
    if st != OK:
        raise MemoryError("oracle_csr_by_target")
    return row_ptr, col, perm


def linear(x, w, b=None) -> np.ndarray:
    """Y = X W^T + b over the last axis of X (nn.Linear convention)."""
    x, w = _f64(x), _f64(w)
    b = None if b is None else _f64(b)
    out_dim, in_dim = w.shape
    rows = x.size // in_dim
    y = np.empty(x.shape[:-1] + (out_dim,), np.float64)
    _load().oracle_linear(rows, in_dim, out_dim, _dp(x), _dp(w), _dp(b), _dp(y))
    return y


def _mask(m):
    return None if m is None else np.ascontiguousarray(np.asarray(m).astype(np.uint8))


def _mp(m):
    return None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def attend(q, k_rows, v_rows, num_heads: int, masked=None):
    """Per-target attention: returns (mixed (E,), weights (n_edges, H)).
    masked (n_edges,) bool drops those edges (key_padding_mask)."""
    q, k_rows, v_rows = _f64(q), _f64(k_rows), _f64(v_rows)
    E = q.shape[-1]
    n = k_rows.shape[0]
    mixed = np.empty(E, np.float64)
    w = np.empty((n, num_heads), np.float64)
    mk = _mask(masked)
    st = _load().oracle_attend_masked(E, num_heads, _dp(q), n, _dp(k_rows), _dp(v_rows), _mp(mk), _dp(mixed),
                                      _dp(w))
    if st != OK:
        raise ValueError(f"oracle_attend status {st}")
    return mixed, w


def forward(query, key, value, params: dict, source_index, target_index, num_heads: int,
            need_weights: bool = True, key_padding_mask=None):
    """Full forward. query (B, L, E), key/value (B, S, E); params holds wq, wk, wv, wo
    (E, E) and bq, bk, bv, bo (E,) or None; key_padding_mask (B, S) bool or None.
    Returns (output (B, L, E), weights (B, nnz, H) or None)."""
    q, k, v = _f64(query), _f64(key), _f64(value)
    B, L, E = q.shape
    S = k.shape[1]
    s, t = _i64a(source_index), _i64a(target_index)
    p = {n: (None if params.get(n) is None else _f64(params[n]))
         for n in ("wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo")}
    out = np.empty((B, L, E), np.float64)
    w = np.empty((B, s.size, num_heads), np.float64) if need_weights else None
    mk = _mask(key_padding_mask)
    if mk is not None and mk.shape != (B, S):
        raise ValueError(f"key_padding_mask must be ({B}, {S})")
    st = _load().oracle_forward_masked(B, L, S, E, num_heads, _dp(q), _dp(k), _dp(v),
                                       _dp(p["wq"]), _dp(p["bq"]), _dp(p["wk"]), _dp(p["bk"]),
                                       _dp(p["wv"]), _dp(p["bv"]), _dp(p["wo"]), _dp(p["bo"]),
                                       s.size, _ip(s), _ip(t), _mp(mk), _dp(out), _dp(w))
    if st != OK:
        raise ValueError(f"oracle_forward status {st}")
    return out, w


def forward_rows(query, key, value, params: dict, source_index, target_index, num_heads: int,
                 rows, key_padding_mask=None):
    """Output rows and edge weights of selected (sample, target) pairs only.

    rows: iterable of (b, t). Projects only the tokens those rows read, in the
    same order of operations as ``forward``. Returns a list of
    (output_row (E,), edge_ids (deg,), weights (deg, H)).
    """
    s_all, t_all = _i64a(source_index), _i64a(target_index)
    res = []
    for b, t in rows:
        e_ids = np.nonzero(t_all == t)[0]
        srcs = s_all[e_ids]
        q_t = linear(np.asarray(query[b, t]), params["wq"], params.get("bq"))
        k_r = linear(np.asarray(key[b][srcs]), params["wk"], params.get("bk")).reshape(len(srcs), -1)
        v_r = linear(np.asarray(value[b][srcs]), params["wv"], params.get("bv")).reshape(len(srcs), -1)
        masked = None if key_padding_mask is None else np.asarray(key_padding_mask)[b][srcs]
        mixed, w = attend(q_t, k_r, v_r, num_heads, masked)
        out = linear(mixed, params["wo"], params.get("bo"))
        res.append((out, e_ids, w))
    return res


def linear_backward(x, w, dy):
    """Gradients of Y = X W^T + b: returns (dX, dW, db)."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    out_dim, in_dim = w.shape
    rows = x.size // in_dim
    dx = np.empty(x.shape, np.float64)
    dw = np.empty((out_dim, in_dim), np.float64)
    db = np.empty(out_dim, np.float64)
    _load().oracle_linear_backward(rows, in_dim, out_dim, _dp(x), _dp(w), _dp(dy), _dp(dx), _dp(dw), _dp(db))
    return dx, dw, db


def backward(query, key, value, params: dict, source_index, target_index, num_heads: int, dout,
             key_padding_mask=None) -> dict:
    """Gradients of sum(output * dout) for the forward of ``forward``: one
    gradient per input (dquery, dkey, dvalue; add them when inputs are one
    tensor), dwq..dwo and dbq..dbo (None when the layer has no bias)."""
    q, k, v = _f64(query), _f64(key), _f64(value)
    B, L, E = q.shape
    S = k.shape[1]
    s, t = _i64a(source_index), _i64a(target_index)
    p = {n: (None if params.get(n) is None else _f64(params[n]))
         for n in ("wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo")}
    g = _f64(dout)
    if g.shape != (B, L, E):
        raise ValueError(f"dout must be ({B}, {L}, {E})")
    mk = _mask(key_padding_mask)
    if mk is not None and mk.shape != (B, S):
        raise ValueError(f"key_padding_mask must be ({B}, {S})")
    r = {"dquery": np.empty((B, L, E)), "dkey": np.empty((B, S, E)), "dvalue": np.empty((B, S, E))}
    for n in ("wq", "wk", "wv", "wo"):
        r["d" + n] = np.empty((E, E))
    for n in ("bq", "bk", "bv", "bo"):
        r["d" + n] = np.empty(E)
    st = _load().oracle_backward(B, L, S, E, num_heads, _dp(q), _dp(k), _dp(v),
                                 _dp(p["wq"]), _dp(p["bq"]), _dp(p["wk"]), _dp(p["bk"]),
                                 _dp(p["wv"]), _dp(p["bv"]), _dp(p["wo"]), _dp(p["bo"]),
                                 s.size, _ip(s), _ip(t), _mp(mk), _dp(g),
                                 _dp(r["dquery"]), _dp(r["dkey"]), _dp(r["dvalue"]),
                                 _dp(r["dwq"]), _dp(r["dbq"]), _dp(r["dwk"]), _dp(r["dbk"]),
                                 _dp(r["dwv"]), _dp(r["dbv"]), _dp(r["dwo"]), _dp(r["dbo"]))
    if st != OK:
        raise ValueError(f"oracle_backward status {st}")
    for n in ("bq", "bk", "bv", "bo"):
        if p[n] is None:
            r["d" + n] = None
    return r


def average_heads(w_head) -> np.ndarray:
    w = _f64(w_head)
    H = w.shape[-1]
    out = np.empty(w.shape[:-1], np.float64)
    _load().oracle_average_heads(w.size // H, H, _dp(w), _dp(out))
    return out
