"""Edge-packed multi-head attention on GB300 (sm_103a).

Thin Python binding over the C ABI of include/pmha.h. Every step of the layer
runs in the library's CUDA kernels; this module only checks tensor shapes,
passes device pointers and the current torch CUDA stream, and allocates
output / workspace tensors with torch. There is no CPU path: without a built
libpmha.so or without a GPU every call raises.

The layer (kpnn2 0.3.0 API reference, "PackedMultiheadAttention"): each
query token attends only to the key tokens along the live edges
(source_index[e], target_index[e]); scores q_t . k_s / sqrt(d) are
softmaxed over the edges into each target, weight the values, and the heads'
mixes go through out_proj.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import (PMHA_BF16, PMHA_F32, PMHA_WEIGHTS_AVG, PMHA_WEIGHTS_NONE, PMHA_WEIGHTS_PER_HEAD,
                   PmhaError)

__all__ = [
    "Graph", "Params", "PackedMultiheadAttention", "PmhaError", "pmha_build_csr", "pmha_graph_info",
    "pmha_graph_split_info",
    "pmha_graph_export", "pmha_forward", "pmha_forward_host", "pmha_edge_weights",
    "pmha_forward_workspace_size", "pmha_edge_weights_workspace_size", "pmha_forward_host_workspace_size",
    "pmha_device_status", "pmha_profile_enable", "pmha_profile_read", "pmha_launch_count",
    "pmha_backward", "pmha_backward_workspace_size", "pmha_graph_export_by_source",
    "WMODES",
]

WMODES = {"none": PMHA_WEIGHTS_NONE, "avg": PMHA_WEIGHTS_AVG, "per_head": PMHA_WEIGHTS_PER_HEAD}
_DTYPES = {torch.float32: PMHA_F32, torch.bfloat16: PMHA_BF16}


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


class Graph:
    """A built per-target edge view (owns the library's pmha_graph)."""

    def __init__(self, handle: int, device: torch.device):
        self._h = ctypes.c_void_p(handle)
        self.device = device
        nnz, L, S, md = (ctypes.c_int64() for _ in range(4))
        _lib.check(_lib.load().pmha_graph_info(self._h, ctypes.byref(nnz), ctypes.byref(L), ctypes.byref(S),
                                               ctypes.byref(md)), "pmha_graph_info")
        self.nnz, self.query_features, self.key_features, self.max_in_degree = nnz.value, L.value, S.value, md.value

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise RuntimeError("graph was destroyed")
        return self._h

    def destroy(self) -> None:
        if self._h is not None and _lib._lib is not None:
            torch.cuda.synchronize(self.device)
            _lib.load().pmha_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


@dataclasses.dataclass
class Params:
    """The four projections (q_proj, k_proj, v_proj, out_proj): (E, E) weights
    stored (out, in) and (E,) biases (None for bias=False), on one CUDA device,
    all float32 or all bfloat16."""
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    bq: torch.Tensor | None
    bk: torch.Tensor | None
    bv: torch.Tensor | None
    bo: torch.Tensor | None
    num_heads: int

    @property
    def embed_dim(self) -> int:
        return int(self.wq.shape[0])

    @property
    def dtype(self) -> torch.dtype:
        return self.wq.dtype

    def as_struct(self) -> _lib.PmhaParams:
        E = self.embed_dim
        if self.dtype not in _DTYPES:
            raise TypeError(f"parameters must be float32 or bfloat16, not {self.dtype}")
        for n in ("wq", "wk", "wv", "wo"):
            w = getattr(self, n)
            if tuple(w.shape) != (E, E) or w.dtype != self.dtype or not w.is_cuda or not w.is_contiguous():
                raise ValueError(f"{n} must be a contiguous ({E}, {E}) CUDA tensor of dtype {self.dtype}")
        for n in ("bq", "bk", "bv", "bo"):
            b = getattr(self, n)
            if b is not None and (tuple(b.shape) != (E,) or b.dtype != self.dtype or not b.is_cuda
                                  or not b.is_contiguous()):
                raise ValueError(f"{n} must be None or a contiguous ({E},) CUDA tensor of dtype {self.dtype}")
        return _lib.PmhaParams(E, int(self.num_heads), _DTYPES[self.dtype],
                               _ptr(self.wq), _ptr(self.wk), _ptr(self.wv), _ptr(self.wo),
                               _ptr(self.bq), _ptr(self.bk), _ptr(self.bv), _ptr(self.bo))

    @staticmethod
    def from_arrays(arrays: dict, num_heads: int, dtype: torch.dtype, device="cuda") -> "Params":
        def t(x):
            return None if x is None else torch.as_tensor(x).to(device=device, dtype=dtype).contiguous()
        return Params(t(arrays["wq"]), t(arrays["wk"]), t(arrays["wv"]), t(arrays["wo"]),
                      t(arrays.get("bq")), t(arrays.get("bk")), t(arrays.get("bv")), t(arrays.get("bo")),
                      num_heads)


def pmha_build_csr(source_index: torch.Tensor, target_index: torch.Tensor, query_features: int,
                   key_features: int, add_self_loops: bool = False, stream=None) -> Graph:
    """Validate the packed edge index (device int64) and build the per-target view."""
    for n, t in (("source_index", source_index), ("target_index", target_index)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int64 and t.dim() == 1):
            raise TypeError(f"{n} must be a 1-D int64 CUDA tensor")
    src, tgt = source_index.contiguous(), target_index.contiguous()
    if src.numel() != tgt.numel():
        raise ValueError("source_index and target_index differ in length")
    out = ctypes.c_void_p()
    with torch.cuda.device(src.device):
        st = _lib.load().pmha_build_csr(_ptr(src), _ptr(tgt), src.numel(), int(query_features), int(key_features),
                                        int(bool(add_self_loops)), _stream_ptr(stream), ctypes.byref(out))
    _lib.check(st, "pmha_build_csr")
    return Graph(out.value, src.device)


def pmha_graph_info(graph: Graph) -> dict:
    return {"nnz": graph.nnz, "query_features": graph.query_features, "key_features": graph.key_features,
            "max_in_degree": graph.max_in_degree}


def pmha_graph_split_info(graph: Graph) -> dict:
    """How the build split the targets: heavy targets (tensor-core path) and the light edges."""
    n, th, ln = (ctypes.c_int64() for _ in range(3))
    _lib.check(_lib.load().pmha_graph_split_info(graph.handle, ctypes.byref(n), ctypes.byref(th), ctypes.byref(ln)),
               "pmha_graph_split_info")
    return {"n_heavy": n.value, "heavy_min_degree": th.value, "light_nnz": ln.value}


def pmha_graph_export(graph: Graph, stream=None):
    """(row_ptr, col, perm) as int32 CUDA tensors."""
    dev = graph.device
    row_ptr = torch.empty(graph.query_features + 1, dtype=torch.int32, device=dev)
    col = torch.empty(graph.nnz, dtype=torch.int32, device=dev)
    perm = torch.empty(graph.nnz, dtype=torch.int32, device=dev)
    _lib.check(_lib.load().pmha_graph_export(graph.handle, _ptr(row_ptr), _ptr(col), _ptr(perm),
                                             _stream_ptr(stream)), "pmha_graph_export")
    return row_ptr, col, perm


def pmha_graph_export_by_source(graph: Graph, stream=None):
    """(src_row_ptr, target) of the per-source view as int32 CUDA tensors."""
    dev = graph.device
    src_row_ptr = torch.empty(graph.key_features + 1, dtype=torch.int32, device=dev)
    target = torch.empty(graph.nnz, dtype=torch.int32, device=dev)
    _lib.check(_lib.load().pmha_graph_export_by_source(graph.handle, _ptr(src_row_ptr), _ptr(target),
                                                       _stream_ptr(stream)), "pmha_graph_export_by_source")
    return src_row_ptr, target


def pmha_forward_workspace_size(graph: Graph, params: Params, batch: int, wmode: str = "none") -> int:
    p = params.as_struct()
    return int(_lib.load().pmha_forward_workspace_size(graph.handle, ctypes.byref(p), int(batch), WMODES[wmode]))


def pmha_edge_weights_workspace_size(graph: Graph, params: Params, batch: int, wmode: str = "avg") -> int:
    p = params.as_struct()
    return int(_lib.load().pmha_edge_weights_workspace_size(graph.handle, ctypes.byref(p), int(batch),
                                                            WMODES[wmode]))


def pmha_forward_host_workspace_size(graph: Graph, params: Params, batch: int, wmode: str = "none") -> int:
    p = params.as_struct()
    return int(_lib.load().pmha_forward_host_workspace_size(graph.handle, ctypes.byref(p), int(batch),
                                                            WMODES[wmode]))


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if not isinstance(workspace, torch.Tensor) or workspace.device != device or not workspace.is_contiguous():
            raise ValueError(f"workspace must be a contiguous tensor on {device}")
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace holds fewer than the {nbytes} bytes needed")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def _check_dest(name, t, shape, dtype, device):
    """A result tensor the caller supplies: exactly `shape` and `dtype`,
    contiguous, on `device` (None: a host tensor). The kernels write it whole,
    so anything smaller or strided is refused before a launch."""
    if not isinstance(t, torch.Tensor) or tuple(t.shape) != tuple(shape) or t.dtype != dtype \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {tuple(shape)} tensor of {dtype}")
    if device is None:
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor here")
    elif t.device != device:
        raise ValueError(f"{name} must live on {device}")


def _check_placement(graph, params, device):
    """The graph and every parameter tensor on the device of the call."""
    if graph.device != device:
        raise ValueError(f"the graph was built on {graph.device}, the call runs on {device}")
    for n in ("wq", "wk", "wv", "wo", "bq", "bk", "bv", "bo"):
        t = getattr(params, n)
        if t is not None and t.device != device:
            raise ValueError(f"parameter {n} lives on {t.device}, the call runs on {device}")


def _check_tokens(name, x, batch, seq, E, dtype, device):
    if not isinstance(x, torch.Tensor) or x.dim() != 3 or tuple(x.shape) != (batch, seq, E):
        raise ValueError(f"{name} must have shape ({batch}, {seq}, {E})")
    if x.dtype != dtype or x.device != device or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor on {device}")


def _check_mask(mask, batch, S, on_device, device=None):
    """key_padding_mask: None, or a contiguous (B, S) bool / uint8 tensor (nonzero = key dropped)."""
    if mask is None:
        return None
    if not isinstance(mask, torch.Tensor) or tuple(mask.shape) != (batch, S) or \
            mask.dtype not in (torch.bool, torch.uint8) or not mask.is_contiguous():
        raise ValueError(f"key_padding_mask must be a contiguous ({batch}, {S}) bool or uint8 tensor")
    if on_device and mask.device != device:
        raise ValueError(f"key_padding_mask must live on {device}")
    if not on_device and mask.is_cuda:
        raise ValueError("key_padding_mask must be a host tensor here")
    return _ptr(mask)


def _weights_shape(graph, batch, H, wmode):
    return (batch, graph.nnz) if wmode == "avg" else (batch, graph.nnz, H)


def pmha_forward(graph: Graph, params: Params, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                 wmode: str = "none", out: torch.Tensor | None = None, weights: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None, key_padding_mask: torch.Tensor | None = None,
                 check: bool = False):
    """One forward pass on device tensors: query (B, L, E), key / value (B, S, E),
    key_padding_mask (B, S) bool (True = key dropped) or None.
    Returns (output (B, L, E), weights or None). The call returns once the work
    is queued; check=True waits for it and raises what the kernels flagged (for
    bfloat16 layers: an fp16 intermediate out of range, i.e. invalid outputs)."""
    B = int(query.shape[0])
    E, H = params.embed_dim, int(params.num_heads)
    dev = query.device
    _check_tokens("query", query, B, graph.query_features, E, params.dtype, dev)
    _check_tokens("key", key, B, graph.key_features, E, params.dtype, dev)
    _check_tokens("value", value, B, graph.key_features, E, params.dtype, dev)
    mp = _check_mask(key_padding_mask, B, graph.key_features, True, dev)
    _check_placement(graph, params, dev)
    p = params.as_struct()
    lib = _lib.load()
    wm = WMODES[wmode]
    if out is None:
        out = torch.empty_like(query)
    else:
        _check_dest("out", out, (B, graph.query_features, E), params.dtype, dev)
    if wm != PMHA_WEIGHTS_NONE:
        if weights is None:
            weights = torch.empty(_weights_shape(graph, B, H, wmode), dtype=torch.float32, device=dev)
        else:
            _check_dest("weights", weights, _weights_shape(graph, B, H, wmode), torch.float32, dev)
    need = lib.pmha_forward_workspace_size(graph.handle, ctypes.byref(p), B, wm)
    if need == 0:
        _lib.check(_lib.PMHA_OK + 1, "pmha_forward_workspace_size")
    ws = _workspace(need, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.pmha_forward(graph.handle, ctypes.byref(p), _ptr(query), _ptr(key), _ptr(value), mp, B, _ptr(out), wm,
                              _ptr(weights) if wm != PMHA_WEIGHTS_NONE else None, _ptr(ws),
                              ws.numel() * ws.element_size(), _stream_ptr(stream))
    _lib.check(st, "pmha_forward")
    if check:
        with torch.cuda.device(dev):
            pmha_device_status(stream)
    return out, (weights if wm != PMHA_WEIGHTS_NONE else None)


def pmha_forward_host(graph: Graph, params: Params, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                      out: torch.Tensor, wmode: str = "none", weights: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None, device=None,
                      key_padding_mask: torch.Tensor | None = None):
    """Forward pass on HOST tensors (pinned for asynchronous copies): the library
    copies the inputs in, runs the layer and copies out (and weights) back, all
    on the stream. Synchronize the stream before reading `out`."""
    B = int(query.shape[0])
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    E, H = params.embed_dim, int(params.num_heads)
    for n, x, seq in (("query", query, graph.query_features), ("key", key, graph.key_features),
                      ("value", value, graph.key_features), ("out", out, graph.query_features)):
        if x.is_cuda or tuple(x.shape) != (B, seq, E) or x.dtype != params.dtype or not x.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor ({B}, {seq}, {E}) of {params.dtype}")
    mp = _check_mask(key_padding_mask, B, graph.key_features, False)
    _check_placement(graph, params, dev)
    wm = WMODES[wmode]
    if wm != PMHA_WEIGHTS_NONE and weights is not None:
        _check_dest("weights", weights, _weights_shape(graph, B, H, wmode), torch.float32, None)
    p = params.as_struct()
    lib = _lib.load()
    need = lib.pmha_forward_host_workspace_size(graph.handle, ctypes.byref(p), B, wm)
    ws = _workspace(need, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.pmha_forward_host(graph.handle, ctypes.byref(p), _ptr(query), _ptr(key), _ptr(value), mp, B,
                                   _ptr(out),
                                   wm, _ptr(weights) if wm != PMHA_WEIGHTS_NONE else None, _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream_ptr(stream))
    _lib.check(st, "pmha_forward_host")
    return out, weights


def pmha_edge_weights(graph: Graph, params: Params, query: torch.Tensor, key: torch.Tensor, wmode: str = "avg",
                      weights: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None,
                      key_padding_mask: torch.Tensor | None = None):
    """Per-edge softmax weights only (no value projection, mix or out_proj)."""
    B = int(query.shape[0])
    E, H = params.embed_dim, int(params.num_heads)
    dev = query.device
    _check_tokens("query", query, B, graph.query_features, E, params.dtype, dev)
    _check_tokens("key", key, B, graph.key_features, E, params.dtype, dev)
    if wmode not in ("avg", "per_head"):
        raise ValueError("wmode must be 'avg' or 'per_head'")
    mp = _check_mask(key_padding_mask, B, graph.key_features, True, dev)
    _check_placement(graph, params, dev)
    p = params.as_struct()
    lib = _lib.load()
    wm = WMODES[wmode]
    if weights is None:
        weights = torch.empty(_weights_shape(graph, B, H, wmode), dtype=torch.float32, device=dev)
    else:
        _check_dest("weights", weights, _weights_shape(graph, B, H, wmode), torch.float32, dev)
    need = lib.pmha_edge_weights_workspace_size(graph.handle, ctypes.byref(p), B, wm)
    ws = _workspace(need, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.pmha_edge_weights(graph.handle, ctypes.byref(p), _ptr(query), _ptr(key), mp, B, wm, _ptr(weights),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream))
    _lib.check(st, "pmha_edge_weights")
    return weights


def pmha_backward_workspace_size(graph: Graph, params: Params, batch: int) -> int:
    p = params.as_struct()
    return int(_lib.load().pmha_backward_workspace_size(graph.handle, ctypes.byref(p), int(batch)))


def pmha_backward(graph: Graph, params: Params, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                  dout: torch.Tensor, key_padding_mask: torch.Tensor | None = None, input_grads: bool = True,
                  param_grads: bool = True, workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Gradients of the layer for dout = dLoss/d(output): recomputes the forward
    from (query, key, value) and returns {"dquery", "dkey", "dvalue"} in the layer
    dtype (one shared tensor when inputs are one tensor, holding the sum) and
    {"dwq", "dwk", "dwv", "dwo", "dbq", "dbk", "dbv", "dbo"} in float32 (None
    for biases the layer does not have)."""
    B = int(query.shape[0])
    E = params.embed_dim
    dev = query.device
    _check_tokens("query", query, B, graph.query_features, E, params.dtype, dev)
    _check_tokens("key", key, B, graph.key_features, E, params.dtype, dev)
    _check_tokens("value", value, B, graph.key_features, E, params.dtype, dev)
    _check_tokens("dout", dout, B, graph.query_features, E, params.dtype, dev)
    mp = _check_mask(key_padding_mask, B, graph.key_features, True, dev)
    _check_placement(graph, params, dev)
    p = params.as_struct()
    lib = _lib.load()
    out = {}
    gx = [None, None, None]
    if input_grads:
        made = {}
        for i, (name, x) in enumerate((("dquery", query), ("dkey", key), ("dvalue", value))):
            if x.data_ptr() not in made:
                made[x.data_ptr()] = torch.empty_like(x)
            out[name] = made[x.data_ptr()]
            gx[i] = _ptr(out[name])
    g = _lib.PmhaGrads()
    if param_grads:
        for n in ("wq", "wk", "wv", "wo"):
            out["d" + n] = torch.empty((E, E), dtype=torch.float32, device=dev)
            setattr(g, n, _ptr(out["d" + n]))
        for n in ("bq", "bk", "bv", "bo"):
            if getattr(params, n) is None:
                out["d" + n] = None
            else:
                out["d" + n] = torch.empty(E, dtype=torch.float32, device=dev)
                setattr(g, n, _ptr(out["d" + n]))
    need = lib.pmha_backward_workspace_size(graph.handle, ctypes.byref(p), B)
    if need == 0:
        _lib.check(_lib.PMHA_OK + 5, "pmha_backward_workspace_size (unsupported shape)")
    ws = _workspace(need, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.pmha_backward(graph.handle, ctypes.byref(p), _ptr(query), _ptr(key), _ptr(value), mp, B, _ptr(dout),
                               gx[0], gx[1], gx[2], ctypes.byref(g), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream_ptr(stream))
    _lib.check(st, "pmha_backward")
    return out


def pmha_device_status(stream=None) -> None:
    """Synchronize the stream; raise if a kernel flagged a condition since the last
    check: a bounded device-side wait gave up, or an fp16 intermediate overflowed."""
    _lib.check(_lib.load().pmha_device_status(_stream_ptr(stream)), "pmha_device_status")


def pmha_profile_enable(on: bool = True) -> None:
    _lib.check(_lib.load().pmha_profile_enable(int(bool(on))), "pmha_profile_enable")


def pmha_profile_read() -> dict:
    """{stage: (launches, total_ms)} since the last read."""
    n_max = 32
    names = ctypes.create_string_buffer(32 * n_max)
    launches = (ctypes.c_int64 * n_max)()
    totals = (ctypes.c_double * n_max)()
    n = ctypes.c_int()
    _lib.check(_lib.load().pmha_profile_read(n_max, names, launches, totals, ctypes.byref(n)), "pmha_profile_read")
    out = {}
    for i in range(min(n.value, n_max)):
        name = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
        out[name] = (int(launches[i]), float(totals[i]))
    return out


def pmha_launch_count() -> int:
    return int(_lib.load().pmha_launch_count())


class PackedMultiheadAttention:
    """The layer as one object: a built graph plus parameters, called like
    kpnn2's PackedMultiheadAttention.forward on batch-first device tensors:
    ``out, w = layer(query, key, value, key_padding_mask=None, need_weights=False,
    average_attn_weights=True)``.
    Reuses one workspace tensor across calls on the current stream."""

    def __init__(self, source_index, target_index, query_features: int, key_features: int, params: Params,
                 add_self_loops: bool = False, device="cuda"):
        dev = torch.device(device)
        src = torch.as_tensor(source_index, dtype=torch.int64).to(dev)
        tgt = torch.as_tensor(target_index, dtype=torch.int64).to(dev)
        self.graph = pmha_build_csr(src, tgt, query_features, key_features, add_self_loops)
        self.params = params
        self.num_heads = params.num_heads
        self.embed_dim = params.embed_dim
        self.nnz = self.graph.nnz
        self._ws = None

    def __call__(self, query, key, value, key_padding_mask=None, need_weights: bool = False,
                 average_attn_weights: bool = True):
        wmode = "none" if not need_weights else ("avg" if average_attn_weights else "per_head")
        B = int(query.shape[0])
        need = pmha_forward_workspace_size(self.graph, self.params, B, wmode)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=query.device)
        return pmha_forward(self.graph, self.params, query, key, value, wmode, workspace=self._ws,
                            key_padding_mask=key_padding_mask)
