"""Seeded synthetic workloads for edge-packed multi-head attention.

This module only draws random graphs and random tensors. It holds none of the
layer's arithmetic, so both the CUDA path and the oracle may take their inputs
from it. Graph shapes follow the workloads the kpnn2 PackedMultiheadAttention
page describes (gene-regulatory priors with regulator fan-out, pathway->gene
bipartite maps, tens of thousands of gene-like nodes); no dataset is read.

Every generator takes an explicit ``numpy.random.Generator``; the five named
workloads seed theirs from ``PCG64(1000 + id)``. Edge lists come back in a
shuffled order (never sorted), as int64 arrays (source_index, target_index).
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "rng_for", "bf16_round", "make_params",
    "make_tokens", "uniform_graph", "regulator_graph", "powerlaw_indegree_graph",
    "bipartite_membership_graph", "complete_graph", "shuffle_edges",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    id: int
    name: str
    batch: int
    query_features: int
    key_features: int
    embed_dim: int
    num_heads: int
    dtype: str                 # "f32" or "bf16": storage type of tokens and parameters
    bipartite: bool            # query tokens differ from key/value tokens
    weights: tuple             # weight modes the workload exercises: "avg", "per_head"
    nnz_hint: int              # the nominal edge count (config 4 draws its own)


WORKLOADS = {
    1: Workload(1, "tiny_f32_n64_E32_H4", 2, 64, 64, 32, 4, "f32", False, ("per_head", "avg"), 256),
    2: Workload(2, "grn_n2000_E128_H8", 32, 2000, 2000, 128, 8, "bf16", False, (), 40_000),
    3: Workload(3, "skewed_n20000_E128_H8", 16, 20_000, 20_000, 128, 8, "bf16", False, (), 400_000),
    4: Workload(4, "bipartite_L500_S20000_E256_H8", 64, 500, 20_000, 256, 8, "bf16", True,
                ("avg", "per_head"), 137_500),
    5: Workload(5, "complete_n1024_E512_H8", 8, 1024, 1024, 512, 8, "bf16", False, (), 1_048_576),
}


def workload(i: int) -> Workload:
    return WORKLOADS[int(i)]


def rng_for(workload_id: int, stream: int) -> np.random.Generator:
    """Independent streams per workload: 0 = graph, 1 = parameters, 2 = tokens."""
    ss = np.random.SeedSequence(1000 + int(workload_id))
    return np.random.Generator(np.random.PCG64(ss.spawn(3)[stream]))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32.

    Inputs are finite. The result converts to torch.bfloat16 exactly."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32, copy=False)
    return bf16_round(x) if dtype == "bf16" else x


def make_params(rng: np.random.Generator, embed_dim: int, dtype: str, bias: bool = True) -> dict:
    """Four (E, E) projections, Xavier-uniform with bound sqrt(6 / (E + E)) as the
    kpnn2 page's reset_parameters describes, and biases U(-0.1, 0.1) (nonzero so
    that the bias path is exercised). Values are rounded to the storage type."""
    E = embed_dim
    bound = np.sqrt(6.0 / (E + E))
    p = {}
    for n in ("q", "k", "v", "o"):
        p["w" + n] = _store(rng.uniform(-bound, bound, size=(E, E)), dtype)
    for n in ("q", "k", "v", "o"):
        p["b" + n] = _store(rng.uniform(-0.1, 0.1, size=(E,)), dtype) if bias else None
    return p


def make_tokens(rng: np.random.Generator, batch: int, seq: int, embed_dim: int,
                dtype: str) -> np.ndarray:
    """Tokens ~ N(0, 1), (batch, seq, embed_dim), rounded to the storage type."""
    x = rng.standard_normal(size=(batch, seq, embed_dim), dtype=np.float32)
    return _store(x, dtype)


def padding_mask(rng: np.random.Generator, batch: int, seq: int, min_keep: float = 0.5) -> np.ndarray:
    """key_padding_mask of samples padded at the end: sample b keeps its first
    n_b ~ U[min_keep * seq, seq] keys and flags the rest (True = padding)."""
    keep = rng.integers(int(np.ceil(min_keep * seq)), seq + 1, size=batch)
    return np.arange(seq)[None, :] >= keep[:, None]


def scattered_mask(rng: np.random.Generator, batch: int, seq: int, p: float) -> np.ndarray:
    """key_padding_mask with each key flagged independently with probability p."""
    return rng.random((batch, seq)) < p


def shuffle_edges(rng, src, tgt):
    p = rng.permutation(len(src))
    return np.ascontiguousarray(src[p], dtype=np.int64), np.ascontiguousarray(tgt[p], dtype=np.int64)


def uniform_graph(rng, query_features: int, key_features: int, nnz: int,
                  min_in_degree: int = 1, self_loops: bool = True):
    """One uniform source per target (when min_in_degree >= 1), then uniform
    (source, target) pairs with duplicates rejected until nnz pairs exist."""
    L, S = query_features, key_features
    if nnz > L * S:
        raise ValueError("more edges than pairs")
    keys = set()
    if min_in_degree >= 1:
        for t in range(L):
            while True:
                s = int(rng.integers(0, S))
                if self_loops or s != t:
                    break
            keys.add(t * S + s)
    while len(keys) < nnz:
        need = nnz - len(keys)
        ts = rng.integers(0, L, size=2 * need + 8)
        ss = rng.integers(0, S, size=2 * need + 8)
        for t, s in zip(ts.tolist(), ss.tolist()):
            if not self_loops and s == t:
                continue
            if len(keys) >= nnz:
                break
            keys.add(t * S + s)
    k = np.fromiter(keys, dtype=np.int64, count=len(keys))
    k.sort()
    return shuffle_edges(rng, k % S, k // S)


def regulator_graph(rng, n: int, nnz: int, regulator_frac: float = 0.1, zipf_s: float = 1.5):
    """Gene-regulatory prior: a seeded 10 % of the nodes act as regulators; a
    regulator of rank r is drawn with probability proportional to r^-zipf_s.
    Every target first gets one edge from a Zipf-drawn regulator, then (Zipf
    regulator, uniform target) pairs are added with duplicates rejected until
    nnz; a regulator whose fan-out reached n is dropped from the draw."""
    n_reg = max(1, int(round(regulator_frac * n)))
    regs = rng.choice(n, size=n_reg, replace=False)
    pw = np.arange(1, n_reg + 1, dtype=np.float64) ** (-zipf_s)
    out_deg = np.zeros(n_reg, np.int64)
    keys = set()
    first = rng.choice(n_reg, size=n, p=pw / pw.sum())
    for t in range(n):
        r = int(first[t])
        keys.add(t * n + int(regs[r]))
        out_deg[r] += 1
    while len(keys) < nnz:
        live = out_deg < n
        p = np.where(live, pw, 0.0)
        p /= p.sum()
        batch = max(1024, nnz - len(keys))
        rs = rng.choice(n_reg, size=batch, p=p)
        ts = rng.integers(0, n, size=batch)
        for r, t in zip(rs.tolist(), ts.tolist()):
            if len(keys) >= nnz:
                break
            if out_deg[r] >= n:
                continue
            key = t * n + int(regs[r])
            if key in keys:
                continue
            keys.add(key)
            out_deg[r] += 1
    k = np.fromiter(keys, dtype=np.int64, count=len(keys))
    k.sort()
    return shuffle_edges(rng, k % n, k // n)


def _powerlaw_exponent_for_mean(kmin: int, kmax: int, mean: float) -> float:
    k = np.arange(kmin, kmax + 1, dtype=np.float64)
    lo, hi = 1.0001, 4.0
    for _ in range(200):
        g = 0.5 * (lo + hi)
        w = k ** (-g)
        m = float((k * w).sum() / w.sum())
        if m > mean:
            lo = g
        else:
            hi = g
    return 0.5 * (lo + hi)


def powerlaw_indegree_graph(rng, n: int, nnz: int, kmax: int = 8000, kmin: int = 1):
    """Skewed in-degrees: iid draws from a discrete power law on [kmin, kmax]
    whose exponent gives mean nnz / n; the largest draw is set to kmax, then
    random nodes are moved by +-1 (staying in [kmin, kmax]) until the degrees
    sum to nnz. Each target's sources are uniform without replacement."""
    mean = nnz / n
    gamma = _powerlaw_exponent_for_mean(kmin, kmax, mean)
    k = np.arange(kmin, kmax + 1, dtype=np.float64)
    p = k ** (-gamma)
    p /= p.sum()
    deg = rng.choice(np.arange(kmin, kmax + 1), size=n, p=p).astype(np.int64)
    top = int(np.argmax(deg))
    deg[top] = kmax
    others = np.delete(np.arange(n), top)
    while True:
        diff = nnz - int(deg.sum())
        if diff == 0:
            break
        pick = rng.choice(others, size=min(abs(diff), len(others)), replace=False)
        if diff > 0:
            pick = pick[deg[pick] < kmax]
            deg[pick] += 1
        else:
            pick = pick[deg[pick] > kmin]
            deg[pick] -= 1
    src = np.empty(nnz, np.int64)
    tgt = np.empty(nnz, np.int64)
    o = 0
    for t in range(n):
        d = int(deg[t])
        src[o:o + d] = rng.choice(n, size=d, replace=False)
        tgt[o:o + d] = t
        o += d
    return shuffle_edges(rng, src, tgt)


def bipartite_membership_graph(rng, n_query: int, n_key: int, m_min: int, m_max: int):
    """Pathway -> gene map: query token i (a pathway) gets m ~ U{m_min..m_max}
    key tokens (genes) uniform without replacement; genes may repeat across
    pathways."""
    m = rng.integers(m_min, m_max + 1, size=n_query)
    src = np.concatenate([rng.choice(n_key, size=int(mi), replace=False) for mi in m])
    tgt = np.repeat(np.arange(n_query, dtype=np.int64), m)
    return shuffle_edges(rng, src.astype(np.int64), tgt)


def complete_graph(rng, n: int):
    """Every ordered pair (s, t), self-loops included, in shuffled order."""
    t, s = np.divmod(np.arange(n * n, dtype=np.int64), n)
    return shuffle_edges(rng, s, t)


def make_graph(workload_id: int):
    """(source_index, target_index) of a named workload."""
    w = workload(workload_id)
    rng = rng_for(w.id, 0)
    if w.id == 1:
        return uniform_graph(rng, w.query_features, w.key_features, w.nnz_hint)
    if w.id == 2:
        return regulator_graph(rng, w.query_features, w.nnz_hint)
    if w.id == 3:
        return powerlaw_indegree_graph(rng, w.query_features, w.nnz_hint, kmax=8000)
    if w.id == 4:
        return bipartite_membership_graph(rng, w.query_features, w.key_features, 50, 500)
    if w.id == 5:
        return complete_graph(rng, w.query_features)
    raise KeyError(workload_id)


def make_inputs(workload_id: int, batch: int | None = None):
    """Tokens and parameters of a named workload: (query, key_value, params).

    key_value is None for attention within one graph (query = key = value)."""
    w = workload(workload_id)
    B = w.batch if batch is None else batch
    params = make_params(rng_for(w.id, 1), w.embed_dim, w.dtype)
    rng = rng_for(w.id, 2)
    xq = make_tokens(rng, B, w.query_features, w.embed_dim, w.dtype)
    xkv = make_tokens(rng, B, w.key_features, w.embed_dim, w.dtype) if w.bipartite else None
    return xq, xkv, params
