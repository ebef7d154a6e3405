"""The seeded synthetic workloads hold the shapes their recipe states: edge
counts, no duplicate pairs, every target with a source, the degree
distributions (regulator fan-out, Zipf-like in-degrees up to 8,000, pathway
sizes 50-500, the complete graph), the parameter and token ranges, exact
storage rounding and determinism."""
import numpy as np
import pytest

import synth


def _pairs(src, tgt, S):
    k = tgt.astype(np.int64) * S + src
    return np.unique(k).size == k.size


@pytest.fixture(scope="module")
def graphs():
    return {i: synth.make_graph(i) for i in synth.WORKLOADS}


@pytest.mark.parametrize("wid", sorted(synth.WORKLOADS))
def test_graph_shape_common(graphs, wid):
    w = synth.workload(wid)
    src, tgt = graphs[wid]
    assert src.dtype == np.int64 and tgt.dtype == np.int64 and src.shape == tgt.shape
    assert src.min() >= 0 and src.max() < w.key_features
    assert tgt.min() >= 0 and tgt.max() < w.query_features
    assert _pairs(src, tgt, w.key_features)                       # no duplicate (source, target)
    assert np.bincount(tgt, minlength=w.query_features).min() >= 1  # every target has a source
    assert not np.all(np.diff(tgt) >= 0)                          # given in shuffled order, not sorted


def test_exact_edge_counts(graphs):
    for wid in (1, 2, 3):
        assert graphs[wid][0].size == synth.workload(wid).nnz_hint
    assert graphs[5][0].size == 1024 * 1024


def test_regulator_fan_out(graphs):
    src, tgt = graphs[2]
    regs = np.unique(src)
    assert regs.size <= 200  # 10 % of 2,000 nodes act as regulators
    fan = np.bincount(src, minlength=2000)[regs]
    assert fan.max() >= 10 * fan.mean()  # Zipf(1.5) over regulator rank: a few hubs
    assert np.bincount(tgt, minlength=2000).mean() == 20.0


def test_skewed_in_degrees(graphs):
    src, tgt = graphs[3]
    deg = np.bincount(tgt, minlength=20_000)
    assert deg.min() >= 1 and deg.max() == 8000 and deg.mean() == 20.0
    assert np.median(deg) <= 5  # most targets have a handful of edges, a few have thousands


def test_pathway_sizes(graphs):
    src, tgt = graphs[4]
    m = np.bincount(tgt, minlength=500)
    assert m.min() >= 50 and m.max() <= 500
    assert abs(src.size - 137_500) < 0.1 * 137_500
    assert np.bincount(src, minlength=20_000).max() > 1  # genes shared by several pathways


def test_complete_graph_has_every_pair(graphs):
    src, tgt = graphs[5]
    assert np.array_equal(np.sort(tgt * 1024 + src), np.arange(1024 * 1024))


def test_determinism():
    a = synth.make_graph(1)
    b = synth.make_graph(1)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    xa, _, pa = synth.make_inputs(2, batch=2)
    xb, _, pb = synth.make_inputs(2, batch=2)
    assert np.array_equal(xa, xb) and all(np.array_equal(pa[k], pb[k]) for k in pa)


@pytest.mark.parametrize("wid", sorted(synth.WORKLOADS))
def test_inputs_shapes_ranges_and_rounding(wid):
    w = synth.workload(wid)
    xq, xkv, p = synth.make_inputs(wid, batch=2)
    E = w.embed_dim
    assert xq.shape == (2, w.query_features, E) and xq.dtype == np.float32
    assert (xkv is not None) == w.bipartite
    if xkv is not None:
        assert xkv.shape == (2, w.key_features, E)
    bound = np.sqrt(6.0 / (2 * E))
    for n in ("wq", "wk", "wv", "wo"):
        assert p[n].shape == (E, E) and np.abs(p[n]).max() <= bound * (1 + 2 ** -8)
    for n in ("bq", "bk", "bv", "bo"):
        assert p[n].shape == (E,) and np.abs(p[n]).max() <= 0.1 * (1 + 2 ** -8)
    assert abs(float(xq.std()) - 1.0) < 0.05
    if w.dtype == "bf16":  # stored values are bfloat16 numbers: the low 16 bits are zero
        for a in (xq, p["wq"], p["bo"]):
            assert not np.any(a.view(np.uint32) & np.uint32(0xFFFF))


def test_bf16_round_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -9], np.float32)
    got = synth.bf16_round(x)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even (1.0); 1 + 3*2^-8 to 1 + 2^-6
    assert np.array_equal(got, np.array([1.0, 1.0, 1.0 + 2 ** -6, -1.0, 1.0], np.float32))
