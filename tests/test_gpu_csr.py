"""GPU: the one-time per-target index build (pmha_build_csr) is bit-exact
against the oracle's CSR, rejects what the kpnn2 constructor rejects, and
does not depend on the order of the given pairs."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _build(src, tgt, L, S, loops=False):
    import graph_sparse_head_gb300 as pmha
    return pmha.pmha_build_csr(torch.as_tensor(src, dtype=torch.int64).to(DEV),
                               torch.as_tensor(tgt, dtype=torch.int64).to(DEV), L, S, loops)


def _export(g):
    import graph_sparse_head_gb300 as pmha
    r, c, p = pmha.pmha_graph_export(g)
    torch.cuda.synchronize()
    return r.cpu().numpy(), c.cpu().numpy(), p.cpu().numpy()


def _check_against_oracle(src, tgt, L, S, loops=False):
    g = _build(src, tgt, L, S, loops)
    s2, t2 = (oracle.append_self_loops(src, tgt, L) if loops else (np.asarray(src), np.asarray(tgt)))
    assert g.nnz == len(s2)
    rp, col, perm = oracle.csr_by_target(s2, t2, L)
    r, c, p = _export(g)
    assert np.array_equal(r, rp)
    assert np.array_equal(c, col)
    assert np.array_equal(p, perm)
    assert g.max_in_degree == int(np.diff(rp).max())
    return g


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_csr_bit_exact_on_workload_graphs(wid):
    w = synth.workload(wid)
    src, tgt = synth.make_graph(wid)
    _check_against_oracle(src, tgt, w.query_features, w.key_features).destroy()
    if w.query_features == w.key_features:
        _check_against_oracle(src, tgt, w.query_features, w.key_features, loops=True).destroy()


@pytest.mark.parametrize("L,S,nnz,seed", [(1, 1, 1, 0), (1, 5000, 4000, 1), (5000, 1, 3000, 2), (7, 9, 40, 3),
                                           (300, 300, 20000, 4), (4097, 3, 5000, 5), (1000, 70000, 9000, 6)])
def test_csr_ragged_and_degenerate(L, S, nnz, seed):
    rng = np.random.default_rng(seed)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=0)
    _check_against_oracle(src, tgt, L, S).destroy()
    if L == S:
        _check_against_oracle(src, tgt, L, S, loops=True).destroy()


def test_csr_split_boundaries():
    # in-degrees around the split size (128 edges per chunk): 127, 128, 129, 256, 257, 1000
    degs = [127, 128, 129, 256, 257, 1000, 0, 1]
    L, S = len(degs), 2000
    rng = np.random.default_rng(8)
    src = np.concatenate([rng.choice(S, d, replace=False) for d in degs])
    tgt = np.repeat(np.arange(L), degs)
    src, tgt = synth.shuffle_edges(rng, src, tgt)
    _check_against_oracle(src, tgt, L, S).destroy()


def test_csr_wide_keys():
    # L * S >= 2^32 takes the 64-bit key path
    L, S = 70000, 70000
    rng = np.random.default_rng(9)
    src, tgt = synth.uniform_graph(rng, L, S, 50000, min_in_degree=0)
    _check_against_oracle(src, tgt, L, S).destroy()


def test_csr_independent_of_input_order():
    rng = np.random.default_rng(10)
    src, tgt = synth.uniform_graph(rng, 500, 400, 6000)
    g1 = _build(src, tgt, 500, 400)
    p = rng.permutation(len(src))
    g2 = _build(src[p], tgt[p], 500, 400)
    r1, c1, p1 = _export(g1)
    r2, c2, p2 = _export(g2)
    assert np.array_equal(r1, r2) and np.array_equal(c1, c2)
    assert np.array_equal(p[p2], p1)  # same edge at each position
    g1.destroy()
    g2.destroy()


@pytest.mark.parametrize("src,tgt,L,S,code", [
    ([0, 1, 2], [0, 1, 3], 3, 3, "PMHA_ERR_INDEX_RANGE"),
    ([0, 3, 2], [0, 1, 2], 3, 3, "PMHA_ERR_INDEX_RANGE"),
    ([0, -1], [0, 1], 3, 3, "PMHA_ERR_INDEX_RANGE"),
    ([0, 1, 0], [2, 2, 2], 3, 3, "PMHA_ERR_DUPLICATE_EDGE"),
    ([5, 5], [0, 0], 1, 6, "PMHA_ERR_DUPLICATE_EDGE"),
])
def test_csr_rejects_bad_indices(src, tgt, L, S, code):
    import graph_sparse_head_gb300 as pmha
    with pytest.raises(pmha.PmhaError) as ei:
        _build(src, tgt, L, S)
    assert ei.value.status_name == code
    # the oracle agrees on the verdict
    assert oracle.validate_edges(src, tgt, L, S) != oracle.OK


def test_csr_rejects_empty_and_bad_loops():
    import graph_sparse_head_gb300 as pmha
    with pytest.raises(pmha.PmhaError) as ei:
        _build([], [], 3, 3)
    assert ei.value.status_name == "PMHA_ERR_EMPTY"
    with pytest.raises(pmha.PmhaError) as ei:
        _build([0], [0], 3, 4, loops=True)
    assert ei.value.status_name == "PMHA_ERR_INVALID_ARG"


def test_self_loop_with_existing_loop_kept_once():
    g = _check_against_oracle([1, 0, 2], [1, 2, 2], 3, 3, loops=True)
    assert g.nnz == 4
    g.destroy()
