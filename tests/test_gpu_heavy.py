"""GPU parity of the tensor-core path for heavy targets (targets with many
incoming edges) against the fp64 oracle, element by element: in-degrees at
and around the 128-edge tile size, ragged last tiles, several head counts,
no bias, bipartite maps, targets without edges beside heavy ones; the split
the build reports; agreement with the same graph built without a split; and
bitwise repeatability (the path has no atomics)."""
import os

import numpy as np
import pytest

from tests._cases import Case, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THRESHOLD = 32  # split degree these tests build with (the library default is no split)


def degree_graph(rng, L, S, degrees):
    """Target t gets degrees[t] distinct uniform sources; edges shuffled."""
    src, tgt = [], []
    for t, k in enumerate(degrees):
        if k:
            src.append(rng.choice(S, size=int(k), replace=False))
            tgt.append(np.full(int(k), t))
    src = np.concatenate(src).astype(np.int64)
    tgt = np.concatenate(tgt).astype(np.int64)
    perm = rng.permutation(len(src))
    return src[perm], tgt[perm]


def mixed_degrees(rng, L, heavy):
    d = rng.integers(0, 9, size=L)  # light targets, some without edges
    d[: len(heavy)] = heavy
    return rng.permutation(d)


def build(c, min_degree=THRESHOLD):
    """Build c's graph with the split threshold set (restored afterwards)."""
    import graph_sparse_head_gb300 as pmha
    old = os.environ.get("PMHA_HEAVY_MIN_DEGREE")
    os.environ["PMHA_HEAVY_MIN_DEGREE"] = str(min_degree)
    try:
        return pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), c.L, c.S)
    finally:
        if old is None:
            del os.environ["PMHA_HEAVY_MIN_DEGREE"]
        else:
            os.environ["PMHA_HEAVY_MIN_DEGREE"] = old


HEAVY = [32, 33, 127, 128, 129, 255, 256, 257, 500, 1000, 1999]


@pytest.mark.parametrize("H,B", [(8, 3), (4, 2), (2, 1), (1, 2)])
def test_heavy_targets_match_oracle(H, B):
    rng = np.random.default_rng(100 + H)
    L = S = 2000
    src, tgt = degree_graph(rng, L, S, mixed_degrees(rng, L, HEAVY))
    c = Case(src, tgt, L, S, 128, H, B, "bf16", seed=H)
    import graph_sparse_head_gb300 as pmha
    g = build(c)
    info = pmha.pmha_graph_split_info(g)
    deg = np.bincount(c.tgt, minlength=L)
    assert info["n_heavy"] == int((deg >= THRESHOLD).sum()) == len(HEAVY)
    assert info["heavy_min_degree"] == THRESHOLD
    assert info["light_nnz"] == int(deg[deg < THRESHOLD].sum())
    _, _, out, _ = c.run(DEV, "none", graph=g)
    ref, _ = c.oracle(need_weights=False)
    assert_close(f"H={H} output", out.float().cpu().numpy(), ref, "bf16")
    # bitwise repeatable
    _, _, out2, _ = c.run(DEV, "none", graph=g)
    assert torch.equal(out, out2)
    g.destroy()


def test_heavy_no_bias_and_all_targets_heavy_but_one():
    rng = np.random.default_rng(7)
    L = S = 3000  # sparse enough (7 % of the pairs) to stay off the dense path
    degs = rng.integers(THRESHOLD, 400, size=L)
    degs[5] = 3  # one light target keeps the split
    src, tgt = degree_graph(rng, L, S, degs)
    c = Case(src, tgt, L, S, 128, 8, 2, "bf16", seed=8, bias=False)
    import graph_sparse_head_gb300 as pmha
    g = build(c)
    assert pmha.pmha_graph_split_info(g)["n_heavy"] == L - 1
    _, _, out, _ = c.run(DEV, "none", graph=g)
    ref, _ = c.oracle(need_weights=False)
    assert_close("no-bias output", out.float().cpu().numpy(), ref, "bf16")
    g.destroy()


def test_heavy_bipartite_key_is_value():
    rng = np.random.default_rng(11)
    L, S = 60, 3000
    degs = rng.integers(20, 700, size=L)
    degs[:3] = [1, 5, THRESHOLD - 1]  # light targets beside the heavy ones
    src, tgt = degree_graph(rng, L, S, degs)
    c = Case(src, tgt, L, S, 128, 8, 3, "bf16", seed=12, bipartite=True)
    import graph_sparse_head_gb300 as pmha
    g = build(c)
    assert pmha.pmha_graph_split_info(g)["n_heavy"] > 0
    _, _, out, _ = c.run(DEV, "none", graph=g)
    ref, _ = c.oracle(need_weights=False)
    assert_close("bipartite output", out.float().cpu().numpy(), ref, "bf16")
    g.destroy()


def test_split_and_unsplit_graphs_agree():
    rng = np.random.default_rng(21)
    L = S = 3000
    src, tgt = degree_graph(rng, L, S, mixed_degrees(rng, L, HEAVY + [2999, 64, 65]))
    c = Case(src, tgt, L, S, 128, 8, 2, "bf16", seed=22)
    import graph_sparse_head_gb300 as pmha
    g_split, g_plain = build(c), build(c, min_degree=0)
    assert pmha.pmha_graph_split_info(g_split)["n_heavy"] > 0
    assert pmha.pmha_graph_split_info(g_plain)["n_heavy"] == 0
    _, _, out_s, _ = c.run(DEV, "none", graph=g_split)
    _, _, out_p, _ = c.run(DEV, "none", graph=g_plain)
    ref, _ = c.oracle(need_weights=False)
    assert_close("split output", out_s.float().cpu().numpy(), ref, "bf16")
    assert_close("unsplit output", out_p.float().cpu().numpy(), ref, "bf16")
    # weights requested: the split graph takes the per-edge path for every target
    _, _, out_w, w = c.run(DEV, "per_head", graph=g_split)
    _, _, out_pw, w_p = c.run(DEV, "per_head", graph=g_plain)
    assert torch.equal(out_w, out_pw) and torch.equal(w, w_p)
    g_split.destroy()
    g_plain.destroy()


def test_default_build_does_not_split():
    rng = np.random.default_rng(5)
    L = S = 500
    src, tgt = degree_graph(rng, L, S, mixed_degrees(rng, L, HEAVY[:4]))
    c = Case(src, tgt, L, S, 128, 8, 1, "bf16", seed=6)
    import graph_sparse_head_gb300 as pmha
    old = os.environ.pop("PMHA_HEAVY_MIN_DEGREE", None)
    try:
        g = pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), L, S)
    finally:
        if old is not None:
            os.environ["PMHA_HEAVY_MIN_DEGREE"] = old
    info = pmha.pmha_graph_split_info(g)
    assert info["n_heavy"] == 0 and info["heavy_min_degree"] == 0 and info["light_nnz"] == len(c.src)
    g.destroy()


def test_skewed_workload_full_size_matches_oracle():
    c = Case.workload(3)  # B = 16, n = 20,000, 400,000 edges: every output element
    import graph_sparse_head_gb300 as pmha
    g = build(c)
    assert pmha.pmha_graph_split_info(g)["n_heavy"] == int((np.bincount(c.tgt) >= THRESHOLD).sum())
    _, _, out, _ = c.run(DEV, "none", graph=g)
    ref, _ = c.oracle(need_weights=False)
    assert_close("workload 3 output (split at 32)", out.float().cpu().numpy(), ref, "bf16")
    g.destroy()


def test_split_graph_with_padding_mask_takes_the_per_edge_path():
    # a key_padding_mask keeps every target on the per-edge kernel: same result as the unsplit graph
    rng = np.random.default_rng(31)
    L = S = 2000
    src, tgt = degree_graph(rng, L, S, mixed_degrees(rng, L, HEAVY))
    c = Case(src, tgt, L, S, 128, 8, 2, "bf16", seed=32)
    import synth
    kpm = synth.padding_mask(rng, c.B, S)
    g_split, g_plain = build(c), build(c, min_degree=0)
    _, _, out_s, _ = c.run(DEV, "none", graph=g_split, kpm=kpm)
    _, _, out_p, _ = c.run(DEV, "none", graph=g_plain, kpm=kpm)
    assert torch.equal(out_s, out_p)
    ref, _ = c.oracle(need_weights=False, kpm=kpm)
    assert_close("masked output", out_s.float().cpu().numpy(), ref, "bf16")
    g_split.destroy()
    g_plain.destroy()


def test_split_graph_backward_equals_unsplit():
    # the backward recomputes the forward on the whole graph, split or not
    import graph_sparse_head_gb300 as pmha
    rng = np.random.default_rng(41)
    L = S = 1500
    src, tgt = degree_graph(rng, L, S, mixed_degrees(rng, L, HEAVY[:8]))
    c = Case(src, tgt, L, S, 128, 8, 2, "bf16", seed=42)
    params = pmha.Params.from_arrays(c.params, c.H, torch.bfloat16, DEV)
    xq, xkv = c.device_inputs(DEV)
    dout = torch.from_numpy(rng.standard_normal(xq.shape).astype(np.float32)).to(DEV).to(torch.bfloat16)
    grads = []
    for g in (build(c), build(c, min_degree=0)):
        r = pmha.pmha_backward(g, params, xq, xkv, xkv, dout)
        pmha.pmha_device_status()
        grads.append({k: v.clone() for k, v in r.items() if v is not None})
        g.destroy()
    assert grads[0].keys() == grads[1].keys()
    for k in grads[0]:
        assert torch.equal(grads[0][k], grads[1][k]), k
