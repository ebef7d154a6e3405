"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

* the kpnn2 PackedMultiheadAttention doctest (edge order, self-loop append,
  shapes; a node with no source outputs the out_proj bias),
* torch.nn.MultiheadAttention in float64 on a complete graph (the dense limit:
  continuiti's MultiHead formula and the tutorial's in_proj slicing),
* the same library routine with an additive -inf mask built from the graph
  (the kpnn2 page: masking nn.MultiheadAttention computes the same mix for
  every node that has a source),
* softmax invariants (non-negative, sums to 1, a single source gets exactly 1),
* invariance to edge order, and brute-force loops for the index work.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _golden


def _params(rng, E, bias=True):
    return synth.make_params(rng, E, "f32", bias=bias)


def _torch_mha(params, E, H):
    mha = torch.nn.MultiheadAttention(E, H, batch_first=True, bias=True, dtype=torch.float64)
    with torch.no_grad():
        mha.in_proj_weight.copy_(torch.from_numpy(
            np.concatenate([params["wq"], params["wk"], params["wv"]]).astype(np.float64)))
        zeros = np.zeros(E)
        bq, bk, bv, bo = (params[n] if params[n] is not None else zeros for n in ("bq", "bk", "bv", "bo"))
        mha.in_proj_bias.copy_(torch.from_numpy(np.concatenate([bq, bk, bv]).astype(np.float64)))
        mha.out_proj.weight.copy_(torch.from_numpy(params["wo"].astype(np.float64)))
        mha.out_proj.bias.copy_(torch.from_numpy(np.asarray(bo, np.float64)))
    mha.eval()
    return mha


def _dense(params, xq, xkv, H, mask=None, average=False):
    E = xq.shape[-1]
    mha = _torch_mha(params, E, H)
    q = torch.from_numpy(xq.astype(np.float64))
    kv = torch.from_numpy(xkv.astype(np.float64))
    with torch.no_grad():
        out, w = mha(q, kv, kv, need_weights=True, attn_mask=mask, average_attn_weights=average)
    return out.numpy(), w.numpy()


# ---------------------------------------------------------------- doctest pins

def test_doctest_edge_order_and_self_loops():
    g = _golden.load("kpnn2_doctest.txt")
    idx = {n: i for i, n in enumerate(g["nodes"].split())}
    src = [idx[n] for n in g["given_source"].split()]
    tgt = [idx[n] for n in g["given_target"].split()]
    s2, t2 = oracle.append_self_loops(src, tgt, len(idx))
    assert [int(x) for x in s2] == [idx[n] for n in g["self_loop_source"].split()]
    assert [int(x) for x in t2] == [idx[n] for n in g["self_loop_target"].split()]
    assert len(s2) == int(g["nnz_with_loops"])
    # an existing self-loop is kept, not duplicated
    s3, t3 = oracle.append_self_loops([1, 0], [1, 2], 3)
    assert list(zip(s3.tolist(), t3.tolist())) == [(1, 1), (0, 2), (0, 0), (2, 2)]


def test_doctest_shapes_weights_and_isolated_node():
    g = _golden.load("kpnn2_doctest.txt")
    idx = {n: i for i, n in enumerate(g["nodes"].split())}
    src = [idx[n] for n in g["given_source"].split()]
    tgt = [idx[n] for n in g["given_target"].split()]
    E, H, B = int(g["embed_dim"]), int(g["num_heads"]), int(g["batch"])
    assert E // H == int(g["head_dim"])
    rng = np.random.default_rng(7)
    p = _params(rng, E)
    x = rng.standard_normal((B, len(idx), E))
    s2, t2 = oracle.append_self_loops(src, tgt, len(idx))
    out, w = oracle.forward(x, x, x, p, s2, t2, H)
    assert out.shape == tuple(_golden.ints(g["output_shape"]))
    assert oracle.average_heads(w).shape == tuple(_golden.ints(g["packed_weights_shape"]))
    # without self-loops: node x has no source, mixes to zeros, outputs out_proj's bias
    L, S, nnz = _golden.ints(g["no_loops_sizes"])
    assert (L, S, nnz) == (len(idx), len(idx), len(src))
    out0, w0 = oracle.forward(x, x, x, p, src, tgt, H)
    for b in range(B):
        assert np.array_equal(out0[b, idx["x"]], p["bo"].astype(np.float64))
    # with a self-loop as its only key, x passes on its own value: weight exactly 1
    x_loop = [e for e in range(len(s2)) if s2[e] == idx["x"] and t2[e] == idx["x"]][0]
    assert np.all(w[:, x_loop, :] == 1.0)
    v = oracle.linear(x, p["wv"], p["bv"])
    ref = oracle.linear(v[:, idx["x"]], p["wo"], p["bo"])
    assert np.allclose(out[:, idx["x"]], ref, rtol=0, atol=1e-14)


# ---------------------------------------------------------- dense-limit pins

@pytest.mark.parametrize("E,H,n,B", [(16, 4, 5, 2), (32, 4, 7, 3), (24, 3, 4, 1)])
def test_complete_graph_equals_torch_mha(E, H, n, B):
    rng = np.random.default_rng(E * 100 + n)
    p = _params(rng, E)
    x = rng.standard_normal((B, n, E))
    src, tgt = synth.complete_graph(rng, n)
    out, w = oracle.forward(x, x, x, p, src, tgt, H)
    ref_out, ref_w = _dense(p, x, x, H, average=False)  # (B, H, L, S)
    assert np.abs(out - ref_out).max() < 1e-12
    assert np.abs(w - ref_w[:, :, tgt, src].transpose(0, 2, 1)).max() < 1e-14
    _, ref_avg = _dense(p, x, x, H, average=True)      # (B, L, S)
    assert np.abs(oracle.average_heads(w) - ref_avg[:, tgt, src]).max() < 1e-14


def test_bias_false_equals_torch_mha_without_bias():
    rng = np.random.default_rng(3)
    E, H, n = 16, 2, 6
    p = _params(rng, E, bias=False)
    x = rng.standard_normal((2, n, E))
    src, tgt = synth.complete_graph(rng, n)
    out, _ = oracle.forward(x, x, x, p, src, tgt, H)
    ref_out, _ = _dense(p, x, x, H)
    assert np.abs(out - ref_out).max() < 1e-12


def test_tutorial_in_proj_slicing_example():
    """The tutorial's E=8, H=2, seq=3 example: the module, its by-hand slicing of
    in_proj_weight into thirds, and the oracle on the complete 3-node graph agree."""
    g = _golden.load("torch_mha_tutorial.txt")
    E, H, n = int(g["embed_dim"]), int(g["num_heads"]), int(g["seq"])
    torch.manual_seed(int(g["seed"]))
    module = torch.nn.MultiheadAttention(embed_dim=E, num_heads=H, batch_first=True)
    x = torch.randn(1, n, E)
    assert tuple(module.in_proj_weight.shape) == tuple(_golden.ints(g["packed_shape"]))
    with torch.no_grad():
        m_out, m_w = module(x, x, x)
    assert tuple(m_out.shape) == tuple(_golden.ints(g["module_output_shape"]))
    assert tuple(m_w.shape) == tuple(_golden.ints(g["averaged_weights_shape"]))
    r = int(g["slice_rows"])
    W = module.in_proj_weight.detach().double().numpy()
    b = module.in_proj_bias.detach().double().numpy()
    p = {"wq": W[:r], "wk": W[r:2 * r], "wv": W[2 * r:], "bq": b[:r], "bk": b[r:2 * r],
         "bv": b[2 * r:], "wo": module.out_proj.weight.detach().double().numpy(),
         "bo": module.out_proj.bias.detach().double().numpy()}
    xs = x.double().numpy()
    src, tgt = synth.complete_graph(np.random.default_rng(0), n)
    out, w = oracle.forward(xs, xs, xs, p, src, tgt, H)
    # float64 module on the same parameters: agreement to rounding
    module64 = module.double()
    with torch.no_grad():
        o64, w64 = module64(x.double(), x.double(), x.double())
    assert np.abs(out - o64.numpy()).max() < 1e-13
    assert np.abs(oracle.average_heads(w) - w64.numpy()[:, tgt, src]).max() < 1e-14
    # the page's own check, at its tolerance, against the float32 module output
    assert np.allclose(out, m_out.double().numpy(), atol=float(g["allclose_atol"]))


# ------------------------------------------------------------ masked-dense pins

@pytest.mark.parametrize("L,S,nnz,E,H,B", [(64, 64, 256, 32, 4, 2), (9, 13, 40, 16, 2, 3),
                                           (20, 6, 50, 8, 1, 1)])
def test_sparse_equals_masked_dense(L, S, nnz, E, H, B):
    rng = np.random.default_rng(L * S + nnz)
    p = _params(rng, E)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E)) if L != S else xq
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=0)
    mask = np.full((L, S), -np.inf)
    mask[tgt, src] = 0.0
    out, w = oracle.forward(xq, xkv, xkv, p, src, tgt, H)
    ref_out, ref_w = _dense(p, xq, xkv, H, mask=torch.from_numpy(mask))
    has_src = np.bincount(tgt, minlength=L) > 0
    assert np.abs(out[:, has_src] - ref_out[:, has_src]).max() < 1e-12
    assert np.abs(w - ref_w[:, :, tgt, src].transpose(0, 2, 1)).max() < 1e-13
    # a target without a source: zeros before out_proj, so exactly the bias
    for t in np.nonzero(~has_src)[0]:
        assert np.array_equal(out[:, t], np.broadcast_to(p["bo"], out[:, t].shape))


# --------------------------------------------------------- softmax invariants

def test_weights_nonnegative_sum_to_one_and_single_source_exact():
    rng = np.random.default_rng(11)
    L = S = 40
    E, H, B = 16, 4, 2
    p = _params(rng, E)
    x = rng.standard_normal((B, L, E))
    src, tgt = synth.uniform_graph(rng, L, S, 70, min_in_degree=1)
    out, w = oracle.forward(x, x, x, p, src, tgt, H)
    assert (w >= 0).all()
    sums = np.zeros((B, L, H))
    for e in range(len(src)):
        sums[:, tgt[e], :] += w[:, e, :]
    assert np.abs(sums - 1.0).max() < 1e-12
    deg = np.bincount(tgt, minlength=L)
    v = oracle.linear(x, p["wv"], p["bv"])
    single = np.nonzero(deg == 1)[0]
    assert len(single) > 0
    for t in single:
        e = int(np.nonzero(tgt == t)[0][0])
        assert np.all(w[:, e, :] == 1.0)
        ref = oracle.linear(v[:, src[e]], p["wo"], p["bo"])
        assert np.abs(out[:, t] - ref).max() < 1e-14


def test_edge_order_invariance():
    rng = np.random.default_rng(5)
    L, S, E, H, B = 30, 30, 16, 2, 2
    p = _params(rng, E)
    x = rng.standard_normal((B, L, E))
    src, tgt = synth.uniform_graph(rng, L, S, 120)
    out, w = oracle.forward(x, x, x, p, src, tgt, H)
    perm = rng.permutation(len(src))
    out2, w2 = oracle.forward(x, x, x, p, src[perm], tgt[perm], H)
    assert np.abs(out - out2).max() < 1e-13
    assert np.abs(w[:, perm] - w2).max() < 1e-15


def test_forward_rows_matches_full_forward():
    rng = np.random.default_rng(9)
    L, S, E, H, B = 12, 17, 16, 4, 3
    p = _params(rng, E)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    src, tgt = synth.uniform_graph(rng, L, S, 60, min_in_degree=0)
    out, w = oracle.forward(xq, xkv, xkv, p, src, tgt, H)
    rows = [(b, t) for b in range(B) for t in range(L)]
    for (b, t), (o, e_ids, we) in zip(rows, oracle.forward_rows(xq, xkv, xkv, p, src, tgt, H, rows)):
        assert np.abs(o - out[b, t]).max() < 1e-13
        assert np.abs(we - w[b, e_ids]).max() < 1e-15


def test_key_bias_does_not_change_the_layer():
    # q_t . (k_s + c) = q_t . k_s + q_t . c: the key bias adds the same amount
    # to every score of one (target, head), and a softmax over that target's
    # edges does not see it. Any bk gives the same weights and output.
    rng = np.random.default_rng(21)
    L, S, E, H, B = 25, 33, 16, 4, 2
    p = _params(rng, E)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    src, tgt = synth.uniform_graph(rng, L, S, 110, min_in_degree=0)
    out, w = oracle.forward(xq, xkv, xkv, p, src, tgt, H)
    p2 = dict(p)
    p2["bk"] = p["bk"] + 3.0 * rng.standard_normal(E)
    out2, w2 = oracle.forward(xq, xkv, xkv, p2, src, tgt, H)
    assert np.abs(w - w2).max() < 1e-12
    assert np.abs(out - out2).max() < 1e-12
    # the query bias is not so: it changes the scores edge by edge
    p3 = dict(p)
    p3["bq"] = p["bq"] + 3.0 * rng.standard_normal(E)
    _, w3 = oracle.forward(xq, xkv, xkv, p3, src, tgt, H)
    assert np.abs(w - w3).max() > 1e-3


def test_value_path_is_affine():
    # With the keys fixed the weights are fixed and sum to 1 over a target's
    # edges, so out = Wo (Wv sum_e w_e x_s + bv) + bo is affine in the value
    # tokens: out(v1 + v2) = out(v1) + out(v2) - (Wo bv + bo) for a target with
    # a source; a target without one outputs bo whatever the values.
    rng = np.random.default_rng(23)
    L, S, E, H, B = 20, 28, 16, 2, 2
    p = _params(rng, E)
    xq = rng.standard_normal((B, L, E))
    xk = rng.standard_normal((B, S, E))
    v1 = rng.standard_normal((B, S, E))
    v2 = rng.standard_normal((B, S, E))
    src, tgt = synth.uniform_graph(rng, L, S, 70, min_in_degree=0)
    o1, w1 = oracle.forward(xq, xk, v1, p, src, tgt, H)
    o2, _ = oracle.forward(xq, xk, v2, p, src, tgt, H)
    o12, w12 = oracle.forward(xq, xk, v1 + v2, p, src, tgt, H)
    assert np.abs(w1 - w12).max() == 0.0  # the weights do not read the values
    deg = np.bincount(tgt, minlength=L)
    assert (deg == 0).any() and (deg > 0).any()
    const = p["wo"].astype(np.float64) @ p["bv"].astype(np.float64) + p["bo"]
    live = deg > 0
    assert np.abs(o12[:, live] - (o1[:, live] + o2[:, live] - const)).max() < 1e-12
    assert np.abs(o12[:, ~live] - p["bo"]).max() == 0.0


def test_node_relabelling_permutes_the_output():
    # Renaming the targets by a permutation pt and the sources by ps (graph
    # and tokens alike) permutes the output rows by pt and leaves each edge's
    # weights unchanged.
    rng = np.random.default_rng(25)
    L, S, E, H, B = 18, 26, 16, 4, 2
    p = _params(rng, E)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    src, tgt = synth.uniform_graph(rng, L, S, 80, min_in_degree=0)
    out, w = oracle.forward(xq, xkv, xkv, p, src, tgt, H)
    pt, ps = rng.permutation(L), rng.permutation(S)  # node t is called pt[t]
    xq2 = np.empty_like(xq)
    xq2[:, pt] = xq
    xkv2 = np.empty_like(xkv)
    xkv2[:, ps] = xkv
    out2, w2 = oracle.forward(xq2, xkv2, xkv2, p, ps[src], pt[tgt], H)
    assert np.abs(out2[:, pt] - out).max() < 1e-13
    assert np.abs(w2 - w).max() < 1e-15


# ------------------------------------------------------------ index work pins

def test_validation_codes():
    assert oracle.validate_edges([], [], 3, 3) == oracle.ERR_EMPTY
    assert oracle.validate_edges([0, 3], [0, 1], 3, 3) == oracle.ERR_RANGE
    assert oracle.validate_edges([0, 1], [0, 4], 3, 5) == oracle.ERR_RANGE
    assert oracle.validate_edges([-1], [0], 3, 3) == oracle.ERR_RANGE
    assert oracle.validate_edges([0, 1, 0], [2, 2, 2], 3, 3) == oracle.ERR_DUPLICATE
    assert oracle.validate_edges([0, 1, 2], [2, 2, 2], 3, 3) == oracle.OK
    assert oracle.validate_edges([4], [0], 1, 5) == oracle.OK
    assert oracle.validate_edges([0], [0], 0, 5) == oracle.ERR_ARG


@pytest.mark.parametrize("L,S,nnz,seed", [(1, 1, 1, 0), (5, 7, 20, 1), (33, 9, 150, 2), (64, 64, 600, 3)])
def test_csr_bruteforce(L, S, nnz, seed):
    rng = np.random.default_rng(seed)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=0)
    row_ptr, col, perm = oracle.csr_by_target(src, tgt, L)
    # brute force with plain loops: for t ascending, the sources into t ascending
    i = 0
    for t in range(L):
        assert row_ptr[t] == i
        srcs = sorted((int(src[e]), e) for e in range(nnz) if tgt[e] == t)
        for s, e in srcs:
            assert col[i] == s and perm[i] == e
            i += 1
    assert row_ptr[L] == nnz == i
    assert sorted(perm.tolist()) == list(range(nnz))


def test_self_loops_bruteforce():
    rng = np.random.default_rng(4)
    for n, nnz in [(1, 1), (6, 10), (25, 80)]:
        src, tgt = synth.uniform_graph(rng, n, n, nnz, min_in_degree=0)
        s2, t2 = oracle.append_self_loops(src, tgt, n)
        have = {(int(a), int(b)) for a, b in zip(src, tgt)}
        missing = [i for i in range(n) if (i, i) not in have]
        assert s2[:nnz].tolist() == src.tolist() and t2[:nnz].tolist() == tgt.tolist()
        assert s2[nnz:].tolist() == missing and t2[nnz:].tolist() == missing


def test_linear_matches_numpy_matmul():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 6, 10))
    w = rng.standard_normal((7, 10))
    b = rng.standard_normal(7)
    assert np.abs(oracle.linear(x, w, b) - (x @ w.T + b)).max() < 1e-13
    assert np.abs(oracle.linear(x, w) - x @ w.T).max() < 1e-13


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(2)
    L, E, H = 50, 16, 4
    p = _params(rng, E)
    x = rng.standard_normal((3, L, E))
    src, tgt = synth.uniform_graph(rng, L, L, 300)
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a, wa = oracle.forward(x, x, x, p, src, tgt, H)
        oracle.set_num_threads(max(2, n0))
        b, wb = oracle.forward(x, x, x, p, src, tgt, H)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(a, b) and np.array_equal(wa, wb)


# ------------------------------------------------------------ key padding mask

@pytest.mark.parametrize("E,H,n,B", [(16, 4, 6, 3), (24, 2, 9, 2)])
def test_key_padding_mask_equals_torch_mha(E, H, n, B):
    """kpnn2 forward(), key_padding_mask: True drops that key's edges from the
    softmax; on the complete graph this is torch's key_padding_mask."""
    rng = np.random.default_rng(E + n)
    p = _params(rng, E)
    x = rng.standard_normal((B, n, E))
    src, tgt = synth.complete_graph(rng, n)
    kpm = rng.random((B, n)) < 0.4
    kpm[:, 0] = False  # every query keeps a live key
    out, w = oracle.forward(x, x, x, p, src, tgt, H, key_padding_mask=kpm)
    mha = _torch_mha(p, E, H)
    with torch.no_grad():
        ref, ref_w = mha(*(torch.from_numpy(x),) * 3, key_padding_mask=torch.from_numpy(kpm), need_weights=True,
                         average_attn_weights=False)
    assert np.abs(out - ref.numpy()).max() < 1e-12
    assert np.abs(w - ref_w.numpy()[:, :, tgt, src].transpose(0, 2, 1)).max() < 1e-14
    # masked keys carry weight 0, live ones sum to 1
    assert np.all(w[kpm[:, src]] == 0.0)


def test_key_padding_mask_drops_every_key_of_a_target():
    """A query whose live keys are all masked mixes to zeros: output = bo."""
    rng = np.random.default_rng(31)
    E, H, n = 16, 2, 8
    p = _params(rng, E)
    x = rng.standard_normal((2, n, E))
    src, tgt = synth.uniform_graph(rng, n, n, 30)
    kpm = np.zeros((2, n), bool)
    t0 = int(tgt[0])
    kpm[1, src[tgt == t0]] = True  # sample 1: every source of t0 masked
    out, w = oracle.forward(x, x, x, p, src, tgt, H, key_padding_mask=kpm)
    assert np.array_equal(out[1, t0], p["bo"].astype(np.float64))
    assert np.all(w[1, tgt == t0] == 0.0)
    out0, _ = oracle.forward(x, x, x, p, src, tgt, H)
    assert np.array_equal(out[0], out0[0])  # sample 0 has no masked key
