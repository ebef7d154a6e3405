"""Pins of the oracle's backward pass (the chain rule of kpnn2
PackedMultiheadAttention, Notes steps 1-5), each independent of the oracle's
own arithmetic:

* torch autograd through torch.nn.MultiheadAttention in float64 on a complete
  graph (the dense limit), all input, weight and bias gradients;
* autograd through dense attention with an additive -inf mask built from a
  sparse graph (the page: masking dense attention with the graph gives the
  same mix), and through torch's key_padding_mask;
* central finite differences of sum(output * dout) on a tiny case;
* exact properties: the key-projection bias gets no gradient (the softmax of
  each target is invariant to a shift shared by its scores), a target
  with a single source passes no gradient into the scores, and a sample
  whose keys are all padding passes none into its tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


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
    return mha


def _torch_grads(params, H, xq, xk, xv, dout, attn_mask=None, key_padding_mask=None):
    """Autograd of sum(out * dout) through nn.MultiheadAttention (float64)."""
    E = xq.shape[-1]
    mha = _torch_mha(params, E, H)
    q, k, v = (torch.from_numpy(np.array(x, np.float64)).requires_grad_(True) for x in (xq, xk, xv))
    out, _ = mha(q, k, v, need_weights=False, attn_mask=attn_mask,
                 key_padding_mask=None if key_padding_mask is None else torch.from_numpy(key_padding_mask))
    (out * torch.from_numpy(dout)).sum().backward()
    W, b = mha.in_proj_weight.grad.numpy(), mha.in_proj_bias.grad.numpy()
    return {"dquery": q.grad.numpy(), "dkey": k.grad.numpy(), "dvalue": v.grad.numpy(),
            "dwq": W[:E], "dwk": W[E:2 * E], "dwv": W[2 * E:], "dbq": b[:E], "dbk": b[E:2 * E],
            "dbv": b[2 * E:], "dwo": mha.out_proj.weight.grad.numpy(), "dbo": mha.out_proj.bias.grad.numpy()}


def _assert_grads(got, ref, tol, names=None):
    for n in names or ref:
        if got[n] is None:
            continue
        err = np.abs(got[n] - ref[n]).max()
        scale = max(np.abs(ref[n]).max(), 1e-300)
        assert err <= tol * max(scale, 1.0), f"{n}: {err:.3e} (scale {scale:.3e})"


@pytest.mark.parametrize("E,H,n,B", [(16, 4, 6, 2), (24, 3, 5, 1), (8, 2, 7, 3)])
def test_complete_graph_gradients_equal_torch_autograd(E, H, n, B):
    rng = np.random.default_rng(100 + E + n)
    p = _params(rng, E)
    xq, xk, xv = (rng.standard_normal((B, n, E)) for _ in range(3))
    dout = rng.standard_normal((B, n, E))
    src, tgt = synth.complete_graph(rng, n)
    got = oracle.backward(xq, xk, xv, p, src, tgt, H, dout)
    ref = _torch_grads(p, H, xq, xk, xv, dout)
    _assert_grads(got, ref, 1e-11)


@pytest.mark.parametrize("L,S,nnz,E,H,B", [(9, 9, 30, 16, 4, 2), (6, 11, 25, 8, 2, 2), (12, 5, 40, 12, 3, 1)])
def test_sparse_gradients_equal_masked_dense_autograd(L, S, nnz, E, H, B):
    rng = np.random.default_rng(L * 7 + S)
    p = _params(rng, E)
    src, tgt = synth.uniform_graph(rng, L, S, nnz)  # every target has a source
    xq = rng.standard_normal((B, L, E))
    xk, xv = rng.standard_normal((B, S, E)), rng.standard_normal((B, S, E))
    dout = rng.standard_normal((B, L, E))
    mask = np.full((L, S), -np.inf)
    mask[tgt, src] = 0.0
    got = oracle.backward(xq, xk, xv, p, src, tgt, H, dout)
    ref = _torch_grads(p, H, xq, xk, xv, dout, attn_mask=torch.from_numpy(mask))
    _assert_grads(got, ref, 1e-11)


def test_key_padding_mask_gradients_equal_torch():
    rng = np.random.default_rng(7)
    E, H, n, B = 16, 4, 8, 3
    p = _params(rng, E)
    xq, xk, xv = (rng.standard_normal((B, n, E)) for _ in range(3))
    dout = rng.standard_normal((B, n, E))
    src, tgt = synth.complete_graph(rng, n)
    kpm = rng.random((B, n)) < 0.4
    kpm[:, 0] = False
    got = oracle.backward(xq, xk, xv, p, src, tgt, H, dout, key_padding_mask=kpm)
    ref = _torch_grads(p, H, xq, xk, xv, dout, key_padding_mask=kpm)
    _assert_grads(got, ref, 1e-11)
    # a dropped key receives nothing through attention
    assert np.all(got["dkey"][kpm] == 0.0) and np.all(got["dvalue"][kpm] == 0.0)


def test_finite_differences():
    rng = np.random.default_rng(11)
    E, H, L, S, B = 4, 2, 4, 5, 2
    p = _params(rng, E)
    src, tgt = synth.uniform_graph(rng, L, S, 11)
    xq = rng.standard_normal((B, L, E))
    xk, xv = rng.standard_normal((B, S, E)), rng.standard_normal((B, S, E))
    kpm = np.zeros((B, S), bool)
    kpm[1, 2] = True
    dout = rng.standard_normal((B, L, E))
    got = oracle.backward(xq, xk, xv, p, src, tgt, H, dout, key_padding_mask=kpm)

    def f(xq_, xk_, xv_, p_):
        out, _ = oracle.forward(xq_, xk_, xv_, p_, src, tgt, H, need_weights=False, key_padding_mask=kpm)
        return float((out * dout).sum())

    h = 1e-6
    inputs = {"dquery": xq, "dkey": xk, "dvalue": xv}
    for name, x in inputs.items():
        for idx in [(0, 0, 0), (1, 1, 3), (1, 3, 2), (0, 2, 1)]:
            if idx[1] >= x.shape[1]:
                continue
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if x is y else y for y in (xq, xk, xv)]
            args_m = [xm if x is y else y for y in (xq, xk, xv)]
            fd = (f(*args_p, p) - f(*args_m, p)) / (2 * h)
            assert abs(fd - got[name][idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx, fd, got[name][idx])
    for name in ("wq", "wk", "wv", "wo", "bq", "bv", "bo"):
        for idx in ([(0, 1), (3, 2), (2, 0)] if name.startswith("w") else [(0,), (3,)]):
            pp = {kk: (None if vv is None else vv.astype(np.float64).copy()) for kk, vv in p.items()}
            pm = {kk: (None if vv is None else vv.astype(np.float64).copy()) for kk, vv in p.items()}
            pp[name][idx] += h
            pm[name][idx] -= h
            fd = (f(xq, xk, xv, pp) - f(xq, xk, xv, pm)) / (2 * h)
            assert abs(fd - got["d" + name][idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx, fd)


@pytest.mark.parametrize("masked", [False, True])
def test_key_bias_gets_no_gradient(masked):
    rng = np.random.default_rng(21)
    E, H, L, S, B = 16, 4, 30, 40, 2
    p = _params(rng, E)
    src, tgt = synth.uniform_graph(rng, L, S, 300)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    kpm = (rng.random((B, S)) < 0.3) if masked else None
    g = oracle.backward(xq, xkv, xkv, p, src, tgt, H, rng.standard_normal((B, L, E)), key_padding_mask=kpm)
    assert np.abs(g["dbk"]).max() < 1e-12 * max(1.0, np.abs(g["dbq"]).max())
    assert np.abs(g["dbq"]).max() > 1e-6  # the query bias does get one


def test_single_source_targets_pass_no_score_gradient():
    rng = np.random.default_rng(5)
    E, H, n, B = 16, 4, 20, 2
    p = _params(rng, E)
    src = rng.integers(0, n, n).astype(np.int64)
    tgt = np.arange(n, dtype=np.int64)
    x = rng.standard_normal((B, n, E))
    g = oracle.backward(x, x, x, p, src, tgt, H, rng.standard_normal((B, n, E)))
    for name in ("dquery", "dwq", "dbq", "dkey", "dwk", "dbk"):
        assert np.all(g[name] == 0.0), name
    assert np.abs(g["dvalue"]).max() > 0.0


def test_bias_false_has_no_bias_gradients():
    # bias=False is the layer with zero biases: the same input and weight gradients
    rng = np.random.default_rng(6)
    E, H, n = 8, 2, 5
    p = _params(rng, E, bias=False)
    src, tgt = synth.complete_graph(rng, n)
    x = rng.standard_normal((1, n, E))
    dout = rng.standard_normal((1, n, E))
    g = oracle.backward(x, x, x, p, src, tgt, H, dout)
    assert all(g[n] is None for n in ("dbq", "dbk", "dbv", "dbo"))
    zero = {**p, "bq": np.zeros(E), "bk": np.zeros(E), "bv": np.zeros(E), "bo": np.zeros(E)}
    ref = _torch_grads(zero, H, x, x, x, dout)
    g["dquery"] = g["dquery"] + g["dkey"] + g["dvalue"]  # one tensor fed all three inputs
    ref["dquery"] = ref["dquery"] + ref["dkey"] + ref["dvalue"]
    _assert_grads(g, ref, 1e-11, names=("dquery", "dwq", "dwk", "dwv", "dwo"))


@pytest.mark.parametrize("masked", [False, True])
def test_output_and_value_bias_gradients_in_closed_form(masked):
    # out = mixed Wo^T + bo, so dbo = sum of dout over all (sample, target) and
    # dmixed = dout Wo. A target with a live key mixes sum_e w_e v_s with
    # weights summing to 1, so bv reaches it with coefficient 1: dbv = sum of
    # dmixed over the (sample, target) pairs that have a live key, and a target
    # without one contributes nothing.
    rng = np.random.default_rng(31)
    E, H, L, S, B = 16, 4, 24, 30, 3
    p = _params(rng, E)
    src, tgt = synth.uniform_graph(rng, L, S, 90, min_in_degree=0)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    kpm = (rng.random((B, S)) < 0.4) if masked else None
    dout = rng.standard_normal((B, L, E))
    g = oracle.backward(xq, xkv, xkv, p, src, tgt, H, dout, key_padding_mask=kpm)
    live = np.zeros((B, L), bool)
    for e in range(src.size):
        live[:, tgt[e]] |= True if kpm is None else ~kpm[:, src[e]]
    assert live.any() and (~live).any()
    dmixed = dout @ p["wo"].astype(np.float64)
    assert np.abs(g["dbo"] - dout.sum(axis=(0, 1))).max() < 1e-12
    assert np.abs(g["dbv"] - dmixed[live].sum(axis=0)).max() < 1e-11


def test_fully_masked_sample_gets_no_input_gradient():
    # every key of sample 1 is padding: its targets mix to zeros (their output
    # is bo whatever the inputs), so nothing flows back into that sample's
    # query, key or value tokens; the other samples do get gradients
    rng = np.random.default_rng(37)
    E, H, L, S, B = 16, 4, 20, 26, 3
    p = _params(rng, E)
    src, tgt = synth.uniform_graph(rng, L, S, 80, min_in_degree=1)
    xq = rng.standard_normal((B, L, E))
    xkv = rng.standard_normal((B, S, E))
    kpm = rng.random((B, S)) < 0.3
    kpm[1] = True
    dout = rng.standard_normal((B, L, E))
    g = oracle.backward(xq, xkv, xkv, p, src, tgt, H, dout, key_padding_mask=kpm)
    for n in ("dquery", "dkey", "dvalue"):
        assert np.all(g[n][1] == 0.0), n
        assert np.abs(g[n][0]).max() > 0 and np.abs(g[n][2]).max() > 0, n


def test_linear_backward_matches_numpy():
    rng = np.random.default_rng(1)
    x, w, dy = rng.standard_normal((7, 5)), rng.standard_normal((3, 5)), rng.standard_normal((7, 3))
    dx, dw, db = oracle.linear_backward(x, w, dy)
    assert np.allclose(dx, dy @ w, atol=1e-14)
    assert np.allclose(dw, dy.T @ x, atol=1e-14)
    assert np.allclose(db, dy.sum(0), atol=1e-14)
