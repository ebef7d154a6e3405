"""GPU parity of key_padding_mask (kpnn2 PackedMultiheadAttention, forward()
argument key_padding_mask): a flagged key drops out of the softmax of every
target it feeds, with weight 0; a target whose keys are all dropped mixes to
zeros, so its output row is exactly out_proj's bias. Checked element by element
against the fp64 oracle, plus the exact properties."""
import numpy as np
import pytest

import oracle
import synth
from tests._cases import Case, assert_close, assert_close_weights, torch_dtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _masked_targets(c, kpm):
    """(B, L) bool: targets with at least one edge, all of whose keys are flagged."""
    deg = np.bincount(c.tgt, minlength=c.L)
    live = np.zeros((c.B, c.L), np.int64)
    for b in range(c.B):
        np.add.at(live[b], c.tgt, ~kpm[b][c.src])
    return (live == 0) & (deg > 0)[None, :]


@pytest.mark.parametrize("wid,B,kind", [(1, 3, "scattered"), (2, 2, "padding"), (3, 1, "padding"),
                                        (4, 2, "scattered"), (5, 2, "padding"), (2, 2, "scattered")])
def test_masked_forward_matches_oracle(wid, B, kind):
    c = Case.workload(wid, batch=B)
    rng = np.random.default_rng(100 + wid)
    kpm = (synth.padding_mask(rng, B, c.S) if kind == "padding" else synth.scattered_mask(rng, B, c.S, 0.4))
    g, params, out, w = c.run(DEV, "per_head", kpm=kpm)
    ref_out, ref_w = c.oracle(kpm=kpm)
    assert_close("output", out.float().cpu().numpy(), ref_out, c.dt)
    wn = w.cpu().numpy()
    assert_close_weights("weights", wn, ref_w, c.dt)
    # flagged keys weigh exactly 0
    dropped = kpm[:, c.src]  # (B, nnz)
    assert np.all(wn[dropped] == 0.0)
    # targets whose keys are all flagged: exactly out_proj's bias
    dead = _masked_targets(c, kpm)
    if dead.any():
        bo = torch.from_numpy(c.params["bo"]).to(DEV).to(out.dtype)
        got = out[torch.from_numpy(dead).to(DEV)]
        assert torch.equal(got, bo.expand_as(got))
    _, _, out2, wa = c.run(DEV, "avg", graph=g, kpm=kpm)
    assert torch.equal(out, out2)
    assert_close_weights("avg weights", wa.cpu().numpy(), oracle.average_heads(ref_w), c.dt)
    g.destroy()


def test_mask_empties_a_whole_unit_of_a_split_target():
    # complete graph, 1024 sources per target (several units of edges each):
    # sample 0 drops keys 0..599, so whole units of every target are dropped
    # and the merge combines empty pieces with live ones; sample 1 drops all
    # keys but one, sample 2 drops every key
    c = Case.workload(5, batch=3)
    kpm = np.zeros((3, c.S), np.bool_)
    kpm[0, :600] = True
    kpm[1, :] = True
    kpm[1, 777] = False
    kpm[2, :] = True
    g, params, out, w = c.run(DEV, "per_head", kpm=kpm)
    ref_out, ref_w = c.oracle(kpm=kpm)
    assert_close("output", out.float().cpu().numpy(), ref_out, c.dt)
    wn = w.cpu().numpy()
    assert_close_weights("weights", wn, ref_w, c.dt)
    # sample 1: the one live key carries weight exactly 1 for every target and head
    live = c.src == 777
    assert np.all(wn[1][live] == 1.0) and np.all(wn[1][~live] == 0.0)
    # sample 2: nothing live, every row is out_proj's bias and every weight 0
    bo = torch.from_numpy(c.params["bo"]).to(DEV).to(out.dtype)
    assert torch.equal(out[2], bo.expand(c.L, -1))
    assert np.all(wn[2] == 0.0)
    g.destroy()


@pytest.mark.parametrize("wid", [1, 3])
def test_empty_mask_equals_no_mask(wid):
    c = Case.workload(wid, batch=2)
    g, params, out, w = c.run(DEV, "per_head")
    _, _, out2, w2 = c.run(DEV, "per_head", graph=g, kpm=np.zeros((2, c.S), np.bool_))
    assert torch.equal(out, out2) and torch.equal(w, w2)
    g.destroy()


@pytest.mark.parametrize("wid", [1, 4])
def test_masked_edge_weights_bit_identical_to_forward(wid):
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(wid, batch=2)
    kpm = synth.scattered_mask(np.random.default_rng(9), 2, c.S, 0.5)
    mask = torch.from_numpy(kpm).to(DEV)
    for mode in ("avg", "per_head"):
        g, params, out, w = c.run(DEV, mode, kpm=kpm)
        xq, xkv = c.device_inputs(DEV)
        w2 = pmha.pmha_edge_weights(g, params, xq, xkv, mode, key_padding_mask=mask)
        pmha.pmha_device_status()
        assert torch.equal(w, w2), mode
        g.destroy()


def test_masked_forward_host_matches_forward():
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(2, batch=2)
    kpm = synth.padding_mask(np.random.default_rng(11), 2, c.S)
    g, params, out, w = c.run(DEV, "avg", kpm=kpm)
    tdt = torch_dtype(c.dt)
    xq = torch.from_numpy(c.xq).to(tdt).pin_memory()
    out_h = torch.empty_like(xq).pin_memory()
    w_h = torch.empty(w.shape, dtype=torch.float32).pin_memory()
    pmha.pmha_forward_host(g, params, xq, xq, xq, out_h, "avg", w_h, key_padding_mask=torch.from_numpy(kpm))
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out_h) and torch.equal(w.cpu(), w_h)
    g.destroy()


def test_layer_object_takes_the_mask():
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(1, batch=2)
    kpm = synth.scattered_mask(np.random.default_rng(12), 2, c.S, 0.3)
    params = pmha.Params.from_arrays(c.params, c.H, torch_dtype(c.dt), DEV)
    layer = pmha.PackedMultiheadAttention(c.src, c.tgt, c.L, c.S, params, device=DEV)
    xq, _ = c.device_inputs(DEV)
    out, w = layer(xq, xq, xq, key_padding_mask=torch.from_numpy(kpm).to(DEV), need_weights=True,
                   average_attn_weights=False)
    pmha.pmha_device_status()
    ref_out, ref_w = c.oracle(kpm=kpm)
    assert_close("output", out.float().cpu().numpy(), ref_out, c.dt)
    assert_close_weights("weights", w.cpu().numpy(), ref_w, c.dt)
    layer.graph.destroy()


def test_mask_argument_errors():
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(1, batch=2)
    params = pmha.Params.from_arrays(c.params, c.H, torch_dtype(c.dt), DEV)
    g = pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), c.L, c.S)
    xq, _ = c.device_inputs(DEV)
    for bad in (torch.zeros((2, c.S + 1), dtype=torch.bool, device=DEV),     # wrong shape
                torch.zeros((2, c.S), dtype=torch.float32, device=DEV),      # wrong dtype
                torch.zeros((2, c.S), dtype=torch.bool)):                    # host tensor for a device call
        with pytest.raises(ValueError):
            pmha.pmha_forward(g, params, xq, xq, xq, "none", key_padding_mask=bad)
    g.destroy()
