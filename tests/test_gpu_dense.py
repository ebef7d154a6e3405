"""GPU parity of the masked-dense tensor-core path (graphs where at least a
quarter of the (target, source) pairs are edges) against the fp64 oracle.
kpnn2 PackedMultiheadAttention, Notes steps 2-4: restricting attention to the
edges equals dense attention with the score matrix masked to the edges, so a
dense graph may run as masked tiles; the result must not change."""
import numpy as np
import pytest

import oracle
import synth
from tests._cases import Case, assert_close, assert_close_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _stages_of(fn):
    import graph_sparse_head_gb300 as pmha
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    try:
        res = fn()
        torch.cuda.synchronize()
        return res, set(pmha.pmha_profile_read())
    finally:
        pmha.pmha_profile_enable(False)


def _dense_pairs(rng, L, S, density):
    keep = rng.random((L, S)) < density
    t, s = np.nonzero(keep)
    return synth.shuffle_edges(rng, s.astype(np.int64), t.astype(np.int64))


@pytest.mark.parametrize("n,E,H,B", [(256, 512, 8, 2), (200, 512, 4, 1), (136, 256, 4, 3)])
def test_complete_graph(n, E, H, B):
    rng = np.random.default_rng(n + E)
    src, tgt = synth.complete_graph(rng, n)
    c = Case(src, tgt, n, n, E, H, B, "bf16", seed=n)
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "none"))
    assert "dense_attn" in stages and "edge_attn" not in stages and "edge_attn_out" not in stages
    ref_out, _ = c.oracle(need_weights=False)
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    g.destroy()


@pytest.mark.parametrize("L,S,E,H,B,density,bip", [
    (300, 300, 256, 4, 2, 0.6, False),   # ragged target tile, some sources missing per row
    (200, 520, 512, 8, 2, 0.8, True),    # bipartite, d = 64
    (129, 136, 256, 2, 1, 0.3, True),    # d = 128, near the density threshold
])
def test_near_complete_graph(L, S, E, H, B, density, bip):
    rng = np.random.default_rng(L * S)
    src, tgt = _dense_pairs(rng, L, S, density)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=L + S, bipartite=bip)
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "per_head"))
    assert "dense_attn" in stages
    ref_out, ref_w = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    assert_close_weights("weights", w.cpu().numpy(), ref_w, "bf16")
    g.destroy()


def test_dense_targets_without_sources_give_bias():
    # rows 0..9 have no source at all: their mix is zero and the output is bo
    rng = np.random.default_rng(3)
    L = S = 256
    keep = rng.random((L, S)) < 0.7
    keep[:10] = False
    t, s = np.nonzero(keep)
    src, tgt = synth.shuffle_edges(rng, s.astype(np.int64), t.astype(np.int64))
    c = Case(src, tgt, L, S, 256, 4, 2, "bf16", seed=4)
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "none"))
    assert "dense_attn" in stages
    bo = torch.from_numpy(c.params["bo"]).to(DEV).to(out.dtype)
    assert torch.equal(out[:, :10], bo.expand(2, 10, -1))
    ref_out, _ = c.oracle(need_weights=False)
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    g.destroy()


def test_dense_with_key_padding_mask():
    rng = np.random.default_rng(8)
    n, E, H, B = 384, 512, 8, 3
    src, tgt = synth.complete_graph(rng, n)
    c = Case(src, tgt, n, n, E, H, B, "bf16", seed=9)
    kpm = synth.padding_mask(rng, B, n)
    kpm[2, :] = True  # a sample whose keys are all padding: every row is out_proj's bias
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "avg", kpm=kpm))
    assert "dense_attn" in stages
    ref_out, ref_w = c.oracle(kpm=kpm)
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    assert_close_weights("avg weights", w.cpu().numpy(), oracle.average_heads(ref_w), "bf16")
    bo = torch.from_numpy(c.params["bo"]).to(DEV).to(out.dtype)
    assert torch.equal(out[2], bo.expand(n, -1))
    g.destroy()


def test_dense_edge_weights_bit_identical_to_forward():
    import graph_sparse_head_gb300 as pmha
    rng = np.random.default_rng(12)
    src, tgt = _dense_pairs(rng, 256, 256, 0.5)
    c = Case(src, tgt, 256, 256, 256, 4, 2, "bf16", seed=13)
    for mode in ("avg", "per_head"):
        g, params, out, w = c.run(DEV, mode)
        xq, xkv = c.device_inputs(DEV)
        w2 = pmha.pmha_edge_weights(g, params, xq, xkv, mode)
        pmha.pmha_device_status()
        assert torch.equal(w, w2), mode
        g.destroy()


def test_sparse_graph_stays_on_the_edge_kernel():
    c = Case.workload(2, batch=1)
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "none"))
    assert ("edge_attn" in stages or "edge_attn_out" in stages) and "dense_attn" not in stages
    g.destroy()


def test_dense_reference_moves_after_the_first_step():
    # Keys scaled by 1, 3, 1 and 5 in consecutive blocks of 128 sources (the
    # dense kernel's steps): in the second and last steps about 40 % of the
    # rows' maxima pass the running softmax reference by more than its lazy
    # threshold and the others do not, so warps rescale O and l for some rows
    # and keep them for the rest; scores reach about 34 log2 units.
    from tests._cases import score_bound
    rng = np.random.default_rng(21)
    L, S, E, H, B = 256, 512, 256, 4, 2
    src, tgt = _dense_pairs(rng, L, S, 1.1)
    xq = synth.make_tokens(rng, B, L, E, "bf16")
    gain = np.repeat(np.array([1.0, 3.0, 1.0, 5.0], np.float32), 128)
    xkv = synth.bf16_round(synth.make_tokens(rng, B, S, E, "bf16") * gain[None, :, None])
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=22, bipartite=True, xq=xq, xkv=xkv)
    # the moves are real: per (sample, head, target), the step maxima in log2 units
    d = E // H
    moved = []
    for b in range(B):
        q = oracle.linear(c.xq[b], c.params["wq"], c.params["bq"]).reshape(L, H, d)
        k = oracle.linear(c.xkv[b], c.params["wk"], c.params["bk"]).reshape(S, H, d)
        s = np.einsum("thc,shc->hts", q, k) * (1.4426950408889634 / np.sqrt(d))
        step_max = s.reshape(H, L, 4, 128).max(axis=3)
        run = np.maximum.accumulate(step_max, axis=2)
        moved.append(step_max[:, :, 1:] > run[:, :, :-1] + 8.0)
    moved = np.stack(moved)
    assert 0.1 < moved[..., 0].mean() < 0.9 and 0.1 < moved[..., 2].mean() < 0.9, moved.mean(axis=(0, 1, 2))
    (g, params, out, w), stages = _stages_of(lambda: c.run(DEV, "per_head"))
    assert "dense_attn" in stages
    ref_out, ref_w = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    assert_close_weights("weights", w.cpu().numpy(), ref_w, "bf16", score_bound=score_bound(c))
    g.destroy()
