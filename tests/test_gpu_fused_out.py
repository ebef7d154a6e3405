"""GPU: out_proj run inside the edge kernel (kpnn2 PackedMultiheadAttention,
Notes step 5, as out_proj tasks in the edge kernel's queue; embed_dim 128),
against the oracle element by element and against the separate out_proj
GEMM (PMHA_FUSED_OUT_PROJ=0): several sample groups with idle slots, row
blocks cut by a ragged tail (L not a multiple of 64), key_padding_mask,
need_weights, targets without edges (whose output row is exactly bo),
bitwise repeatability, and embed_dim 256 staying on the separate GEMM."""
import numpy as np
import pytest

import synth
from tests._cases import Case, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _stages(fn):
    import graph_sparse_head_gb300 as pmha
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    try:
        res = fn()
        torch.cuda.synchronize()
        return res, set(pmha.pmha_profile_read())
    finally:
        pmha.pmha_profile_enable(False)


def _run(c, fused, monkeypatch, kpm=None, wmode="none"):
    monkeypatch.setenv("PMHA_FUSED_OUT_PROJ", "1" if fused else "0")
    (g, params, out, w), stages = _stages(lambda: c.run(DEV, wmode, kpm=kpm))
    inside = fused and c.E == 128  # the fused path holds a 128 x 128 Wo per block
    assert ("edge_attn_out" in stages) == inside and ("out_proj" in stages) == (not inside), stages
    return g, out, w


@pytest.mark.parametrize("L,S,nnz,E,H,B,bip,masked", [
    (300, 300, 2999, 128, 8, 6, False, False),    # two sample groups, the second half idle; 5 row blocks, ragged
    (200, 400, 3001, 128, 4, 7, True, False),     # bipartite, 2 groups, 3 live slots in the last
    (1000, 1000, 9000, 128, 4, 9, False, True),   # 3 groups (out_proj tasks between edge tasks); masked keys
    (640, 640, 12800, 128, 8, 13, False, False),  # 4 groups, L a multiple of 64
    (200, 400, 3001, 256, 8, 3, True, False),     # embed_dim 256: out_proj stays a GEMM
])
def test_fused_matches_oracle_and_unfused(L, S, nnz, E, H, B, bip, masked, monkeypatch):
    rng = np.random.default_rng(nnz + E)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=1)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=L + B, bipartite=bip)
    kpm = synth.padding_mask(np.random.default_rng(3), B, S) if masked else None
    ref, _ = c.oracle(need_weights=False, kpm=kpm)
    g1, fused, _ = _run(c, True, monkeypatch, kpm=kpm)
    g2, split, _ = _run(c, False, monkeypatch, kpm=kpm)
    assert_close("fused output", fused.float().cpu().numpy(), ref, "bf16")
    assert_close("unfused output", split.float().cpu().numpy(), ref, "bf16")
    # same inputs to the product (the mixed rows), summed in another order:
    # at most a couple of bf16 steps apart
    d = (fused.float() - split.float()).abs()
    step = split.float().abs().clamp_min(2.0 ** -20) * 2.0 ** -7
    assert bool((d <= 2 * step + 1e-6).all()), float((d / step).max())
    g3, again, _ = _run(c, True, monkeypatch, kpm=kpm)
    assert torch.equal(fused, again)  # bitwise repeatable
    for g in (g1, g2, g3):
        g.destroy()


def test_targets_without_edges_get_exactly_the_bias(monkeypatch):
    # 400 targets, 300 edges: most targets have none and their rows are bo
    rng = np.random.default_rng(5)
    L = S = 400
    src, tgt = synth.uniform_graph(rng, L, S, 300, min_in_degree=0)
    c = Case(src, tgt, L, S, 128, 8, 5, "bf16", seed=9)
    g, out, _ = _run(c, True, monkeypatch)
    empty = np.setdiff1d(np.arange(L), tgt)
    assert empty.size > 100
    bo = torch.from_numpy(np.asarray(c.params["bo"], np.float32)).to(torch.bfloat16)
    got = out[:, torch.from_numpy(empty)].cpu()
    assert torch.equal(got, bo.expand_as(got))
    ref, _ = c.oracle(need_weights=False)
    assert_close("output", out.float().cpu().numpy(), ref, "bf16")
    g.destroy()


@pytest.mark.parametrize("wmode", ["avg", "per_head"])
def test_fused_with_weights(wmode, monkeypatch):
    # the raw-score write-out and the out_proj tasks in one kernel
    from tests._cases import assert_close_weights
    import oracle
    rng = np.random.default_rng(31)
    src, tgt = synth.uniform_graph(rng, 500, 3000, 20000, min_in_degree=1)
    c = Case(src, tgt, 500, 3000, 128, 8, 5, "bf16", seed=4, bipartite=True)
    g, out, w = _run(c, True, monkeypatch, wmode=wmode)
    ref, ref_w = c.oracle(need_weights=True)
    assert_close("output", out.float().cpu().numpy(), ref, c.dt)
    wr = ref_w if wmode == "per_head" else oracle.average_heads(ref_w)
    assert_close_weights("weights", w.cpu().numpy(), wr, c.dt)
    g.destroy()
