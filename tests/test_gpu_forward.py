"""GPU parity of pmha_forward / pmha_edge_weights / pmha_forward_host against
the fp64 oracle, element by element, at sizes the oracle finishes in seconds
(several GEMM tiles and a ragged tail), plus the exact properties the kpnn2
page fixes (single source -> weight 1, no source -> out_proj bias, weights sum
to 1, independence of edge order)."""
import numpy as np
import pytest

import oracle
import synth
from tests._cases import Case, assert_close, assert_close_weights, score_bound, torch_dtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _small(wid, B):
    """A workload at its own graph and widths, with fewer samples."""
    return Case.workload(wid, batch=B)


@pytest.mark.parametrize("wid,B", [(1, 2), (2, 2), (3, 1), (4, 2), (5, 1)])
def test_forward_matches_oracle_small_batch(wid, B):
    c = _small(wid, B)
    wmode = "per_head"
    g, params, out, w = c.run(DEV, wmode)
    ref_out, ref_w = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, c.dt)
    assert_close_weights("weights", w.cpu().numpy(), ref_w, c.dt)
    # averaged weights, same inputs
    _, _, out2, wa = c.run(DEV, "avg", graph=g)
    assert torch.equal(out, out2)
    assert_close_weights("avg weights", wa.cpu().numpy(), oracle.average_heads(ref_w), c.dt)
    g.destroy()


@pytest.mark.parametrize("L,S,nnz,E,H,B,dt,bip", [
    (64, 64, 256, 32, 4, 3, "f32", False),      # fp32, 4 lanes per row
    (130, 70, 900, 64, 4, 2, "f32", True),      # fp32, d = 16
    (257, 257, 3000, 64, 4, 2, "bf16", False),  # bf16 width without a tensor-core tile -> CUDA-core GEMM
    (200, 333, 4000, 256, 4, 2, "bf16", True),  # d = 64
    (150, 150, 2000, 512, 16, 1, "bf16", False),  # 16 channels per lane, d = 32
    (100, 100, 1200, 32, 4, 2, "bf16", False),  # 4 lanes per row
    (90, 90, 800, 8, 2, 2, "f32", False),       # the tutorial's widths (E = 8, H = 2)
    (129, 129, 1500, 128, 2, 2, "bf16", False),  # d = 64 on E = 128
    (60, 600, 15000, 128, 8, 3, "bf16", True),  # bipartite, ~250 edges per target: split targets
])
def test_forward_shapes_and_dtypes(L, S, nnz, E, H, B, dt, bip):
    rng = np.random.default_rng(L * 31 + E)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=0)
    c = Case(src, tgt, L, S, E, H, B, dt, seed=E + H, bipartite=bip)
    g, params, out, w = c.run(DEV, "per_head")
    ref_out, ref_w = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, dt)
    assert_close_weights("weights", w.cpu().numpy(), ref_w, dt)
    g.destroy()


@pytest.mark.parametrize("E", [128, 256, 512])  # 256, 512: the 128 x 256 projection tiles, without bias
def test_key_differs_from_value_and_no_bias(E):
    rng = np.random.default_rng(3)
    L, S, H, B = 300, 500, 8, 2
    src, tgt = synth.bipartite_membership_graph(rng, L, S, 5, 60)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=4, bipartite=True, bias=False)
    xv = synth.make_tokens(rng, B, S, E, "bf16")
    import graph_sparse_head_gb300 as pmha
    params = pmha.Params.from_arrays(c.params, H, torch.bfloat16, DEV)
    g = pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), L, S)
    xq, xk = c.device_inputs(DEV)
    v = torch.from_numpy(xv).to(DEV).to(torch.bfloat16)
    out, w = pmha.pmha_forward(g, params, xq, xk, v, "avg")
    pmha.pmha_device_status()
    ref_out, ref_w = oracle.forward(c.xq, c.xkv, xv, c.params, c.src, c.tgt, H)
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    assert_close_weights("avg weights", w.cpu().numpy(), oracle.average_heads(ref_w), "bf16")
    g.destroy()


def test_self_loops_appended_and_weights_in_given_order():
    # the kpnn2 doctest graph: x->a, a->b, b->a, a->y with nodes a, b, x, y = 0..3
    src, tgt = [0, 0, 1, 2], [1, 3, 0, 0]
    c = Case(src, tgt, 4, 4, 32, 4, 2, "f32", seed=1)
    g, params, out, w = c.run(DEV, "per_head", add_self_loops=True)
    assert g.nnz == 8 and tuple(w.shape) == (2, 8, 4)
    s2, t2 = oracle.append_self_loops(c.src, c.tgt, 4)
    ref_out, ref_w = c.oracle(src=s2, tgt=t2)
    assert_close("output", out.float().cpu().numpy(), ref_out, "f32")
    assert_close_weights("weights", w.cpu().numpy(), ref_w, "f32")
    # x (node 2) has only its self-loop: weight exactly 1
    assert torch.all(w[:, 6, :] == 1.0)
    g.destroy()
    # without self-loops x has no source: output is exactly out_proj's bias
    g, params, out, w = c.run(DEV, "avg")
    bo = torch.from_numpy(c.params["bo"]).to(DEV)
    assert torch.equal(out[:, 2, :], bo.expand(2, -1))
    g.destroy()


@pytest.mark.parametrize("L,S,nnz,E,H,B,bip", [
    (300, 300, 2999, 128, 8, 6, False),  # two sample groups of 4, the second half empty; last unit 7 positions
    (200, 400, 3001, 256, 8, 3, True),   # 2 samples a warp: the second group has one; last unit 9 positions
    (150, 150, 2113, 512, 8, 1, False),  # a whole warp per sample, d = 64 over 4 lanes; last unit 1 position
])
def test_sample_groups_and_ragged_last_unit(L, S, nnz, E, H, B, bip):
    # The edge kernel walks sample groups of 32 / (E / 16) samples per warp:
    # slots past the batch compute on the last sample and store nothing, and
    # the graph's last unit of positions is short and odd-sized here.
    import graph_sparse_head_gb300 as pmha
    rng = np.random.default_rng(nnz)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=1)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=E + B, bipartite=bip)
    g, params, out, w = c.run(DEV, "per_head")
    ref_out, ref_w = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, "bf16")
    assert_close_weights("weights", w.cpu().numpy(), ref_w, "bf16")
    xq, xkv = c.device_inputs(DEV)
    w2 = pmha.pmha_edge_weights(g, params, xq, xkv, "per_head")
    pmha.pmha_device_status()
    assert torch.equal(w, w2)
    g.destroy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_single_source_targets_exact(dt):
    # every target has exactly one source: weights are exactly 1, the mix is
    # the source's value row, and the layer is out_proj(v_proj(x_source))
    n, E, H, B = 700, 128, 8, 2
    rng = np.random.default_rng(5)
    src = rng.integers(0, n, n)
    tgt = np.arange(n)
    src, tgt = synth.shuffle_edges(rng, src, tgt)
    c = Case(src, tgt, n, n, E, H, B, dt, seed=6)
    g, params, out, w = c.run(DEV, "per_head")
    assert torch.all(w == 1.0)
    ref_out, _ = c.oracle()
    assert_close("output", out.float().cpu().numpy(), ref_out, dt)
    g.destroy()


@pytest.mark.parametrize("L,S,nnz,E,H,B,dt,bip,scale,masked", [
    (300, 300, 9000, 128, 8, 2, "bf16", False, 2.0, False),
    (60, 600, 15000, 128, 8, 2, "bf16", True, 2.0, False),   # split targets: pieces merged
    (300, 300, 9000, 128, 8, 2, "bf16", False, 2.0, True),    # with a key_padding_mask
    (130, 70, 900, 64, 4, 2, "f32", True, 3.0, False),
    (64, 64, 256, 32, 4, 3, "f32", False, 3.0, False),
])
def test_sharp_scores_move_the_softmax_reference(L, S, nnz, E, H, B, dt, bip, scale, masked):
    # Tokens scaled up so that scores spread over tens of log2 units within one
    # target: the running softmax reference has to move many times, by more
    # than its lazy threshold, and the weights are close to one-hot.
    rng = np.random.default_rng(L + 7 * E)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=1)
    rnd = synth.bf16_round if dt == "bf16" else (lambda x: x.astype(np.float32))
    xq = rnd(synth.make_tokens(rng, B, L, E, dt) * np.float32(scale))
    xkv = rnd(synth.make_tokens(rng, B, S, E, dt) * np.float32(scale)) if bip else xq
    c = Case(src, tgt, L, S, E, H, B, dt, seed=E, bipartite=bip, xq=xq, xkv=xkv)
    kpm = synth.padding_mask(rng, B, S) if masked else None
    g, params, out, w = c.run(DEV, "per_head", kpm=kpm)
    ref_out, ref_w = c.oracle(kpm=kpm)
    assert np.nanmax(ref_w) > 0.99  # the spread is real: some weights are one-hot
    assert_close("output", out.float().cpu().numpy(), ref_out, dt)
    assert_close_weights("weights", w.cpu().numpy(), ref_w, dt, score_bound=score_bound(c))
    g.destroy()


@pytest.mark.parametrize("wid", [2, 4])
def test_weights_sum_to_one_per_target_and_head(wid):
    c = _small(wid, 2)
    g, params, out, w = c.run(DEV, "per_head")
    wn = w.double().cpu().numpy()
    assert (wn >= 0).all()
    sums = np.zeros((c.B, c.L, c.H))
    np.add.at(sums, (slice(None), c.tgt), wn)
    deg = np.bincount(c.tgt, minlength=c.L)
    assert np.abs(sums[:, deg > 0] - 1.0).max() < 1e-4
    assert np.all(sums[:, deg == 0] == 0.0)
    g.destroy()


@pytest.mark.parametrize("wid", [1, 3, 4])
def test_edge_weights_bit_identical_to_forward(wid):
    import graph_sparse_head_gb300 as pmha
    c = _small(wid, 2)
    for mode in ("avg", "per_head"):
        g, params, out, w = c.run(DEV, mode)
        xq, xkv = c.device_inputs(DEV)
        w2 = pmha.pmha_edge_weights(g, params, xq, xkv, mode)
        pmha.pmha_device_status()
        assert torch.equal(w, w2), mode
        g.destroy()


@pytest.mark.parametrize("wid", [1, 3])
def test_results_independent_of_edge_order(wid):
    c = _small(wid, 2)
    g, params, out, w = c.run(DEV, "per_head")
    rng = np.random.default_rng(77)
    p = rng.permutation(len(c.src))
    c2 = Case(c.src[p], c.tgt[p], c.L, c.S, c.E, c.H, c.B, c.dt, 0, xq=c.xq, xkv=c.xkv, params=c.params)
    g2, _, out2, w2 = c2.run(DEV, "per_head")
    assert torch.equal(out, out2)
    assert torch.equal(w[:, torch.from_numpy(p).to(DEV)], w2)
    g.destroy()
    g2.destroy()


@pytest.mark.parametrize("wid,mode", [(2, "none"), (4, "avg"), (1, "per_head")])
def test_forward_host_matches_forward(wid, mode):
    import graph_sparse_head_gb300 as pmha
    c = _small(wid, 2)
    g, params, out, w = c.run(DEV, mode)
    tdt = torch_dtype(c.dt)
    xq = torch.from_numpy(c.xq).to(tdt).pin_memory()
    xkv = xq if c.xkv is c.xq else torch.from_numpy(c.xkv).to(tdt).pin_memory()
    out_h = torch.empty_like(xq).pin_memory()
    w_h = None if w is None else torch.empty(w.shape, dtype=torch.float32).pin_memory()
    pmha.pmha_forward_host(g, params, xq, xkv, xkv, out_h, mode, w_h)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out_h)
    if w is not None:
        assert torch.equal(w.cpu(), w_h)
    g.destroy()


def test_argument_errors():
    import graph_sparse_head_gb300 as pmha
    c = _small(1, 2)
    g, params, out, w = c.run(DEV, "none")
    xq, _ = c.device_inputs(DEV)
    small_ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        pmha.pmha_forward(g, params, xq, xq, xq, "none", workspace=small_ws)
    # through the C ABI directly: workspace too small, bad weight mode
    import ctypes
    lib = pmha._lib.load()
    p = params.as_struct()
    st = lib.pmha_forward(g.handle, ctypes.byref(p), xq.data_ptr(), xq.data_ptr(), xq.data_ptr(), None, 2,
                          out.data_ptr(), 0, None, small_ws.data_ptr(), 16, None)
    assert pmha._lib.STATUS_NAMES[st] == "PMHA_ERR_WORKSPACE"
    st = lib.pmha_forward(g.handle, ctypes.byref(p), xq.data_ptr(), xq.data_ptr(), xq.data_ptr(), None, 2,
                          out.data_ptr(), 7, None, small_ws.data_ptr(), 16, None)
    assert pmha._lib.STATUS_NAMES[st] == "PMHA_ERR_INVALID_ARG"
    st = lib.pmha_forward(g.handle, ctypes.byref(p), xq.data_ptr() + 4, xq.data_ptr(), xq.data_ptr(), None, 2,
                          out.data_ptr(), 0, None, small_ws.data_ptr(), 16, None)
    assert pmha._lib.STATUS_NAMES[st] == "PMHA_ERR_INVALID_ARG"
    bad = pmha._lib.PmhaParams(32, 5, 0, p.wq, p.wk, p.wv, p.wo, None, None, None, None)
    assert lib.pmha_forward_workspace_size(g.handle, ctypes.byref(bad), 2, 0) == 0
    pmha.pmha_device_status()
    g.destroy()


def test_binding_refuses_mismatched_results_before_launch():
    import graph_sparse_head_gb300 as pmha
    c = _small(1, 2)
    g, params, out, w = c.run(DEV, "per_head")
    xq, _ = c.device_inputs(DEV)
    n0 = pmha.pmha_launch_count()
    bad_calls = [
        dict(out=torch.empty(2, c.L, c.E - 1, dtype=out.dtype, device=DEV)),          # short rows
        dict(out=torch.empty(2, c.L, c.E, dtype=torch.float64, device=DEV)),          # dtype
        dict(out=torch.empty(2, c.E, c.L, dtype=out.dtype, device=DEV).transpose(1, 2)),  # strided
        dict(weights=torch.empty(2, c.src.size, dtype=torch.float32, device=DEV)),   # avg shape for per_head
        dict(workspace=torch.empty(1 << 20, dtype=torch.uint8)),                      # host workspace
    ]
    for kw in bad_calls:
        with pytest.raises(ValueError):
            pmha.pmha_forward(g, params, xq, xq, xq, "per_head", **kw)
    with pytest.raises(ValueError):
        pmha.pmha_edge_weights(g, params, xq, xq, "avg", weights=torch.empty(2, c.src.size + 1, device=DEV))
    assert pmha.pmha_launch_count() == n0  # nothing was launched
    pmha.pmha_device_status()
    g.destroy()


@pytest.mark.parametrize("fused", [True, False, None])
def test_launch_counter_and_profile(fused, monkeypatch):
    import graph_sparse_head_gb300 as pmha
    if fused is None:  # the default: out_proj as its own GEMM
        monkeypatch.delenv("PMHA_FUSED_OUT_PROJ", raising=False)
    else:
        monkeypatch.setenv("PMHA_FUSED_OUT_PROJ", "1" if fused else "0")
    c = _small(2, 1)
    n0 = pmha.pmha_launch_count()
    pmha.pmha_profile_enable(True)
    g, params, out, w = c.run(DEV, "none")
    prof = pmha.pmha_profile_read()
    pmha.pmha_profile_enable(False)
    assert pmha.pmha_launch_count() > n0
    assert prof["proj_qkv"][0] == 1  # fused Q|K|V
    if fused:  # out_proj runs inside the edge kernel
        assert "edge_attn_out" in prof and prof["edge_attn_out"][0] == 1 and prof["edge_attn_out"][1] > 0
        assert "out_proj" not in prof and "edge_attn" not in prof
    else:
        assert "edge_attn" in prof and prof["edge_attn"][0] == 1 and prof["edge_attn"][1] > 0
        assert prof["out_proj"][0] == 1
    g.destroy()


def test_fp16_intermediate_overflow_is_reported():
    import graph_sparse_head_gb300 as pmha
    rng = np.random.default_rng(21)
    n, E, H = 200, 128, 8
    src, tgt = synth.uniform_graph(rng, n, n, 1000)
    c = Case(src, tgt, n, n, E, H, 1, "bf16", seed=2)
    c.xq = synth.bf16_round(c.xq * 3.0e5)  # projections far beyond 65504
    c.xkv = c.xq
    params = pmha.Params.from_arrays(c.params, H, torch.bfloat16, DEV)
    g = pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), n, n)
    xq, _ = c.device_inputs(DEV)
    pmha.pmha_forward(g, params, xq, xq, xq, "none")
    with pytest.raises(pmha.PmhaError) as ei:
        pmha.pmha_device_status()
    assert ei.value.status_name == "PMHA_ERR_OVERFLOW"
    pmha.pmha_device_status()  # the flag is cleared by the report
    # the binding's check=True reports it from the call itself
    with pytest.raises(pmha.PmhaError) as ei:
        pmha.pmha_forward(g, params, xq, xq, xq, "none", check=True)
    assert ei.value.status_name == "PMHA_ERR_OVERFLOW"
    out, _ = pmha.pmha_forward(g, params, xq[:, :, :] * 0, xq * 0, xq * 0, "none", check=True)  # in range: no error
    g.destroy()
