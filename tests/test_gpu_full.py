"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: every output element of every workload against the oracle
(the bipartite workload 4 also every per-head and head-averaged weight, the
oracle run in chunks of samples), plus properties that hold at any size
(weights sum to 1, edge_weights == forward weights)."""
import numpy as np
import pytest

import oracle
import synth
from tests._cases import Case, assert_close, assert_close_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.mark.parametrize("wid", [1, 2, 3, 5])
def test_full_workload_every_element(wid):
    c = Case.workload(wid)
    wmode = "per_head" if wid == 1 else "none"
    g, params, out, w = c.run(DEV, wmode)
    ref_out, ref_w = c.oracle(need_weights=wid == 1)
    assert_close(f"workload {wid} output", out.float().cpu().numpy(), ref_out, c.dt)
    if wid == 1:
        assert_close_weights("workload 1 weights", w.cpu().numpy(), ref_w, c.dt)
    g.destroy()


@pytest.mark.parametrize("wid", [2, 3])
def test_full_workload_fused_out_proj_every_element(wid, monkeypatch):
    # out_proj inside the edge kernel (PMHA_FUSED_OUT_PROJ=1) at full size:
    # every output element against the oracle
    monkeypatch.setenv("PMHA_FUSED_OUT_PROJ", "1")
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(wid)
    pmha.pmha_profile_enable(True)
    pmha.pmha_profile_read()
    g, params, out, _ = c.run(DEV, "none")
    stages = set(pmha.pmha_profile_read())
    pmha.pmha_profile_enable(False)
    assert "edge_attn_out" in stages and "out_proj" not in stages, stages
    ref_out, _ = c.oracle(need_weights=False)
    assert_close(f"workload {wid} fused output", out.float().cpu().numpy(), ref_out, c.dt)
    g.destroy()


def test_full_bipartite_every_element():
    # workload 4 at full size (B=64, 500 pathways x 20,000 genes, E=256,
    # need_weights): every output element, every per-head weight and every
    # head-averaged weight against the oracle, which runs in chunks of samples
    # so that host memory stays bounded
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(4)
    g, params, out, w = c.run(DEV, "per_head")
    out_n = out.float().cpu().numpy()
    w_n = w.cpu().numpy()
    del w
    xq, xkv = c.device_inputs(DEV)
    wa = pmha.pmha_forward(g, params, xq, xkv, xkv, "avg")[1]
    pmha.pmha_device_status()
    wa_n = wa.cpu().numpy()
    chunk = 16
    for b0 in range(0, c.B, chunk):
        sl = slice(b0, min(c.B, b0 + chunk))
        ref_out, ref_w = oracle.forward(c.xq[sl], c.xkv[sl], c.xkv[sl], c.params, c.src, c.tgt, c.H, True)
        assert_close(f"output samples {sl.start}-{sl.stop - 1}", out_n[sl], ref_out, c.dt)
        assert_close_weights(f"per-head weights samples {sl.start}-{sl.stop - 1}", w_n[sl], ref_w, c.dt)
        assert_close_weights(f"averaged weights samples {sl.start}-{sl.stop - 1}", wa_n[sl],
                             oracle.average_heads(ref_w), c.dt)
    # every target's weights sum to 1 per head, and their head average too
    for b in range(c.B):
        for h in range(c.H):
            s_bh = np.bincount(c.tgt, weights=w_n[b, :, h].astype(np.float64), minlength=c.L)
            assert np.abs(s_bh - 1.0).max() < 1e-4, (b, h)
        s_b = np.bincount(c.tgt, weights=wa_n[b].astype(np.float64), minlength=c.L)
        assert np.abs(s_b - 1.0).max() < 1e-4, b
    # the weights-only call is bit-identical
    w2 = pmha.pmha_edge_weights(g, params, xq, xkv, "avg")
    pmha.pmha_device_status()
    assert torch.equal(wa, w2)
    g.destroy()


def test_full_skewed_with_padding_mask_every_element():
    # the benchmark's key_padding_mask variant: samples padded at the end
    c = Case.workload(3)
    kpm = synth.padding_mask(np.random.default_rng(7), c.B, c.S)
    g, params, out, w = c.run(DEV, "none", kpm=kpm)
    ref_out, _ = c.oracle(need_weights=False, kpm=kpm)
    assert_close("workload 3 masked output", out.float().cpu().numpy(), ref_out, c.dt)
    g.destroy()


@pytest.mark.parametrize("wid", [3, 4, 5])
def test_full_graph_backward_two_samples(wid):
    # the workload's full graph and widths, two samples: every gradient element
    from tests.test_gpu_backward import _check, _run
    c = Case.workload(wid, batch=2)
    g, got, ref, tensors = _run(c)
    _check(got, ref, tensors, c.dt)
    g.destroy()
