"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: every output element against the oracle where its fp64
forward finishes in seconds (workloads 1, 2, 3, 5), and sampled rows computed
one by one by the oracle for the bipartite workload 4, plus properties that
hold at any size (weights sum to 1, edge_weights == forward weights)."""
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


def test_full_bipartite_sampled_rows_and_weights():
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(4)
    g, params, out, w = c.run(DEV, "avg")
    out_n = out.float().cpu().numpy()
    w_n = w.cpu().numpy()
    deg = np.bincount(c.tgt, minlength=c.L)
    rng = np.random.default_rng(4)
    rows = [(0, int(np.argmax(deg))), (c.B - 1, int(np.argmin(deg))), (c.B - 1, c.L - 1)]
    rows += [(int(b), int(t)) for b, t in zip(rng.integers(0, c.B, 40), rng.integers(0, c.L, 40))]
    ref = oracle.forward_rows(c.xq, c.xkv, c.xkv, c.params, c.src, c.tgt, c.H, rows)
    got_o = np.stack([out_n[b, t] for b, t in rows])
    ref_o = np.stack([r[0] for r in ref])
    assert_close("sampled output rows", got_o, ref_o, "bf16")
    got_w = np.concatenate([w_n[b, r[1]] for (b, t), r in zip(rows, ref)])
    ref_w = np.concatenate([oracle.average_heads(r[2]) for r in ref])
    assert_close_weights("sampled avg weights", got_w, ref_w, "bf16")
    # every target's averaged weights sum to 1
    sums = np.zeros((c.B, c.L))
    np.add.at(sums, (slice(None), c.tgt), w_n.astype(np.float64))
    assert np.abs(sums - 1.0).max() < 1e-4
    # weights-only call is bit-identical
    xq, xkv = c.device_inputs(DEV)
    w2 = pmha.pmha_edge_weights(g, params, xq, xkv, "avg")
    pmha.pmha_device_status()
    assert torch.equal(w, w2)
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
