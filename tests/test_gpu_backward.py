"""GPU parity of pmha_backward (the chain rule of kpnn2 PackedMultiheadAttention,
Notes steps 1-5) against the fp64 oracle's backward, gradient by gradient, on
the same seeded inputs; plus the per-source view it walks, determinism, and
the exact properties (the key bias gets no gradient; inputs that are one
tensor get the sum of their roles' gradients)."""
import numpy as np
import pytest

import oracle
import synth
from tests._cases import TOL, Case, assert_close, half_ulp, rel_err, torch_dtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NAMES_X = ("dquery", "dkey", "dvalue")
NAMES_P = ("dwq", "dwk", "dwv", "dwo", "dbq", "dbk", "dbv", "dbo")


def _run(c, kpm=None, xv=None, add_self_loops=False):
    """GPU backward and oracle backward of sum(out * dout) for a Case."""
    import graph_sparse_head_gb300 as pmha
    rng = np.random.default_rng(c.L + c.S + c.E)
    dout = synth.make_tokens(rng, c.B, c.L, c.E, c.dt)
    params = pmha.Params.from_arrays(c.params, c.H, torch_dtype(c.dt), DEV)
    g = pmha.pmha_build_csr(torch.from_numpy(c.src).to(DEV), torch.from_numpy(c.tgt).to(DEV), c.L, c.S,
                            add_self_loops)
    xq, xkv = c.device_inputs(DEV)
    v = xkv if xv is None else torch.from_numpy(xv).to(DEV).to(torch_dtype(c.dt))
    mask = None if kpm is None else torch.from_numpy(kpm).to(DEV)
    got = pmha.pmha_backward(g, params, xq, xkv, v, torch.from_numpy(dout).to(DEV).to(torch_dtype(c.dt)),
                             key_padding_mask=mask)
    pmha.pmha_device_status()
    src, tgt = c.src, c.tgt
    if add_self_loops:
        src, tgt = oracle.append_self_loops(src, tgt, c.L)
    ref = oracle.backward(c.xq, c.xkv, c.xkv if xv is None else xv, c.params, src, tgt, c.H, dout,
                          key_padding_mask=kpm)
    return g, got, ref, (xq, xkv, v)


def _sum_shared(got, ref, tensors):
    """Reference gradients per distinct input tensor (the GPU writes the sum)."""
    xq, xk, xv = tensors
    refs = {"dquery": ref["dquery"].copy(), "dkey": ref["dkey"].copy(), "dvalue": ref["dvalue"].copy()}
    ptr = {"dquery": xq.data_ptr(), "dkey": xk.data_ptr(), "dvalue": xv.data_ptr()}
    out = {}
    for n in NAMES_X:
        tot = sum(refs[m] for m in NAMES_X if ptr[m] == ptr[n])
        out[n] = tot
    return out


def _check(got, ref, tensors, dt):
    refx = _sum_shared(got, ref, tensors)
    for n in NAMES_X:
        assert_close(n, got[n].float().cpu().numpy(), refx[n], dt)
    for n in NAMES_P:
        if ref[n] is None:
            assert got[n] is None
            continue
        if n == "dbk":
            continue  # zero in exact arithmetic: checked on its own below
        err, rms = rel_err(got[n].cpu().numpy(), ref[n])
        assert err <= TOL[dt] * rms, f"{n}: max-abs {err:.3e} > {TOL[dt]} x RMS {rms:.3e}"
    if ref["dbk"] is not None:
        # the key bias gets no gradient: only rounding remains, far below the query bias's
        assert np.abs(got["dbk"].cpu().numpy()).max() <= TOL[dt] * np.sqrt((ref["dbq"] ** 2).mean())


@pytest.mark.parametrize("wid,B", [(1, 2), (2, 2), (3, 1), (4, 2), (5, 1)])
def test_backward_matches_oracle_workloads(wid, B):
    c = Case.workload(wid, batch=B)
    g, got, ref, tensors = _run(c)
    _check(got, ref, tensors, c.dt)
    g.destroy()


@pytest.mark.parametrize("L,S,nnz,E,H,B,dt,bip", [
    (64, 64, 256, 32, 4, 3, "f32", False),     # 1 channel per lane, d = 8
    (90, 90, 800, 8, 2, 2, "f32", False),       # E < 32
    (130, 70, 900, 64, 4, 2, "f32", True),      # 2 channels per lane
    (257, 257, 3000, 128, 8, 2, "bf16", False),
    (200, 333, 4000, 256, 8, 2, "bf16", True),  # 8 channels per lane, d = 32
    (150, 150, 2000, 512, 16, 1, "bf16", False),  # 16 channels per lane, d = 32
    (60, 600, 15000, 128, 4, 2, "bf16", True),  # ~250 edges per target: split targets
    (600, 60, 15000, 128, 4, 2, "bf16", True),  # ~250 edges per source: split sources
])
def test_backward_shapes_and_dtypes(L, S, nnz, E, H, B, dt, bip):
    rng = np.random.default_rng(L * 31 + S + E)
    src, tgt = synth.uniform_graph(rng, L, S, nnz, min_in_degree=0)
    c = Case(src, tgt, L, S, E, H, B, dt, seed=E + H + 1, bipartite=bip)
    g, got, ref, tensors = _run(c)
    _check(got, ref, tensors, dt)
    g.destroy()


def test_backward_with_mask_and_separate_value():
    rng = np.random.default_rng(41)
    L, S, E, H, B = 300, 500, 128, 8, 2
    src, tgt = synth.bipartite_membership_graph(rng, L, S, 5, 60)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=42, bipartite=True)
    xv = synth.make_tokens(rng, B, S, E, "bf16")
    kpm = synth.scattered_mask(rng, B, S, 0.3)
    g, got, ref, tensors = _run(c, kpm=kpm, xv=xv)
    _check(got, ref, tensors, "bf16")
    # a dropped key receives nothing through attention: its key gradient is exactly 0
    dk = got["dkey"].float().cpu().numpy()
    assert np.all(dk[kpm] == 0.0)
    g.destroy()


@pytest.mark.parametrize("E,H,B", [
    (256, 8, 3),   # 16 lanes a sample, 2 lanes a head; one sample group with an idle slot
    (512, 8, 2),   # 32 lanes a sample, 4 lanes a head
    (256, 16, 5),  # one lane a head; 3 sample groups, the last half idle
])
def test_backward_wide_rows_with_mask(E, H, B):
    # the per-edge ring kernels for rows of 16 and 32 lanes, heads over
    # several lanes, with dropped keys: a dropped key's k gradient is exactly 0
    rng = np.random.default_rng(E + H + B)
    L, S = 180, 400
    src, tgt = synth.bipartite_membership_graph(rng, L, S, 4, 40)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=E * H + B, bipartite=True)
    kpm = synth.scattered_mask(rng, B, S, 0.25)
    g, got, ref, tensors = _run(c, kpm=kpm)
    _check(got, ref, tensors, "bf16")
    dk = got["dkey"].float().cpu().numpy()
    assert np.all(dk[kpm] == 0.0)
    g.destroy()


def test_backward_fully_masked_sample():
    # every key of sample 1 is padding: its targets' records are {+inf, 0}, so
    # the per-edge kernels give that sample exactly zero dq, dk and dv, and
    # its input gradients are exactly zero
    rng = np.random.default_rng(43)
    L, S, E, H, B = 150, 300, 128, 8, 3
    src, tgt = synth.bipartite_membership_graph(rng, L, S, 5, 40)
    c = Case(src, tgt, L, S, E, H, B, "bf16", seed=44, bipartite=True)
    kpm = synth.scattered_mask(rng, B, S, 0.2)
    kpm[1] = True
    g, got, ref, tensors = _run(c, kpm=kpm)
    _check(got, ref, tensors, "bf16")
    for n in ("dquery", "dkey"):
        assert int(torch.count_nonzero(got[n][1])) == 0, n
        assert int(torch.count_nonzero(got[n][0])) > 0, n
    g.destroy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_backward_self_loops_and_no_bias(dt):
    rng = np.random.default_rng(50)
    n, E, H, B = 80, 64, 4, 2
    src, tgt = synth.uniform_graph(rng, n, n, 300, min_in_degree=0)
    c = Case(src, tgt, n, n, E, H, B, dt, seed=51, bias=False)
    g, got, ref, tensors = _run(c, add_self_loops=True)
    _check(got, ref, tensors, dt)
    g.destroy()


def test_shared_input_gets_one_summed_gradient_and_results_are_deterministic():
    import graph_sparse_head_gb300 as pmha
    c = Case.workload(3, batch=1)
    g, got, ref, tensors = _run(c)
    assert got["dquery"] is got["dkey"] is got["dvalue"]
    xq, xkv, v = tensors
    params = pmha.Params.from_arrays(c.params, c.H, torch_dtype(c.dt), DEV)
    rng = np.random.default_rng(c.L + c.S + c.E)
    dout = torch.from_numpy(synth.make_tokens(rng, c.B, c.L, c.E, c.dt)).to(DEV).to(torch_dtype(c.dt))
    again = pmha.pmha_backward(g, params, xq, xkv, v, dout)
    for n in ("dquery",) + NAMES_P:
        if got[n] is not None:
            assert torch.equal(got[n], again[n]), n
    g.destroy()


@pytest.mark.parametrize("wid", [2, 3, 4])
def test_by_source_view_bit_exact(wid):
    import graph_sparse_head_gb300 as pmha
    w = synth.workload(wid)
    src, tgt = synth.make_graph(wid)
    g = pmha.pmha_build_csr(torch.from_numpy(src).to(DEV), torch.from_numpy(tgt).to(DEV), w.query_features,
                            w.key_features)
    srp, target = pmha.pmha_graph_export_by_source(g)
    order = np.lexsort((tgt, src))
    ref_t = tgt[order].astype(np.int32)
    ref_rp = np.concatenate([[0], np.cumsum(np.bincount(src, minlength=w.key_features))]).astype(np.int32)
    assert np.array_equal(srp.cpu().numpy(), ref_rp)
    assert np.array_equal(target.cpu().numpy(), ref_t)
    g.destroy()
