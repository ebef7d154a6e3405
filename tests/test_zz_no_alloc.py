"""GPU: pmha_forward_noalloc, the forward pass for callers that cannot
allocate device memory at call time (their allocator owns the device, or
cudaMalloc / cudaFree may not run where they call the layer). It takes its
workspace from a fixed scratch array inside the library instead of from the
caller. Called here through the C ABI, twice in a row: both calls must equal
pmha_forward's results bit for bit (the same kernels run on the same inputs,
only the workspace differs), and the first is also held to the oracle at the
tolerance the other parity tests use.
The file name sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests._cases import Case, assert_close, assert_close_weights

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _noalloc(lib, g, p, xq, xkv, out, wmode, w):
    import graph_sparse_head_gb300 as pmha
    st = lib.pmha_forward_noalloc(g.handle, ctypes.byref(p), xq.data_ptr(), xkv.data_ptr(), xkv.data_ptr(), None,
                                  xq.shape[0], out.data_ptr(), pmha.WMODES[wmode],
                                  None if w is None else w.data_ptr(), torch.cuda.current_stream().cuda_stream)
    pmha._lib.check(st, "pmha_forward_noalloc")


@pytest.mark.parametrize("wid,B,wmode", [(1, 2, "per_head"), (2, 4, "avg"), (4, 1, "none")])
def test_noalloc_matches_forward_on_two_calls(wid, B, wmode):
    import graph_sparse_head_gb300 as pmha
    lib = pmha._lib.load()
    c = Case.workload(wid, batch=B)
    g, params, ref_out, ref_w = c.run(DEV, wmode)
    p = params.as_struct()
    assert lib.pmha_forward_workspace_size(g.handle, ctypes.byref(p), B, pmha.WMODES[wmode]) <= (64 << 20)
    xq, xkv = c.device_inputs(DEV)
    oracle_out, oracle_w = c.oracle(need_weights=ref_w is not None)
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        w = None if ref_w is None else torch.full_like(ref_w, float("nan"))
        _noalloc(lib, g, p, xq, xkv, out, wmode, w)
        pmha.pmha_device_status()
        assert torch.equal(out, ref_out), f"call {call}: output differs from pmha_forward"
        if w is not None:
            assert torch.equal(w, ref_w), f"call {call}: weights differ from pmha_forward"
        if call == 0:
            assert_close("noalloc output", out.float().cpu().numpy(), oracle_out, c.dt)
            if w is not None:
                wo = oracle_w if wmode == "per_head" else oracle.average_heads(oracle_w)
                assert_close_weights("noalloc weights", w.cpu().numpy(), wo, c.dt)
    g.destroy()


def test_noalloc_rejects_problems_beyond_its_scratch():
    import graph_sparse_head_gb300 as pmha
    lib = pmha._lib.load()
    c = Case.workload(3, batch=4)  # needs about 100 MB of workspace
    g, params, ref_out, _ = c.run(DEV, "none")
    p = params.as_struct()
    xq, xkv = c.device_inputs(DEV)
    out = torch.empty_like(ref_out)
    st = lib.pmha_forward_noalloc(g.handle, ctypes.byref(p), xq.data_ptr(), xkv.data_ptr(), xkv.data_ptr(), None, 4,
                                  out.data_ptr(), 0, None, torch.cuda.current_stream().cuda_stream)
    assert pmha._lib.STATUS_NAMES[st] == "PMHA_ERR_WORKSPACE"
    assert b"scratch" in lib.pmha_last_error()
    g.destroy()
