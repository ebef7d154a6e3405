"""Shared helpers of the GPU tests: run the CUDA path through the binding and
the oracle on the same seeded synthetic inputs, and compare."""
from __future__ import annotations

import numpy as np

import synth

# Outputs: max-abs error relative to the RMS of the oracle's output (the
# stated bar), after allowing every element the half unit in the last place
# of its own rounding to the output type: that rounding alone reaches 2.1 % of
# RMS on workload 2 in bf16 (the oracle's output, correctly rounded to bf16,
# misses the bare bar), so no bf16 result could pass without it.
# Weights are compared element by element, relative to the oracle's weight:
# |w - w_ref| <= TOL_w * w_ref + EPS_W. The relative part follows the
# arithmetic: a weight 2^(s - m) / l moves by ln(2) times the error of its
# score, and rounding q and k to the intermediate type perturbs each score by
# a relative 2^-10 (fp16) or 2^-23 (fp32) of its size, so TOL_w = TOL while
# every |score| stays within 16 log2 units (all generated workloads: at most
# about 10) and grows in proportion beyond that (tests that scale the tokens
# up on purpose). EPS_W absorbs weights that underflow (2^-126 flushes to 0).
TOL = {"bf16": 2e-2, "f32": 1e-5}
EPS_W = {"bf16": 1e-7, "f32": 1e-12}
SCORE_SPAN = 16.0
MANTISSA_BITS = {"bf16": 8, "f32": 24}  # significand bits, implicit bit included


def half_ulp(x, dt):
    """Half the spacing of the output type's values at |x| (0 at 0)."""
    _, e = np.frexp(np.abs(np.asarray(x, np.float64)))  # |x| = f 2^e, f in [0.5, 1)
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - MANTISSA_BITS[dt] - 1))


def torch_dtype(dt):
    import torch
    return torch.float32 if dt == "f32" else torch.bfloat16


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    rms = float(np.sqrt((ref ** 2).mean())) if ref.size else 1.0
    return err, rms


def assert_close(name, got, ref, dt):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err, rms = rel_err(got, ref)
    excess = float((np.abs(got - ref) - half_ulp(np.maximum(np.abs(got), np.abs(ref)), dt)).max()) if ref.size else 0
    assert excess <= TOL[dt] * rms, (f"{name}: max-abs error beyond the output rounding {excess:.4e} > {TOL[dt]} x "
                                     f"RMS {rms:.4e} (raw max-abs {err:.4e})")
    return excess / rms


def assert_close_weights(name, got, ref, dt, score_bound=None):
    """Per element: |got - ref| <= TOL_w * ref + EPS_W (see above); score_bound
    is the largest |score| (log2 units) of the compared targets, if known."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = TOL[dt] * max(1.0, (score_bound or 0.0) / SCORE_SPAN)
    if not ref.size:
        return 0.0
    assert np.all(np.isfinite(got)), f"{name}: non-finite weights"
    excess = np.abs(got - ref) - (tol * np.abs(ref) + EPS_W[dt])
    i = int(np.argmax(excess))
    assert excess.flat[i] <= 0.0, (f"{name}: weight {got.flat[i]:.6e} vs oracle {ref.flat[i]:.6e} "
                                   f"(element {i}) beyond {tol:.3g} x w + {EPS_W[dt]:g}")
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(ref > 0, np.abs(got - ref) / ref, 0.0)
    return float(rel.max())


def score_bound(case, src=None, tgt=None):
    """Largest |q_t . k_s| log2(e) / sqrt(d) over the edges and heads of a case,
    from the oracle's projections (a tolerance input, not an expected value)."""
    import oracle
    src = case.src if src is None else np.asarray(src)
    tgt = case.tgt if tgt is None else np.asarray(tgt)
    p = case.params
    d = case.E // case.H
    best = 0.0
    for b in range(case.B):
        q = oracle.linear(case.xq[b], p["wq"], p.get("bq"))
        k = oracle.linear(case.xkv[b], p["wk"], p.get("bk"))
        s = np.einsum("ehc,ehc->eh", q[tgt].reshape(-1, case.H, d), k[src].reshape(-1, case.H, d))
        best = max(best, float(np.abs(s).max()) * 1.4426950408889634 / np.sqrt(d))
    return best


class Case:
    """One seeded problem: graph, tokens and parameters (numpy, rounded to dt)."""

    def __init__(self, src, tgt, L, S, E, H, B, dt, seed, bipartite=False, bias=True, xq=None, xkv=None,
                 params=None):
        self.src, self.tgt = np.asarray(src, np.int64), np.asarray(tgt, np.int64)
        self.L, self.S, self.E, self.H, self.B, self.dt = L, S, E, H, B, dt
        rng = np.random.default_rng(seed)
        self.params = params if params is not None else synth.make_params(rng, E, dt, bias=bias)
        self.xq = xq if xq is not None else synth.make_tokens(rng, B, L, E, dt)
        if bipartite or L != S:
            self.xkv = xkv if xkv is not None else synth.make_tokens(rng, B, S, E, dt)
        else:
            self.xkv = self.xq

    @staticmethod
    def workload(wid, batch=None):
        w = synth.workload(wid)
        src, tgt = synth.make_graph(wid)
        xq, xkv, params = synth.make_inputs(wid, batch)
        B = xq.shape[0]
        return Case(src, tgt, w.query_features, w.key_features, w.embed_dim, w.num_heads, B, w.dtype, 0,
                    bipartite=w.bipartite, xq=xq, xkv=xkv if xkv is not None else xq, params=params)

    # ------------------------------------------------------------ CUDA path
    def device_inputs(self, dev):
        import torch
        tdt = torch_dtype(self.dt)
        xq = torch.from_numpy(self.xq).to(dev).to(tdt)
        xkv = xq if self.xkv is self.xq else torch.from_numpy(self.xkv).to(dev).to(tdt)
        return xq, xkv

    def run(self, dev, wmode="none", add_self_loops=False, graph=None, kpm=None):
        """kpm: (B, S) bool numpy key_padding_mask or None."""
        import torch
        import graph_sparse_head_gb300 as pmha
        params = pmha.Params.from_arrays(self.params, self.H, torch_dtype(self.dt), dev)
        if graph is None:
            graph = pmha.pmha_build_csr(torch.from_numpy(self.src).to(dev), torch.from_numpy(self.tgt).to(dev),
                                        self.L, self.S, add_self_loops)
        xq, xkv = self.device_inputs(dev)
        mask = None if kpm is None else torch.from_numpy(np.ascontiguousarray(kpm, dtype=np.bool_)).to(dev)
        out, w = pmha.pmha_forward(graph, params, xq, xkv, xkv, wmode, key_padding_mask=mask)
        pmha.pmha_device_status()
        return graph, params, out, w

    # ------------------------------------------------------------ oracle
    def oracle(self, need_weights=True, src=None, tgt=None, kpm=None):
        import oracle
        src = self.src if src is None else src
        tgt = self.tgt if tgt is None else tgt
        return oracle.forward(self.xq, self.xkv, self.xkv, self.params, src, tgt, self.H, need_weights,
                              key_padding_mask=kpm)
