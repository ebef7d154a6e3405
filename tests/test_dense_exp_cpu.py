"""CPU: the FMA-pipe 2^x of the dense-tile kernel (ex2_fma in dense_attn.cu),
restated in float32 numpy from the constants and steps of that source, held
to the precision its result is used in: within half an fp16 step (2^-12
relative) of 2^x wherever 2^x is an fp16 normal or subnormal the softmax
can produce (x in [-24, kLazy + 1/2]), and below the smallest fp16
subnormal further down. Pins the fitted cubic (a wrong or mistyped
coefficient, a dropped term or a wrong exponent shift fails)."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "graph_sparse_head_gb300", "csrc", "dense_attn.cu")


def _coeffs():
    s = open(SRC).read()
    return [np.float32(float(re.search(r"kExpC%d = ([-0-9.e+]+)f" % i, s).group(1))) for i in range(4)]


def _fma(a, b, c):
    # float32 fused multiply-add: the float64 product of two float32 values is exact
    return (a.astype(np.float64) * np.float64(b) + np.asarray(c, np.float64)).astype(np.float32)


def ex2_fma(x):
    c0, c1, c2, c3 = _coeffs()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    f = (x - (t - np.float32(12582912.0)).astype(np.float32)).astype(np.float32)
    p = _fma(f, c3, np.full_like(f, c2))
    p = _fma(p, f, np.full_like(f, c1))
    p = _fma(p, f, np.full_like(f, c0))
    bits = (p.view(np.uint32).astype(np.uint64) + ((t.view(np.uint32).astype(np.uint64) << np.uint64(23)) & np.uint64(0xFFFFFFFF))) & np.uint64(0xFFFFFFFF)
    return bits.astype(np.uint32).view(np.float32)


def test_coefficients_are_the_minimax_cubic_of_2_pow_f():
    f = np.linspace(-0.5, 0.5, 100001).astype(np.float32)
    c0, c1, c2, c3 = _coeffs()
    p = _fma(_fma(_fma(f, c3, np.full_like(f, c2)), f, np.full_like(f, c1)), f, np.full_like(f, c0))
    rel = np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)
    assert rel.max() < 8e-5
    # equioscillation of a minimax fit: the error reaches its bound at both ends
    assert rel[0] > 6e-5 and rel[-1] > 6e-5


def test_within_half_an_fp16_step_where_fp16_resolves_it():
    x = np.linspace(-24.0, 8.5, 2_000_001).astype(np.float32)
    got = ex2_fma(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    assert np.abs(got / want - 1.0).max() < 2.0 ** -12
    # integers are exact up to the cubic's error at f = 0
    xi = np.arange(-24, 9).astype(np.float32)
    assert np.abs(ex2_fma(xi).astype(np.float64) / np.exp2(xi.astype(np.float64)) - 1.0).max() < 8e-5


def test_far_below_the_reference_it_is_negligible_and_finite():
    x = np.concatenate([np.linspace(-125.0, -24.0, 10001), [-1e4, -3e38]]).astype(np.float32)
    y = ex2_fma(x)
    assert np.all(np.isfinite(y)) and np.all(y >= 0) and np.all(y < 2.0 ** -23)
