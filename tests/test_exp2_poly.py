"""The FMA-pipe exp2 of the CUDA kernels, emulated step by step in fp32 numpy,
stays within its stated relative-error bound against 2^x (CPU only).

The kernel function (csrc/ptx.cuh, exp2_poly) is: clamp x at -125, round to
the nearest integer j with the 1.5*2^23 trick, f = x - j, Horner degree-4
polynomial in f, add j to the exponent bits, 0 below -125.  The constants are
read from the CUDA source so this test checks what the kernels compile.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "tiled_exact_attention_fa2_gb300", "csrc", "ptx.cuh")


def _coefficients():
    body = open(SRC).read()
    body = body[body.index("float exp2_poly(float x)"):]
    body = body[:body.index("return x < -125.f")]
    c = [float(v) for v in re.findall(r"fmaf\(([0-9.e-]+)f, f, ([0-9.e-]+)f\)", body)[0]]
    rest = [float(v) for v in re.findall(r"fmaf\(p, f, ([0-9.e-]+)f\)", body)]
    return [c[0], c[1]] + rest  # highest degree first


def exp2_poly_emulated(x):
    x = np.asarray(x, dtype=np.float32)
    xc = np.maximum(x, np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (xc + magic).astype(np.float32)
    j = (t - magic).astype(np.float32)
    f = (xc - j).astype(np.float32)
    cs = [np.float32(v) for v in _coefficients()]
    p = cs[0]
    for ck in cs[1:]:
        p = (p * f + ck).astype(np.float32)  # fmaf: exact product then one rounding; numpy rounds twice
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    r = bits.view(np.float32)
    return np.where(x < -125.0, np.float32(0.0), r)


def test_coefficients_parse():
    assert len(_coefficients()) == 5
    assert _coefficients()[-1] == 1.0


def test_relative_error_bound():
    x = np.concatenate([np.linspace(-125, 64, 2_000_001, dtype=np.float32),
                        np.float32([0, -0.5, 0.5, -1, 1, 8, -8])])
    got = exp2_poly_emulated(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1)
    assert rel.max() < 1e-5, rel.max()


def test_exact_points_and_underflow():
    assert exp2_poly_emulated(np.float32(0.0)) == 1.0
    assert exp2_poly_emulated(np.float32(-126.0)) == 0.0
    assert exp2_poly_emulated(np.float32(-np.inf)) == 0.0
    for k in range(-20, 21):
        v = float(exp2_poly_emulated(np.float32(k)))
        assert abs(v / 2.0 ** k - 1) < 1e-6
