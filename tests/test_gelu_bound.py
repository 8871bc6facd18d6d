"""The epilogue's GELU arithmetic against the error bound the GPU tolerance relies on.

The kernels evaluate erf-GELU in fp32 with Abramowitz & Stegun 7.1.28 (see
`csrc/gelu.cuh`); `tests/helpers.py` allows g = 1e-6 of |v| for that evaluation on the bias
part of the pre-activation.  This test reads the coefficients out of the CUDA source, replays
both forms (the scalar one for fp32 outputs, the packed one for bf16 outputs) in fp32 with
numpy, with the hardware reciprocal taken anywhere within one unit in the last place, and
checks the error against the exact erf-GELU (scipy, fp64) over [-8, 8].  It runs no device
code: it pins the stated bounds, so that a change of coefficients or of the evaluation order
that breaks them fails here on the CPU.
"""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")

GELU_CUH = os.path.join(os.path.dirname(__file__), "..", "convolution_forward_implicit_gb300", "csrc", "gelu.cuh")
F32 = np.float32


def _body(src: str, head: str) -> str:
    i = src.index(head)
    return src[i:src.index("\n}\n", i)]


def _coeffs():
    src = open(GELU_CUH).read()
    scalar = _body(src, "__device__ __forceinline__ float gelu(float v)")
    packed = _body(src, "__device__ __forceinline__ void gelu2(float& a, float& b)")
    num = r"(-?[0-9.]+(?:e[-+]?[0-9]+)?)f"
    # scalar: y = fmaf(z, c6, c5); then y = fmaf(z, y, c) for c5..c0
    s = [float(x) for x in re.findall(r"fmaf\(z, " + num + ", " + num + r"\)", scalar)[0]]
    s += [float(x) for x in re.findall(r"fmaf\(z, y, " + num + r"\)", scalar)]
    scale = float(re.findall(r"fabsf\(v\) \* " + num, scalar)[0])
    # packed: the first pair of constants, then one constant pair per Horner step
    p = [float(x) for x in re.findall(r"f2pk\(" + num + ", " + r"-?[0-9.]+(?:e[-+]?[0-9]+)?f\)", packed)]
    return scale, s, p


def _fma(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F32)


def _rcp(y, ulp):
    r = (F32(1) / y).astype(F32)
    if ulp:
        r = np.nextafter(r, F32(np.inf) if ulp > 0 else F32(0)).astype(F32)
    return r


def _scalar(v, scale, c, ulp):
    z = (np.abs(v) * F32(scale)).astype(F32)
    y = _fma(z, F32(c[0]), F32(c[1]))
    for k in c[2:]:
        y = _fma(z, y, F32(k))
    for _ in range(4):
        y = (y * y).astype(F32)
    return _fma((F32(-0.5) * np.abs(v)).astype(F32), _rcp(y, ulp), np.maximum(v, F32(0)))


def _packed(v, c, ulp):
    u = (-np.abs(v)).astype(F32)
    y = _fma(u, F32(c[0]), F32(c[1]))
    for k in c[2:]:
        y = _fma(u, y, F32(k))
    for _ in range(4):
        y = (y * y).astype(F32)
    return _fma(u, _rcp(y, ulp), np.maximum(v, F32(0)))


def _worst(fn):
    v = np.linspace(-8.0, 8.0, 400001).astype(F32)
    v = v[v != 0]
    exact = 0.5 * v.astype(np.float64) * (1.0 + scipy_special.erf(v.astype(np.float64) / np.sqrt(2.0)))
    return max(float(np.max(np.abs(fn(v, ulp).astype(np.float64) - exact) / np.abs(v.astype(np.float64))))
               for ulp in (0, 1, -1))


def test_coefficients_are_found():
    scale, s, p = _coeffs()
    assert abs(scale - 2 ** -0.5) < 1e-7
    assert len(s) == 7 and s[-1] == 1.0      # a6 .. a1 and the constant 1 of A&S 7.1.28
    assert len(p) == 7                       # the same polynomial, folded, in -|v|
    # folding: coefficient k of the packed form is (-1)^k 2^(1/16) a_k / sqrt(2)^k
    for k, (a, b) in enumerate(zip(reversed(s), reversed(p))):
        assert b == pytest.approx((-1) ** k * 2 ** (1 / 16) * a * 2 ** (-k / 2), rel=2e-7)


def test_scalar_form_within_the_stated_bound():
    scale, s, _ = _coeffs()
    err = _worst(lambda v, ulp: _scalar(v, scale, s, ulp))
    assert err < 9.5e-7          # the bound stated in gelu.cuh
    assert err < 1e-6            # GELU_EVAL in the GPU tolerance


def test_packed_form_within_the_stated_bound():
    _, _, p = _coeffs()
    err = _worst(lambda v, ulp: _packed(v, p, ulp))
    assert err < 1.25e-6         # the bound stated in gelu.cuh; far below bf16 rounding (2^-9)


def test_a_dropped_coefficient_breaks_the_bound():
    """The check has teeth: the scalar form without its a6 term misses the bound."""
    scale, s, _ = _coeffs()
    broken = [0.0] + s[1:]
    assert _worst(lambda v, ulp: _scalar(v, scale, broken, ulp)) > 1e-6
