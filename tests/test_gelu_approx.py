"""The kernels' GELU evaluates erfc by Abramowitz & Stegun, Handbook of
Mathematical Functions, eq. 7.1.26 (host check of the constants as typed in
csrc/epilogue.cuh; the GPU check is test_gpu_parity.test_gelu_grid).

The published bound is |error| <= 1.5e-7 on z >= 0.  This re-evaluates the
same formula in float64 with the constants the kernel uses and checks it
against scipy's erfc, so a mistyped constant fails here.
"""

import os
import re

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "precision_matmul_dg_gb300", "csrc", "epilogue.cuh")


def kernel_constants():
    text = open(SRC).read()
    body = text[text.index("float gelu_erf"):]
    body = body[:body.index("}")]
    vals = dict(re.findall(r"\b(p|a[1-5]) = (-?[0-9.]+)f", body))
    return {k: float(v) for k, v in vals.items()}


def test_constants_meet_the_published_bound():
    c = kernel_constants()
    assert set(c) == {"p", "a1", "a2", "a3", "a4", "a5"}
    z = np.linspace(0.0, 10.0, 200001)
    s = 1.0 / (1.0 + c["p"] * z)
    poly = ((((c["a5"] * s + c["a4"]) * s + c["a3"]) * s + c["a2"]) * s + c["a1"]) * s
    approx = poly * np.exp(-z * z)
    err = np.abs(approx - scipy_special.erfc(z))
    assert err.max() <= 1.5e-7


def test_gelu_form_matches_erf_gelu():
    # t * (1 - q) for t >= 0 and t * q for t < 0, q = erfc(|t|/sqrt 2)/2, is
    # t * Phi(t) = t (1 + erf(t / sqrt 2)) / 2
    t = np.linspace(-12.0, 12.0, 4801)
    q = 0.5 * scipy_special.erfc(np.abs(t) / np.sqrt(2.0))
    form = t * np.where(t >= 0, 1.0 - q, q)
    exact = 0.5 * t * (1.0 + scipy_special.erf(t / np.sqrt(2.0)))
    assert np.allclose(form, exact, rtol=1e-12, atol=1e-15)


def test_folded_form_is_the_same_function():
    # The kernel folds 1/sqrt 2 into p, 1/2 into a1..a5 and evaluates
    # exp(-z^2) as 2^(-t^2 log2(e) / 2): in float64 this is the same value.
    c = kernel_constants()
    t = np.linspace(-12.0, 12.0, 48001)
    z = np.abs(t) / np.sqrt(2.0)
    s = 1.0 / (1.0 + c["p"] * z)
    poly = ((((c["a5"] * s + c["a4"]) * s + c["a3"]) * s + c["a2"]) * s + c["a1"]) * s
    q = 0.5 * poly * np.exp(-z * z)
    kp, ke = c["p"] * 0.70710678118654752, -0.72134752044448170
    s2 = 1.0 / (1.0 + kp * np.abs(t))
    half_poly = ((((0.5 * c["a5"] * s2 + 0.5 * c["a4"]) * s2 + 0.5 * c["a3"]) * s2
                  + 0.5 * c["a2"]) * s2 + 0.5 * c["a1"]) * s2
    q2 = half_poly * np.exp2(t * t * ke)
    assert np.allclose(q2, q, rtol=1e-13, atol=1e-300)
    assert abs(ke + np.log2(np.e) / 2) < 1e-16
