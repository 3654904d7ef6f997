"""CPU pins of the software exponential's polynomial (soft_exp2x2 in
common.cuh): the constants in the source reach the stated relative error on
a dense grid when evaluated in FP32 the way the kernel does, p(0) = 1, and
the committed fit reproduces them."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "online_softmax_02_gb300", "csrc")


def _constants():
    src = open(os.path.join(CSRC, "common.cuh")).read()
    return [np.float32(float(re.search(r"kExp2C%d = ([0-9.eE+-]+)f;" % k, src).group(1)))
            for k in (1, 2, 3)]


def _horner32(f):
    c1, c2, c3 = _constants()
    f = f.astype(np.float32)
    p = np.float32(c3) * f + c2
    p = p.astype(np.float32) * f + c1
    p = p.astype(np.float32) * f + np.float32(1)
    return p.astype(np.float32)


def test_poly_relative_error_on_reduced_range():
    f = np.linspace(-0.5, 0.5, 200_001)
    rel = np.abs(_horner32(f).astype(np.float64) / np.exp2(f) - 1)
    assert rel.max() <= 1.02e-4
    assert rel.max() >= 0.9e-4      # the minimax error, not a loose over-estimate


def test_poly_is_one_at_zero():
    assert _horner32(np.array([0.0]))[0] == np.float32(1.0)


def test_fit_reproduces_constants():
    pytest.importorskip("scipy")
    sys.path.insert(0, CSRC)
    try:
        import exp2_poly_fit
    finally:
        sys.path.pop(0)
    c, rel = exp2_poly_fit.fit()
    assert np.allclose(c, _constants(), rtol=1e-5, atol=0)
    assert rel <= 1.02e-4
