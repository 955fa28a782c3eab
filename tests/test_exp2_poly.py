"""The polynomial exp2 of the forward kernel's softmax (Cody-Waite reduction
plus a minimax polynomial), checked on the host: the coefficients written in
the CUDA source are the ones the Remez generator produces, and the float32
evaluation, modelled step for step, stays within its relative-error bound
against exact 2^x over the whole range the softmax can feed it."""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_76_gb300", "csrc")


def _generator():
    spec = importlib.util.spec_from_file_location("exp2_minimax", os.path.join(CSRC, "exp2_minimax.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _source_coefficients(degree):
    src = open(os.path.join(CSRC, "fa_common.cuh")).read()
    body = src[src.index("__device__ __forceinline__ float2 exp2_poly2"):]
    branch = body.split("if constexpr (DEG == 3) {")[1]
    part = branch.split("} else {")[0] if degree == 3 else branch.split("} else {")[1].split("}")[0]
    vals = [float(v) for v in re.findall(r"make_float2\(([0-9.e+-]+)f, \1f\)", part)]
    # Horner from the top: the literals appear as c_n, c_{n-1}, ..., c_0
    return np.array(vals[::-1], dtype=np.float32)


@pytest.mark.parametrize("degree", [2, 3])
def test_source_coefficients_match_generator(degree):
    gen = _generator()
    c_src = _source_coefficients(degree)
    c_gen = gen.coefficients_f32(degree)
    assert c_src.shape == (degree + 1,)
    np.testing.assert_array_equal(c_src, c_gen)


@pytest.mark.parametrize("degree,bound", [(2, 1.8e-3), (3, 8.0e-5)])
def test_float32_evaluation_error(degree, bound):
    gen = _generator()
    c = gen.coefficients_f32(degree)
    # the softmax feeds x = s*c - m <= TAU (8) and anything below; values under
    # -126 are clamped there
    x = np.concatenate([np.linspace(-125.5, 8.0, 1_000_001), np.linspace(-1.0, 1.0, 100_001)]).astype(np.float32)
    y = gen.eval_exp2_f32(x, c).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() < bound
    # integers reduce to f = 0: the result is 2^n times p(0) exactly
    xi = np.arange(-125, 9, dtype=np.float32)
    yi = gen.eval_exp2_f32(xi, c).astype(np.float64)
    np.testing.assert_allclose(yi / np.exp2(xi.astype(np.float64)), np.float64(c[0]), rtol=0, atol=0)


def test_clamp_and_minus_infinity():
    gen = _generator()
    c = gen.coefficients_f32(3)
    y = gen.eval_exp2_f32(np.array([-np.inf, -1000.0, -126.0], dtype=np.float32), c)
    assert np.all(np.isfinite(y)) and np.all(y > 0)
    assert np.all(y <= np.float32(2.0**-125))  # stands in for an underflow to zero
    assert y[0] == y[1] == y[2]


def test_remez_equioscillation():
    """The minimax error alternates in sign with equal magnitude at degree+2
    points, the defining property of the best approximation."""
    gen = _generator()
    for degree in (2, 3):
        cf, err = gen.remez(degree)
        x = np.linspace(gen.LO, gen.HI, 200_001)
        e = np.polynomial.polynomial.polyval(x, cf) / 2.0**x - 1.0
        sign = np.sign(e)
        runs = np.split(np.arange(len(x)), np.flatnonzero(np.diff(sign)) + 1)
        peaks = np.array([np.max(np.abs(e[r])) for r in runs])
        assert len(runs) >= degree + 2
        assert peaks.max() == pytest.approx(err, rel=1e-9)
        assert peaks[np.argsort(peaks)[-(degree + 2):]].min() > 0.99 * err
