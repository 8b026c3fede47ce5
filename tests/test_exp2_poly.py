"""The FMA-pipe 2^x of the optional polynomial exponential (KDA_EXP2_POLY), on CPU.

The device function (ex2_poly in the kernels' common header) reduces x to n + f with
n = round(x) by the 1.5 * 2^23 rounding trick and f in [-1/2, 1/2], evaluates the fitted
polynomial for 2^f in Horner form with fused multiply-adds, and adds n to the exponent
field. This test emulates those float32 steps with numpy (each fused multiply-add as one
rounding of the exact float64 result) and checks the error bound against exact 2^x, the
special values, and that the committed coefficients are the generator's output.
"""
from __future__ import annotations

import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "chunked_gated_delta_02_gb300", "csrc")


def _coefficients():
    text = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    c = [float(m) for m in re.findall(r"kExp2PolyC\d = ([-+0-9.e]+)f;", text)]
    bound = float(re.search(r"kExp2PolyMaxRelErr = ([-+0-9.e]+)f;", text).group(1))
    return np.array(c, np.float32), bound


def _fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def ex2_poly_emulated(x):
    c, _ = _coefficients()
    x = np.asarray(x, np.float32)
    xc = np.maximum(x, np.float32(-126.0))
    M = np.float32(12582912.0)
    t = (xc + M).astype(np.float32)
    f = (xc - (t - M).astype(np.float32)).astype(np.float32)
    p = np.full_like(f, c[5])
    for j in (4, 3, 2, 1, 0):
        p = _fma32(p, f, np.full_like(f, c[j]))
    n = t.view(np.int32).astype(np.int64) - 0x4B400000
    bits = (p.view(np.int32).astype(np.int64) + (n << 23)).astype(np.int32)
    r = bits.view(np.float32)
    return np.where(x < -126.0, np.float32(0.0), r)


def test_coefficients_are_the_generators_output():
    spec = importlib.util.spec_from_file_location("gen_exp2_poly", os.path.join(CSRC, "gen_exp2_poly.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    c, bound = _coefficients()
    fitted = gen.fit().astype(np.float32)
    assert np.array_equal(fitted, c)
    assert c[0] == 1.0
    assert abs(gen.max_rel_error(c) - bound) <= 1e-3 * bound


def test_relative_error_bound():
    # polynomial error (header bound) plus the rounding of five float32 fused multiply-adds,
    # damped by |f| <= 1/2 in Horner form: below 3e-7 relative over the whole range used
    _, bound = _coefficients()
    x = np.concatenate([np.linspace(-126.0, 0.0, 400001), np.linspace(0.0, 20.0, 100001),
                        np.random.default_rng(0).uniform(-8.0, 0.0, 200000)]).astype(np.float32)
    got = ex2_poly_emulated(x).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(got / exact - 1.0)
    assert bound < 1.2e-7
    assert rel.max() < 3e-7, rel.max()


def test_special_values():
    ints = np.arange(-126, 30, dtype=np.float32)
    assert np.array_equal(ex2_poly_emulated(ints).astype(np.float64), np.exp2(ints.astype(np.float64)))
    assert np.all(ex2_poly_emulated(np.array([-126.5, -200.0, -1e30], np.float32)) == 0.0)
    half = ex2_poly_emulated(np.array([-0.5, 0.5], np.float32)).astype(np.float64)
    assert np.allclose(half, [2 ** -0.5, 2 ** 0.5], rtol=3e-7, atol=0)
