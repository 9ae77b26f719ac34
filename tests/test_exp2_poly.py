"""The FMA-pipe exp2 (ex2_poly2 in ptx.cuh, C-ABI attn_selftest_exp2_poly),
checked on the CPU against the mathematics.

- Its coefficients are the ones exp2_poly_fit.py derives from 2^f on
  [-1/2, 1/2] (the fit is rerun here and compared with the header).
- The algorithm (clamp to [-126, 127], n = round(x) through x + 1.5 * 2^23,
  f = x - n, degree-4 Horner for 2^f, n added to the exponent field),
  emulated step by step in fp32 with numpy, stays within 2^-18 relative
  error of exp2 in fp64 over [-125, 127], and below 2^-125 (not negative)
  under -126.
"""

import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_47_gb300", "csrc")
BOUND = 2.0 ** -18


def _fit_module():
    spec = importlib.util.spec_from_file_location("exp2_poly_fit", os.path.join(CSRC, "exp2_poly_fit.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def header_coefficients():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    vals = {int(k): float(v) for k, v in re.findall(r"kEx2C(\d) = ([0-9.e+-]+)f", text)}
    return np.array([vals[i] for i in range(5)], dtype=np.float32)


def emulate(x, c):
    """The device algorithm step by step in fp32."""
    x = np.minimum(np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0)), np.float32(127.0))
    magic = np.float32(1.5 * 2.0 ** 23)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic).astype(np.float32)).astype(np.float32)
    q = np.full_like(f, c[4])
    for k in (3, 2, 1, 0):
        q = (q * f + c[k]).astype(np.float32)
    bits = q.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def test_header_coefficients_are_the_fit():
    c = header_coefficients()
    fit = _fit_module().fit()
    assert np.allclose(c, fit, rtol=1e-6, atol=0), (c, fit)


def test_fit_meets_its_bound_on_the_reduced_range():
    mod = _fit_module()
    c = header_coefficients()
    f = np.linspace(-0.5, 0.5, 100001, dtype=np.float32)
    rel = np.abs(mod.horner_f32(c, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)
    assert rel.max() < BOUND


def test_emulated_algorithm_within_bound():
    c = header_coefficients()
    rng = np.random.default_rng(7)
    x = np.concatenate([np.linspace(-125.0, 127.0, 400001), rng.uniform(-125.0, 127.0, 100000),
                        np.arange(-125, 128, dtype=np.float64), np.arange(-125, 127) + 0.5]).astype(np.float32)
    y = emulate(x, c).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < BOUND, float(rel.max())


def test_emulated_algorithm_underflow_and_exact_powers():
    c = header_coefficients()
    low = emulate(np.array([-126.5, -150.0, -1e30, -np.inf], dtype=np.float32), c).astype(np.float64)
    assert np.all(low >= 0.0) and np.all(low < 2.0 ** -125)
    # Integers: f = 0, so 2^n * c0 with c0 within the bound of 1.
    n = np.arange(-120, 120, dtype=np.float32)
    y = emulate(n, c).astype(np.float64)
    assert np.all(np.abs(y / np.exp2(n.astype(np.float64)) - 1.0) < BOUND)
