"""The Gaussian selection's normal tail: Phi(-x) = phi(x) R(x) with the Mills
ratio R in the rational form t P(t), t = 1 / (1 + x / 4), whose coefficients
csrc/mills_ratio.h holds.  Evaluated here in fp32 exactly as the kernel does
(Horner in fp32 FMA order), against scipy's erfcx: the relative error of R,
and of the resulting Phi, stays below 6e-7 over the range where phi(x) is a
normal fp32 number."""
from __future__ import annotations

import os
import re

import numpy as np
from scipy.special import erfc, erfcx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "sparse_long_context_08_b300", "csrc", "mills_ratio.h")


def _coefficients():
    text = open(HDR).read()
    cmap = float(re.search(r"kMillsMap = ([-0-9.e]+)f", text).group(1))
    arr = re.search(r"kMillsP\[\d+\] = \{([^}]*)\}", text).group(1)
    coef = np.array([float(v.strip().rstrip("f")) for v in arr.split(",")], dtype=np.float32)
    return np.float32(cmap), coef


def _fma32(a, b, c):
    # one rounding, as fmaf: the fp64 product-sum of fp32 inputs is exact to
    # well below fp32 resolution, then rounded once
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _mills32(x):
    cmap, p = _coefficients()
    x = x.astype(np.float32)
    t = (np.float32(1.0) / _fma32(np.full_like(x, cmap), x, np.ones_like(x))).astype(np.float32)
    acc = np.full_like(x, p[-1])
    for c in p[-2::-1]:
        acc = _fma32(acc, t, np.full_like(x, c))
    return (t * acc).astype(np.float32)


def test_mills_ratio_relative_error():
    x = np.concatenate([np.linspace(0.0, 13.0, 400001), np.geomspace(1e-6, 13.0, 20001)])
    x32 = x.astype(np.float32)
    ref = np.sqrt(np.pi / 2) * erfcx(x32.astype(np.float64) / np.sqrt(2))
    rel = np.abs(_mills32(x32).astype(np.float64) - ref) / ref
    assert rel.max() < 6e-7, rel.max()


def test_tail_probability_matches_erfc():
    x = np.linspace(0.0, 9.0, 90001).astype(np.float32)
    phi = np.exp(-0.5 * x.astype(np.float64) ** 2) / np.sqrt(2 * np.pi)
    tail = phi * _mills32(x).astype(np.float64)
    ref = 0.5 * erfc(x.astype(np.float64) / np.sqrt(2))
    assert np.max(np.abs(tail - ref) / ref) < 6e-7
    # Phi(u) for u >= 0 is 1 - tail: the tail is at most 1/2, so its absolute
    # error is at most half the relative bound
    assert np.max(np.abs((1 - tail) - (1 - ref))) < 3e-7


def test_coefficients_reproduce_from_the_generator():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "gen_mills_ratio", os.path.join(ROOT, "sparse_long_context_08_b300", "csrc",
                                        "gen_mills_ratio.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    coef, err = gen.fit()
    _, committed = _coefficients()
    assert err < 1e-7
    assert np.array_equal(coef.astype(np.float32), committed)
