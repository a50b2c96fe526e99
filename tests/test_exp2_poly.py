"""The FMA-pipe exponential of the dense kernel's softmax: its coefficients are the minimax fit
that the fitting script derives, and its float32 evaluation (range reduction included) stays
within the fit's relative error of 2^x over the arguments the softmax produces."""

import os
import re

import numpy as np
import pytest

from shared_prefix_kv_decode_gb300 import exp2_poly_fit as E

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "shared_prefix_kv_decode_gb300",
                   "csrc", "tc_util.cuh")


def header_coefficients():
    src = open(HDR).read()
    body = src[src.index("float ex2_poly3(float x)"):]
    body = body[:body.index("return")]
    nums = [float(v) for v in re.findall(r"fmaf\([^;]*?([0-9]\.[0-9]+)f\)", body)]
    c3 = float(re.search(r"fmaf\(([0-9]\.[0-9]+)f, f,", body).group(1))
    # Horner order in the source: (c3, c2), c1, c0
    return [nums[2], nums[1], nums[0], c3]


def test_packed_variant_uses_the_same_coefficients():
    src = open(HDR).read()
    body = src[src.index("uint64_t ex2_poly3_x2(uint64_t x2)"):]
    body = body[:body.index("return")]
    got = sorted(set(float(v) for v in re.findall(r"([0-9]\.[0-9]{6,})f", body)))
    assert got == sorted(header_coefficients()), got


def test_header_matches_fit():
    pytest.importorskip("scipy")
    coef, err = E.fit(3)
    assert err < 8e-5
    hc = header_coefficients()
    assert np.allclose(hc, np.float32(coef).astype(np.float64), rtol=0, atol=1e-7), (hc, coef)


def test_eval_relative_error():
    coef = header_coefficients()
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-30.0, 8.0, 200000), np.linspace(-0.5, 0.5, 10001),
                        np.arange(-40, 9, dtype=np.float64) + 0.5]).astype(np.float32)
    y = E.eval_f32(coef, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() < 8e-5, rel.max()


def test_eval_special():
    coef = header_coefficients()
    x = np.array([0.0, 1.0, -1.0, 8.0, -np.inf, -126.0, -1000.0], dtype=np.float32)
    y = E.eval_f32(coef, x)
    assert abs(y[0] - 1) < 1e-4 and abs(y[1] - 2) < 2e-4 and abs(y[2] - 0.5) < 1e-4 and abs(y[3] - 256) < 0.03
    assert np.all(y[4:] >= 0) and np.all(y[4:] < 1e-37)
