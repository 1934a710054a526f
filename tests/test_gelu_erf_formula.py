"""The erf inside the MLP layer-1 epilogue is Abramowitz & Stegun, "Handbook of Mathematical
Functions", formula 7.1.26.  This reads the constants out of the CUDA source and checks, in
float64, that the formula they make meets the published bound |error| <= 1.5e-7 against
scipy's erf (a mistyped constant breaks it), and that the GELU built on it keeps within
the MLP parity tolerance's scale of exact GELU.
"""
import os
import re

import numpy as np
from scipy.special import erf

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "communication_overlapped_gemm_gb300", "csrc", "tl_gemm_ops.cu")


def constants():
    src = open(SRC).read()
    body = src[src.index("float gelu_erf(float x) {"):]
    body = body[: body.index("\n}\n")]
    p = float(re.search(r"1\.0f \+ ([0-9.]+)f \* z", body).group(1))
    a = [float(v) for v in re.findall(r"(-?[0-9]\.[0-9]+)f", body.split("poly =")[1].split(";")[0])]
    return p, a


def erf_as(x, p, a):
    z = np.abs(x)
    t = 1.0 / (1.0 + p * z)
    poly = sum(ak * t ** (k + 1) for k, ak in enumerate(a))
    return np.sign(x) * (1.0 - poly * np.exp(-z * z))


def test_constants_are_the_published_ones_and_meet_the_bound():
    p, a = constants()
    assert len(a) == 5
    x = np.linspace(-8.0, 8.0, 400001)
    err = np.max(np.abs(erf_as(x, p, a) - erf(x)))
    assert err <= 1.5e-7, err


def test_gelu_on_the_formula_is_close_to_exact():
    p, a = constants()
    x = np.linspace(-12.0, 12.0, 200001)
    g = 0.5 * x * (1.0 + erf_as(x / np.sqrt(2.0), p, a))
    ref = 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))
    assert np.max(np.abs(g - ref)) <= 12.0 * 1.5e-7
