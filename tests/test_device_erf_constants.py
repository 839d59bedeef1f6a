"""The device GeLU evaluates erf with Abramowitz & Stegun eq. 7.1.26 (|error| <= 1.5e-7).

The constants are read from the CUDA header itself, so a mistyped digit there fails this CPU test.
"""
import math
import os
import re

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tensor_transformer_mlp_tp_gb300",
                   "csrc", "ptx.cuh")


def _constants():
    text = open(HDR).read()
    vals = dict(re.findall(r"\b(kP|kA[1-5])\s*=\s*(-?[0-9.]+)f", text))
    return {k: float(v) for k, v in vals.items()}


def test_as_7_1_26_error_bound():
    c = _constants()
    assert set(c) == {"kP", "kA1", "kA2", "kA3", "kA4", "kA5"}
    worst = 0.0
    for i in range(60001):
        z = i * 1e-4
        t = 1.0 / (1.0 + c["kP"] * z)
        poly = t * (c["kA1"] + t * (c["kA2"] + t * (c["kA3"] + t * (c["kA4"] + t * c["kA5"]))))
        worst = max(worst, abs((1.0 - poly * math.exp(-z * z)) - math.erf(z)))
    assert worst <= 1.5e-7
