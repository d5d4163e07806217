"""Constants written into the kernels, checked on the host: the polynomial the d = 128
kernels' front-end uses for log(1 + t) on [0, 1] is read out of its source and evaluated
in float32 against numpy's log1p (worst relative error below 5e-7), and the fit script
beside it regenerates the same coefficients."""

from __future__ import annotations

import os
import re
import subprocess
import sys

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "chunkwise_gated_linear_gb300", "csrc")


def _coefficients():
    src = open(os.path.join(CSRC, "tc_util.cuh"), encoding="utf-8").read()
    body = re.search(r"float log1p_01\(float t\) \{(.*?)\n\}", src, flags=re.S).group(1)
    return [float(v) for v in re.findall(r"([-+]?\d\.\d+e[-+]\d+)f", body)]


def test_log1p_polynomial_accuracy_in_float32():
    c = np.array(_coefficients(), dtype=np.float32)
    assert len(c) == 8
    t = np.linspace(0.0, 1.0, 200001, dtype=np.float32)
    p = np.full_like(t, c[0])
    for a in c[1:]:
        p = (p * t + a).astype(np.float32)  # Horner in float32, as the kernel does
    y = (p * t).astype(np.float64)
    ref = np.log1p(t.astype(np.float64))
    rel = np.abs(y - ref)[1:] / ref[1:]
    assert rel.max() < 5e-7, rel.max()
    assert y[0] == 0.0


def test_fit_script_reproduces_the_coefficients():
    out = subprocess.run([sys.executable, os.path.join(CSRC, "fit_log1p.py")], capture_output=True,
                         text=True, check=True).stdout.splitlines()[0]
    fitted = [float(v.rstrip("f")) for v in out.split(", ")]
    assert np.allclose(fitted, _coefficients(), rtol=1e-7, atol=0)
