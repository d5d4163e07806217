"""GPU parity of the fused front-end (q/k L2 norm, beta sigmoid, the gated gate from its
pre-activation) against the fp64 oracle of the front-end followed by the recurrence.

Every kernel is covered: the persistent kernel applies the front-end while staging; the
one-CTA-per-unit, d = 64 and fp32 kernels get it as a separate pass; the recurrent kernel
applies it per token (or as a separate pass when asked). Tolerances as for the plain
forward pass: relative L2 2e-2 for bf16, 1e-5 for fp32.
"""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_frontend_inputs
from kda_cases import TOL, run_gpu_fe, run_oracle_fe

pytestmark = pytest.mark.gpu


def _check(x, tag="", **kw):
    o, ht = run_gpu_fe(x, **kw)
    o_r, ht_r = run_oracle_fe(x)
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    e_o, e_h = rel_l2(o, o_r), rel_l2(ht, ht_r)
    print(f"{tag} rel_l2 o={e_o:.3e} ht={e_h:.3e}")
    assert e_o <= TOL[x.dtype], (tag, e_o)
    assert e_h <= TOL[x.dtype], (tag, e_h)
    return o, ht


@pytest.mark.parametrize("gate", ["channel", "head"])
@pytest.mark.parametrize("path", ["fused", "unfused", "one_cta", "recurrent", "recurrent_unfused"])
def test_bf16_d128_all_parts(gate, path):
    # ragged packed sequences with grouped heads: the persistent kernel takes 8 units
    x = make_frontend_inputs((1, 63, 130, 200), 2, 4, 128, 128, seed=201, h0=True, gate=gate,
                             varlen=True)
    kw = dict(fused={}, unfused=dict(unfused_frontend=True), one_cta=dict(one_cta_per_unit=True),
              recurrent=dict(recurrent=True),
              recurrent_unfused=dict(recurrent=True, unfused_frontend=True))[path]
    _check(x, f"{gate} {path}", **kw)


@pytest.mark.parametrize("parts", ["norm", "sigmoid", "gate", "norm+gate"])
def test_parts_switch_independently(parts):
    x = make_frontend_inputs((150, 70), 1, 2, 128, 128, seed=202, h0=True,
                             qk_l2norm="norm" in parts, beta_sigmoid=parts == "sigmoid",
                             gate_act="gate" in parts)
    _check(x, parts)


def test_decay_only_with_front_end():
    x = make_frontend_inputs((190,), 2, 2, 128, 128, seed=203, h0=True, beta=False)
    _check(x, "decay-only")
    _check(x, "decay-only recurrent", recurrent=True)


@pytest.mark.parametrize("d_k,d_v", [(64, 64), (64, 128)])
def test_bf16_d64_separate_pass(d_k, d_v):
    x = make_frontend_inputs((129, 40), 1, 2, d_k, d_v, seed=204, h0=True)
    _check(x, f"d{d_k}x{d_v}")


@pytest.mark.parametrize("gate", ["channel", "head"])
def test_fp32(gate):
    x = make_frontend_inputs((100, 37), 1, 2, 128, 128, seed=205, dtype="f32", h0=True, gate=gate)
    _check(x, f"f32 {gate}")
    _check(x, f"f32 {gate} recurrent", recurrent=True)


def test_large_magnitudes_and_empty_sequences():
    # q, k with |x| ~ 100 (the norm must still bring them to unit length), and
    # sequences of length 0 and 1 among full chunks
    x = make_frontend_inputs((0, 1, 64, 0, 129), 2, 2, 128, 128, seed=206, h0=True, qk_std=9.0,
                             varlen=True)
    _check(x, "large |q|, empty sequences")


def test_fused_agrees_with_separate_pass():
    x = make_frontend_inputs((256, 100), 2, 4, 128, 128, seed=207, h0=True, varlen=True)
    o1, h1 = run_gpu_fe(x)
    o2, h2 = run_gpu_fe(x, unfused_frontend=True)
    # both bf16; the separate pass rounds the normalised q, k to bf16 before the kernel
    e_o, e_h = rel_l2(o1, o2), rel_l2(h1, h2)
    print(f"fused vs separate pass: o={e_o:.3e} ht={e_h:.3e}")
    assert e_o < 1e-2 and e_h < 1e-2


def test_benchmark_shape_sampled_units():
    """The benchmark's shape (B = 2, T = 8192, H = 32, d = 128) through the fused path, in
    the launch configuration of the timed run; five units against the oracle."""
    x = make_frontend_inputs((8192, 8192), 32, 32, 128, 128, seed=208, h0=True)
    o, ht = run_gpu_fe(x)
    units = [(0, 0), (0, 17), (1, 5), (1, 31), (0, 31)]
    ref = run_oracle_fe(x, units=units)
    T = 8192
    for (n, h), (o_u, ht_u) in zip(units, ref):
        e_o = rel_l2(o[n * T:(n + 1) * T, h], o_u)
        e_h = rel_l2(ht[n, h], ht_u)
        print(f"unit ({n},{h}): o={e_o:.3e} ht={e_h:.3e}")
        assert e_o <= TOL["bf16"] and e_h <= TOL["bf16"]
