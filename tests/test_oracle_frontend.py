"""Pins of the front-end oracle (no GPU needed): the q/k normalisation, the beta
sigmoid and the Gated DeltaNet gate against closed forms, library routines and
invariants, and the fused recurrence against a hand-solved one-token case.

A plausible slip — the epsilon outside the square root or missing, exp(A_log) taken as
A_log, the bias added per head instead of per channel (or transposed), a dropped minus
sign, the sigmoid's argument negated, the scale applied before the norm — fails one.
"""

from __future__ import annotations

import math

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_frontend_inputs
from oracle import kda_recurrence
from oracle.frontend import gate, kda_fused_recurrence, l2norm, prepare, sigmoid, softplus


def test_l2norm_closed_forms():
    # (3, 4) has length 5: the result is (0.6, 0.8) scaled by 5 / sqrt(25 + 1e-6)
    y = l2norm(np.array([3.0, 4.0]))
    f = 5.0 / math.sqrt(25.0 + 1e-6)
    assert np.allclose(y, [0.6 * f, 0.8 * f], rtol=0, atol=1e-15)
    # a vector with squared length 1e-6 comes out at length 1 / sqrt(2): the epsilon sits
    # inside the square root, beside the sum of squares
    z = l2norm(np.array([1e-3, 0.0, 0.0]))
    assert abs(np.linalg.norm(z) - 1 / math.sqrt(2)) < 1e-12
    # the zero vector stays zero (no division by zero)
    assert np.array_equal(l2norm(np.zeros(5)), np.zeros(5))


def test_l2norm_against_library_norm_and_axis():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 3, 16))
    y = l2norm(x)
    # against numpy's norm, up to the epsilon's relative effect 1e-6 / (2 |x|^2)
    ref = x / np.linalg.norm(x, axis=-1, keepdims=True)
    assert np.max(np.abs(y - ref)) < 1e-7
    # normalised over the last axis only: each (token, head) row on its own
    assert np.allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-7)
    assert np.allclose(l2norm(10.0 * x), l2norm(x), atol=1e-8)


def test_sigmoid_against_library_and_symmetry():
    from scipy.special import expit

    b = np.linspace(-40, 40, 801)
    assert np.max(np.abs(sigmoid(b) - expit(b))) < 1e-15
    assert sigmoid(np.array(0.0)) == 0.5
    assert np.allclose(sigmoid(b) + sigmoid(-b), 1.0, atol=1e-15)
    assert np.isfinite(sigmoid(np.array([-1000.0, 1000.0]))).all()


def test_softplus_closed_forms():
    assert abs(softplus(np.array(0.0)) - math.log(2.0)) < 1e-15
    x = np.linspace(-30, 30, 601)
    assert np.max(np.abs(softplus(x) - np.logaddexp(0.0, x))) < 1e-14
    # softplus(x) - softplus(-x) = x
    assert np.allclose(softplus(x) - softplus(-x), x, atol=1e-13)
    assert softplus(np.array(800.0)) == 800.0


def _inv_softplus(s):
    return np.log(np.expm1(s))


def test_gate_closed_form_per_head_and_per_channel():
    # choose a so that softplus(a + dt_bias) equals a chosen s: then g = -exp(A_log) * s
    H, d = 3, 5
    A_log = np.log(np.array([0.5, 1.0, 2.0]))
    s_head = np.array([0.01, 0.1, 1.0])
    bias_h = np.array([-4.0, -3.0, -2.0])
    a_head = _inv_softplus(s_head)[None, :] - bias_h[None, :]
    g = gate(a_head, A_log, bias_h)
    assert np.allclose(g, [[-0.005, -0.1, -2.0]], rtol=1e-12, atol=0)
    # per channel: A_log indexes the head, dt_bias the (head, channel) pair
    bias_c = np.arange(H * d, dtype=np.float64).reshape(H, d) * -0.25
    s = np.linspace(0.01, 0.5, H * d).reshape(H, d)
    a_c = (_inv_softplus(s) - bias_c)[None]
    g = gate(a_c, A_log, bias_c)[0]
    assert np.allclose(g, -np.array([0.5, 1.0, 2.0])[:, None] * s, rtol=1e-12, atol=0)
    # no bias: softplus(a) directly; g < 0 for any a
    a = np.linspace(-20, 20, 41)[None, :, None] * np.ones((2, 1, 4))
    g = gate(a, np.zeros(41), None)
    assert (g < 0).all() and np.allclose(g, -np.logaddexp(0.0, a))


def test_disabled_front_end_is_the_plain_recurrence():
    x = make_frontend_inputs((37, 20), 2, 4, 8, 6, dtype="f32", seed=11, h0=True,
                             qk_l2norm=False, beta_sigmoid=False, gate_act=False)
    o_f, h_f = kda_fused_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale,
                                    qk_l2norm=False, beta_sigmoid=False)
    o_r, h_r = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale)
    assert np.array_equal(o_f, o_r) and np.array_equal(h_f, h_r)


@pytest.mark.parametrize("gate_mode", ["channel", "head"])
def test_one_token_closed_form(gate_mode):
    """One token with q orthogonal to k, solved by hand.

    With q = c e_0 and k = c' e_1 (orthogonal), h0 given, and the gate chosen through
    softplus(a + dt_bias) = s so that g = -exp(A_log) s: the erase read sees only row 1 of
    the decayed state and the output sees only row 0, so
        o = scale * c / sqrt(c^2 + 1e-6) * exp(g_0) * h0[0, :].
    The state row 1 becomes exp(g_1) h0[1] + kh_1 * sigmoid(b) * (v - kh_1 exp(g_1) h0[1])
    with kh_1 = c' / sqrt(c'^2 + 1e-6)."""
    d_k, d_v = 4, 3
    c, c2, bl = 3e-3, 2.0, 0.7
    q = np.zeros((1, 1, d_k)); q[0, 0, 0] = c
    k = np.zeros((1, 1, d_k)); k[0, 0, 1] = c2
    v = np.array([[[1.0, -2.0, 0.5]]])
    h0 = np.arange(d_k * d_v, dtype=np.float64).reshape(1, 1, d_k, d_v) / 10.0 - 0.3
    A_log = np.array([math.log(0.8)])
    if gate_mode == "channel":
        s = np.array([0.05, 0.2, 0.01, 0.3])
        dt_bias = np.array([[-3.0, -2.5, -4.0, -1.0]])
        a = (_inv_softplus(s) - dt_bias[0])[None, None, :]
        gv = -0.8 * s
    else:
        s0 = 0.15
        dt_bias = np.array([-3.0])
        a = np.array([[_inv_softplus(s0) - dt_bias[0]]])
        gv = -0.8 * s0 * np.ones(d_k)
    b = np.array([[bl]])
    scale = 0.37
    cu = np.array([0, 1])
    o, ht = kda_fused_recurrence(q, k, v, a, b, h0, cu, scale, A_log=A_log, dt_bias=dt_bias)
    qh0 = c / math.sqrt(c * c + 1e-6)
    kh1 = c2 / math.sqrt(c2 * c2 + 1e-6)
    o_ref = scale * qh0 * math.exp(gv[0]) * h0[0, 0, 0]
    assert np.allclose(o[0, 0], o_ref, rtol=5e-7, atol=1e-9)  # inputs pass as float32
    beta = 1.0 / (1.0 + math.exp(-bl))
    row1 = math.exp(gv[1]) * h0[0, 0, 1]
    u = beta * (v[0, 0] - kh1 * row1)
    assert np.allclose(ht[0, 0, 1], row1 + kh1 * u, rtol=5e-7, atol=1e-8)
    for r in (0, 2, 3):
        assert np.allclose(ht[0, 0, r], math.exp(gv[r]) * h0[0, 0, r], rtol=5e-7, atol=1e-8)


def test_norm_makes_the_result_scale_free_in_q_and_k():
    x = make_frontend_inputs((50,), 2, 2, 16, 8, dtype="f32", seed=12, h0=True)
    args = (x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale)
    kw = dict(A_log=x.A_log, dt_bias=x.dt_bias)
    o1, h1 = kda_fused_recurrence(x.q, x.k, *args, **kw)
    o2, h2 = kda_fused_recurrence(8.0 * x.q, 3.0 * x.k, *args, **kw)
    assert rel_l2(o1, o2) < 1e-6 and rel_l2(h1, h2) < 1e-6
    # without the norm the same rescaling changes the result completely
    o3, _ = kda_fused_recurrence(8.0 * x.q, 3.0 * x.k, *args, qk_l2norm=False, **kw)
    o4, _ = kda_fused_recurrence(x.q, x.k, *args, qk_l2norm=False, **kw)
    assert rel_l2(o3, o4) > 0.1


def test_prepare_parts_switch_independently():
    x = make_frontend_inputs((9,), 1, 2, 4, 4, dtype="f32", seed=13)
    q, k, beta, g = prepare(x.q, x.k, x.beta, x.g, qk_l2norm=False, beta_sigmoid=False)
    assert q is x.q and k is x.k and beta is x.beta and g is x.g
    q, k, beta, g = prepare(x.q, x.k, x.beta, x.g, A_log=x.A_log, dt_bias=x.dt_bias)
    assert np.allclose(np.linalg.norm(q, axis=-1), 1.0, atol=1e-6)
    assert ((beta > 0) & (beta < 1)).all()
    # the recipe keeps the per-token decay in the lower-bounded range [0.9, 1)
    assert (np.exp(g) >= 0.899).all() and (np.exp(g) < 1.0).all()
