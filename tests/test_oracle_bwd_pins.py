"""Pins of the backward oracle (no GPU needed).

The gradients are checked against what mathematics fixes independently of the adjoint
code: central finite differences of the forward oracle on every input element of tiny
problems (per-channel and per-head gates, decay-only, grouped heads, ragged and empty
sequences, with and without h0 and dht), the closed-form gradients of the parallel
retention form, and the pass-through of an empty sequence.
"""

from __future__ import annotations

import numpy as np
import pytest

from inputs import make_inputs
from oracle import kda_recurrence, kda_recurrence_bwd


def _loss(x, do, dht, **over):
    args = dict(q=x.q, k=x.k, v=x.v, g=x.g, beta=x.beta, h0=x.h0)
    args.update(over)
    o, ht = kda_recurrence(args["q"], args["k"], args["v"], args["g"], args["beta"], args["h0"],
                           x.cu_seqlens, x.scale)
    L = float(np.sum(o * do.astype(np.float64)))
    if dht is not None:
        L += float(np.sum(ht * dht.astype(np.float64)))
    return L


def _fd(x, do, dht, name, h=1e-3):
    """Central differences of the loss in every element of input `name` (float32 steps,
    exact denominators)."""
    base = getattr(x, name).astype(np.float32)
    grad = np.zeros(base.shape)
    flat = base.reshape(-1)
    for i in range(flat.size):
        p, m = flat.copy(), flat.copy()
        p[i] = np.float32(flat[i] + h)
        m[i] = np.float32(flat[i] - h)
        Lp = _loss(x, do, dht, **{name: p.reshape(base.shape)})
        Lm = _loss(x, do, dht, **{name: m.reshape(base.shape)})
        grad.reshape(-1)[i] = (Lp - Lm) / (float(p[i]) - float(m[i]))
    return grad


def _case(kind):
    if kind == "channel":
        x = make_inputs((5, 0, 7), 1, 2, 4, 3, dtype="f32", seed=31, h0=True)
    elif kind == "head":
        x = make_inputs((6, 5), 1, 2, 4, 3, dtype="f32", seed=32, h0=True, gate="head")
    elif kind == "decay_only":
        x = make_inputs((6, 4), 2, 2, 3, 4, dtype="f32", seed=33, h0=True, beta=False)
    else:  # no h0, no dht
        x = make_inputs((9,), 1, 1, 4, 2, dtype="f32", seed=34, h0=False)
    rng = np.random.default_rng(7)
    do = rng.standard_normal(x.v.shape).astype(np.float32)
    dht = None
    if kind != "bare":
        dht = rng.standard_normal((x.N, x.H_v, x.d_k, x.d_v)).astype(np.float32)
    return x, do, dht


@pytest.mark.parametrize("kind", ["channel", "head", "decay_only", "bare"])
def test_gradients_match_central_differences(kind):
    x, do, dht = _case(kind)
    r = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dht, x.cu_seqlens, x.scale)
    names = ["q", "k", "v", "g"] + (["beta"] if x.beta is not None else []) + (["h0"] if x.h0 is not None else [])
    key = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    for name in names:
        fd = _fd(x, do, dht, name)
        an = r[key[name]]
        err = np.max(np.abs(fd - an))
        scale = max(np.max(np.abs(an)), 1e-12)
        print(f"{kind} d{name}: max |fd - analytic| = {err:.2e} (max |grad| {scale:.2e})")
        assert err <= 2e-5 * scale + 1e-9, (kind, name, err, scale)
    if x.beta is None:
        assert r["dbeta"] is None


def test_retention_closed_form():
    """Decay-only with one constant scalar gate log(alpha) and no initial state is the
    retention form O = scale (Q K^T * D) V, D[t, s] = alpha^(t - s) for s <= t; its
    gradients are scale (Q K^T * D)^T dO, scale (dO V^T * D) K and scale (dO V^T * D)^T Q,
    for the gate of token r scale sum over s < r <= t of (q_t . k_s)(dO_t . v_s) D[t, s],
    and for the initial state scale sum_t alpha^(t + 1) q_t dO_t^T."""
    T, dk, dv, alpha = 11, 5, 4, 0.83
    rng = np.random.default_rng(9)
    q = rng.standard_normal((T, 1, dk)).astype(np.float32)
    k = rng.standard_normal((T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    do = rng.standard_normal((T, 1, dv)).astype(np.float32)
    g = np.full((T, 1), np.float32(np.log(alpha)), dtype=np.float32)
    scale = 0.7
    cu = np.array([0, T])
    r = kda_recurrence_bwd(q, k, v, g, None, None, do, None, cu, scale)
    a = float(np.exp(np.float64(g[0, 0])))
    ti, si = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    D = np.where(si <= ti, a ** (ti - si).astype(np.float64), 0.0)
    Q, K, V, dO = (z[:, 0].astype(np.float64) for z in (q, k, v, do))
    P = (Q @ K.T) * D
    R = (dO @ V.T) * D
    assert np.allclose(r["dv"][:, 0], scale * P.T @ dO, rtol=1e-12, atol=1e-12)
    assert np.allclose(r["dq"][:, 0], scale * R @ K, rtol=1e-12, atol=1e-12)
    assert np.allclose(r["dk"][:, 0], scale * R.T @ Q, rtol=1e-12, atol=1e-12)
    W = scale * (Q @ K.T) * (dO @ V.T) * D  # W[t, s]: the pair's weight in the loss
    dg = np.array([sum(W[t, s] for t in range(T) for s in range(T) if s < rr <= t) for rr in range(T)])
    assert np.allclose(r["dg"][:, 0], dg, rtol=1e-11, atol=1e-12)
    # the initial state (zero here) reaches o_t decayed by alpha^(t + 1)
    dh0 = scale * sum(a ** (t + 1) * np.outer(Q[t], dO[t]) for t in range(T))
    assert np.allclose(r["dh0"][0, 0], dh0, rtol=1e-12, atol=1e-12)


def test_empty_sequence_passes_the_state_gradient_through():
    x = make_inputs((0, 3), 1, 1, 3, 2, dtype="f32", seed=35, h0=True)
    rng = np.random.default_rng(3)
    do = rng.standard_normal(x.v.shape).astype(np.float32)
    dht = rng.standard_normal((2, 1, 3, 2)).astype(np.float32)
    r = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dht, x.cu_seqlens, x.scale)
    assert np.array_equal(r["dh0"][0], dht[0].astype(np.float64))


def test_zero_cotangents_give_zero_gradients():
    x = make_inputs((8,), 1, 1, 4, 4, dtype="f32", seed=36, h0=True)
    r = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, np.zeros_like(x.v), None, x.cu_seqlens,
                           x.scale)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert not np.any(r[key]), key


def test_sampled_units_match_full_run():
    x = make_inputs((20, 13), 1, 2, 4, 3, dtype="f32", seed=37, h0=True)
    do = np.random.default_rng(5).standard_normal(x.v.shape).astype(np.float32)
    full = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, None, x.cu_seqlens, x.scale)
    part = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, None, x.cu_seqlens, x.scale,
                              units=[(1, 1)])[0]
    s, e = x.cu_seqlens[1], x.cu_seqlens[2]
    assert np.array_equal(part["dv"], full["dv"][s:e, 1])
    assert np.array_equal(part["dg"], full["dg"][s:e, 1])
    assert np.array_equal(part["dh0"], full["dh0"][1, 1])
