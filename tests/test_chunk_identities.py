"""The chunk identities the GPU kernels are built on, checked in fp64 against the oracle's
token recurrence (no GPU needed).

The chunk form (DPLR page §5.3.5; KDA page §3.2-3.3) advances the state with
S' = Diag(e^{γ_n}) S + K̄ᵀ Ṽ, K̄ = K ⊙ e^{γ_n - γ}. The persistent kernel's consumer never
forms K̄: since K̄ = Km · Diag(e^{γ_n}) with Km = K ⊙ e^{-γ}, it keeps R = S_c + Kmᵀ Ṽ and
applies Diag(e^{γ_n}) where the state is read (the next chunk's rescale, its bf16 copy,
the final state). Both forms must give the recurrence's outputs and final state.
"""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from oracle import kda_recurrence

C = 64


def _chunk_factors(q, k, v, g, beta, scale):
    """Per-chunk factors of one unit (rows = tokens of the chunk), fp64."""
    gam = np.cumsum(g, axis=0)                      # chunk-local cumulative log gate
    eg = np.exp(gam[-1])                            # e^{γ_n}, per channel
    qp = scale * q * np.exp(gam)
    kp = k * np.exp(gam)
    km = k * np.exp(-gam)
    n = q.shape[0]
    m = np.tril(kp @ km.T, -1)                      # strictly lower
    a = np.tril(qp @ km.T)                          # lower with the diagonal
    t = np.linalg.inv(np.eye(n) + beta[:, None] * m)
    w = t @ (beta[:, None] * kp)
    u = t @ (beta[:, None] * v)
    return qp, km, eg, a, w, u


def _two_forms(x):
    q, k, v = (np.asarray(a, np.float64)[:, 0] for a in (x.q, x.k, x.v))
    g = np.asarray(x.g, np.float64)[:, 0]
    beta = np.asarray(x.beta, np.float64)[:, 0]
    d_k, d_v = q.shape[1], v.shape[1]
    s = np.zeros((d_k, d_v))                        # the chunk form with K̄
    r, eg_prev = np.zeros((d_k, d_v)), np.ones(d_k)  # the deferred form: S_c = Diag(eg_prev) R
    o_std, o_def = np.zeros_like(v), np.zeros_like(v)
    for c0 in range(0, q.shape[0], C):
        sl = slice(c0, min(c0 + C, q.shape[0]))
        qp, km, eg, a, w, u = _chunk_factors(q[sl], k[sl], v[sl], g[sl], beta[sl], x.scale)
        kb = km * eg
        vt = u - w @ s
        o_std[sl] = qp @ s + a @ vt
        s = eg[:, None] * s + kb.T @ vt
        s_c = eg_prev[:, None] * r                  # the consumer's rescale of R
        vt2 = u - w @ s_c
        o_def[sl] = qp @ s_c + a @ vt2
        r = s_c + km.T @ vt2
        eg_prev = eg
    return o_std, s, o_def, eg_prev[:, None] * r


@pytest.mark.parametrize("length", [1, 64, 150, 300])
def test_deferred_gate_scaling_equals_chunk_form_and_recurrence(length):
    x = make_inputs((length,), 1, 1, 8, 6, seed=3, dtype="f32")
    o_ref, ht_ref = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, None, x.cu_seqlens, x.scale)
    o_std, s_std, o_def, s_def = _two_forms(x)
    assert rel_l2(o_def, o_std) < 1e-12 and rel_l2(s_def, s_std) < 1e-12
    assert rel_l2(o_std, np.asarray(o_ref)[:, 0]) < 1e-10
    assert rel_l2(s_std, np.asarray(ht_ref)[0, 0]) < 1e-10


def test_dropping_the_final_scaling_is_detected():
    """The final state needs the last chunk's Diag(e^{γ_n}): R alone is wrong."""
    x = make_inputs((150,), 1, 1, 8, 6, seed=3, dtype="f32")
    _, ht_ref = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, None, x.cu_seqlens, x.scale)
    q, k, v = (np.asarray(a, np.float64)[:, 0] for a in (x.q, x.k, x.v))
    g = np.asarray(x.g, np.float64)[:, 0]
    beta = np.asarray(x.beta, np.float64)[:, 0]
    r, eg_prev = np.zeros((8, 6)), np.ones(8)
    for c0 in range(0, 150, C):
        sl = slice(c0, min(c0 + C, 150))
        qp, km, eg, a, w, u = _chunk_factors(q[sl], k[sl], v[sl], g[sl], beta[sl], x.scale)
        s_c = eg_prev[:, None] * r
        r = s_c + km.T @ (u - w @ s_c)
        eg_prev = eg
    assert rel_l2(r, np.asarray(ht_ref)[0, 0]) > 1e-3
