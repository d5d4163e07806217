"""Pins of the oracle against what the pages and the mathematics fix (no GPU needed).

Each test checks the oracle against something other than itself: values the pages
print, closed forms, textbook special cases, an independent brute-force statement of
the recurrence from explicit matrices, the WY product identity, and invariants
(packing, grouped heads, resumption). A plausible mistake in the oracle — a dropped
term, a wrong sign, index or decay position, a transposed operand — fails at least one.
"""

from __future__ import annotations

import os

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from oracle import kda_chunked, kda_recurrence, naive_gram, separable_gram

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(lengths=(37,), H_k=2, H_v=2, d_k=8, d_v=6, seed=0, **kw):
    kw.setdefault("dtype", "f32")
    return make_inputs(lengths, H_k, H_v, d_k, d_v, seed=seed, **kw)


def _run(x, **kw):
    return kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, **kw)


# ---------------------------------------------------------------------------------------
# Values printed on the pages
# ---------------------------------------------------------------------------------------

def _read_golden():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "scalar_decay_worked_example.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "alpha":
                cur = {"alpha": float(vals[0]), "Gamma": []}
                blocks.append(cur)
            elif key == "Gamma_row":
                cur["Gamma"].append([float(x) for x in vals])
            else:
                cur[key] = [float(x) for x in vals]
    return blocks


def test_worked_example_cumulative_decay_and_mask():
    """Scalar-decay page §2.2: gamma and Gamma for alpha = 0.5 and 0.9 with C = 4.

    gamma_t is read from the oracle as the decay of a unit initial state (k = v = 0,
    decay-only form); Gamma[i, j] as the weight with which a one-hot v_j written at
    token j reaches the output at token i (q = k = 1).
    """
    blocks = _read_golden()
    for blk in blocks:
        a = blk["alpha"]
        C = 4
        g = np.full((C, 1), np.log(a), dtype=np.float64).astype(np.float32)
        cu = np.array([0, C], dtype=np.int32)
        if "gamma" in blk:
            q = np.ones((C, 1, 1), np.float32)
            k = np.zeros((C, 1, 1), np.float32)
            v = np.zeros((C, 1, 1), np.float32)
            h0 = np.ones((1, 1, 1, 1), np.float32)
            o, ht = kda_recurrence(q, k, v, g, None, h0, cu, 1.0)
            np.testing.assert_allclose(o[:, 0, 0], blk["gamma"], rtol=1e-6)
            np.testing.assert_allclose(ht[0, 0, 0, 0], blk["gamma"][-1], rtol=1e-6)
            gamma = np.asarray(blk["gamma"])
            np.testing.assert_allclose(gamma[3] / gamma[0], blk["Gamma_4_1"][0], rtol=1e-12)
        q = np.ones((C, 1, 1), np.float32)
        k = np.ones((C, 1, 1), np.float32)
        v = np.eye(C, dtype=np.float32)[:, None, :]
        o, _ = kda_recurrence(q, k, v, g, None, None, cu, 1.0)
        Gamma = o[:, 0, :]
        want = np.zeros((C, C))
        for i in range(C):
            for j in range(i + 1):
                want[i, j] = a ** (i - j)
        np.testing.assert_allclose(Gamma, want, rtol=1e-6, atol=1e-7)  # g is fp32-rounded
        if blk["Gamma"]:
            np.testing.assert_allclose(Gamma, np.asarray(blk["Gamma"]), rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------------------------------
# Closed forms and textbook special cases
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("alpha", [0.9, 0.5, 1.0])
def test_decay_only_constant_alpha_equals_retention_parallel_form(alpha):
    """Decay-gating page §1 (Eq. 5): O = (Q K^T ⊙ D) V, D_nm = alpha^(n-m) for n >= m.

    The oracle's decay-only recurrence with one constant gate per head, h0 = 0, must
    equal the parallel retention form; alpha = 1 is causal linear attention.
    """
    x = _small(lengths=(29, 40), H_k=2, H_v=2, d_k=8, d_v=5, gate="head", seed=3, beta=False)
    x.g[:] = np.float32(np.log(alpha))
    o, _ = kda_recurrence(x.q, x.k, x.v, x.g, None, None, x.cu_seqlens, x.scale)
    for n in range(x.N):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        L = e - s
        idx = np.arange(L)
        diff = idx[:, None] - idx[None, :]
        a64 = float(np.exp(np.float64(np.float32(np.log(alpha)))))
        D = np.where(diff >= 0, a64 ** np.maximum(diff, 0), 0.0)
        for h in range(x.H_v):
            Q = x.q[s:e, h].astype(np.float64)
            K = x.k[s:e, h].astype(np.float64)
            V = x.v[s:e, h].astype(np.float64)
            want = x.scale * ((Q @ K.T) * D) @ V
            assert rel_l2(o[s:e, h], want) < 1e-12


def test_beta_zero_is_pure_per_channel_decay_of_h0():
    """KDA page §3.4 degenerate check "beta -> 0": only the decaying initial state is left.

    o_t = scale * h0^T (exp(G_t) ⊙ q_t) and ht = Diag(exp(G_T)) h0, with G_t the
    whole-sequence cumulative sum of the per-channel log gates.
    """
    x = _small(lengths=(23, 17), H_k=1, H_v=2, d_k=8, d_v=6, h0=True, seed=4)
    x.beta[:] = 0.0
    o, ht = _run(x)
    for n in range(x.N):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        for h in range(x.H_v):
            G = np.cumsum(x.g[s:e, h].astype(np.float64), axis=0)
            h0 = x.h0[n, h].astype(np.float64)
            want_o = x.scale * np.einsum("dv,td->tv", h0, np.exp(G) * x.q[s:e, 0])
            assert rel_l2(o[s:e, h], want_o) < 1e-12
            assert rel_l2(ht[n, h], np.exp(G[-1])[:, None] * h0) < 1e-12


def _paper_layout_brute_force(x, n, h):
    """S_t = S_0 prod_{tau<=t} H_tau + sum_tau beta_tau v_tau k_tau^T prod_{tau<i<=t} H_i.

    Paper layout (S in R^{d_v x d_k}) with H_tau = Diag(a_tau)(I - beta_tau k k^T), every
    product formed from scratch for every t ("RNN的复兴04:线性注意力并行计算DPLR" §3.1,
    the unrolled state; "TileLang 实战：KDA 从零到一–Kimi Delta Attention" §3.1).
    """
    s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
    hk = h // (x.H_v // x.H_k)
    d_k = x.d_k
    I = np.eye(d_k)
    ks = x.k[s:e, hk].astype(np.float64)
    qs = x.q[s:e, hk].astype(np.float64)
    vs = x.v[s:e, h].astype(np.float64)
    gs = x.g[s:e, h].astype(np.float64)
    if gs.ndim == 1:
        gs = np.repeat(gs[:, None], d_k, axis=1)
    bs = x.beta[s:e, h].astype(np.float64)
    Hm = [np.diag(np.exp(gs[t])) @ (I - bs[t] * np.outer(ks[t], ks[t])) for t in range(e - s)]
    S0 = np.zeros((x.d_v, d_k)) if x.h0 is None else x.h0[n, h].astype(np.float64).T
    outs, S = [], S0
    for t in range(e - s):
        P = I.copy()
        for tau in range(t + 1):
            P = P @ Hm[tau]
        S = S0 @ P
        for tau in range(t + 1):
            R = I.copy()
            for i in range(tau + 1, t + 1):
                R = R @ Hm[i]
            S = S + bs[tau] * np.outer(vs[tau], ks[tau]) @ R
        outs.append(x.scale * S @ qs[t])
    return np.array(outs), S


@pytest.mark.parametrize("gate", ["channel", "head"])
def test_brute_force_explicit_products_tiny(gate):
    """T <= 16: the oracle equals the unrolled product form built from explicit matrices."""
    x = _small(lengths=(16, 9), H_k=1, H_v=2, d_k=5, d_v=4, h0=True, gate=gate, seed=5, a_lo=0.6)
    o, ht = _run(x)
    for n in range(x.N):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        for h in range(x.H_v):
            want_o, S = _paper_layout_brute_force(x, n, h)
            assert rel_l2(o[s:e, h], want_o) < 1e-12
            assert rel_l2(ht[n, h], S.T) < 1e-12


def test_gate_zero_is_deltanet():
    """KDA page §3.4 degenerate check "g -> 0": plain DeltaNet, S <- S (I - b k k^T) + b v k^T."""
    x = _small(lengths=(21,), H_k=1, H_v=1, d_k=6, d_v=5, h0=True, seed=6)
    x.g[:] = 0.0
    o, ht = _run(x)
    S = x.h0[0, 0].astype(np.float64).T
    I = np.eye(x.d_k)
    for t in range(21):
        k = x.k[t, 0].astype(np.float64)
        b = float(x.beta[t, 0])
        S = S @ (I - b * np.outer(k, k)) + b * np.outer(x.v[t, 0].astype(np.float64), k)
        assert rel_l2(o[t, 0], x.scale * S @ x.q[t, 0].astype(np.float64)) < 1e-12
    assert rel_l2(ht[0, 0], S.T) < 1e-12


def test_wy_product_identity():
    """DPLR page §2: prod_tau (Lambda_tau - x_tau y_tau^T) = D_t - W_t^T Y_t.

    Lambda = Diag(a), x = beta (a ⊙ k), y = k, so that the product is the KDA
    transition. W is built with the page's recursion
    w_t = D_{t-1} x_t - sum_{tau<t} (nu_tau^{(t-1)T} x_t) w_tau,  nu_tau^{(t)} = D_{tau+1:t} y_tau.
    The oracle's state with v = 0 and S_0 = I is that product (transposed layout).
    """
    x = _small(lengths=(12,), H_k=1, H_v=1, d_k=6, d_v=6, seed=7, a_lo=0.7)
    x.v[:] = 0.0
    d = x.d_k
    h0 = np.eye(d, dtype=np.float32)[None, None]
    a = np.exp(x.g[:, 0].astype(np.float64))
    k = x.k[:, 0].astype(np.float64)
    b = x.beta[:, 0].astype(np.float64)
    for t in range(1, 13):
        xs = [b[i] * a[i] * k[i] for i in range(t)]
        D = lambda lo, hi: np.prod(a[lo:hi], axis=0)  # noqa: E731  diag of D_{lo+1:hi}
        ws = []
        for tt in range(t):
            w = D(0, tt) * xs[tt]
            for tau in range(tt):
                nu = D(tau + 1, tt) * k[tau]
                w = w - (nu @ xs[tt]) * ws[tau]
            ws.append(w)
        P_wy = np.diag(D(0, t)) - sum(np.outer(ws[tau], D(tau + 1, t) * k[tau]) for tau in range(t))
        P_bf = np.eye(d)
        for tau in range(t):
            P_bf = P_bf @ (np.diag(a[tau]) - np.outer(xs[tau], k[tau]))
        assert rel_l2(P_wy, P_bf) < 1e-12
        cu = np.array([0, t], dtype=np.int32)
        _, ht = kda_recurrence(x.q[:t], x.k[:t], x.v[:t], x.g[:t], x.beta[:t], h0, cu, 1.0)
        assert rel_l2(ht[0, 0].T, P_wy) < 1e-12


# ---------------------------------------------------------------------------------------
# The chunk algebra against the definition
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("pairing", ["row", "col"])
def test_chunked_restatement_equals_recurrence(C, pairing):
    """KDA page §3.4: chunkwise = token recurrence; C = 1 is the recurrence itself
    ("Gated DeltaNet": a chunk of one token is the recurrent step). Lengths are not
    multiples of C, so tail chunks are covered."""
    x = _small(lengths=(70, 45), H_k=1, H_v=2, d_k=8, d_v=6, h0=True, seed=8)
    o_r, ht_r = _run(x)
    o_c, ht_c = kda_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, C, pairing)
    assert rel_l2(o_c, o_r) < 1e-12
    assert rel_l2(ht_c, ht_r) < 1e-12


def test_mixed_beta_pairing_is_detected():
    """KDA page §3.3 note 3: mixing the two beta pairings is wrong with random beta."""
    x = _small(lengths=(64,), H_k=1, H_v=1, d_k=8, d_v=6, seed=9)
    o_r, _ = _run(x)
    o_m, _ = kda_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, 16, "mixed")
    assert rel_l2(o_m, o_r) > 1e-2
    x.beta[:] = 0.5  # the mistake hides when every beta is equal
    o_r, _ = _run(x)
    o_m, _ = kda_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, 16, "mixed")
    assert rel_l2(o_m, o_r) < 1e-12


def test_separable_gram_equals_entrywise():
    """KDA page §1.2: (K e^gamma)(K e^-gamma)^T equals the entrywise decay-weighted products."""
    rng = np.random.default_rng(10)
    K = rng.standard_normal((64, 16))
    gam = np.cumsum(np.log(rng.uniform(0.9, 0.999, (64, 16))), axis=0)
    sep = separable_gram(K, gam)
    nai = naive_gram(K, K, gam, gam, strict=True)
    lower = np.tril(np.ones((64, 64), bool), -1)
    assert rel_l2(sep[lower], nai[lower]) < 1e-14


def test_equal_channel_gate_is_scalar_gate():
    """KDA page §3.4: a per-channel gate with equal channels reduces to the scalar gate."""
    x = _small(lengths=(33,), H_k=2, H_v=2, d_k=8, d_v=6, h0=True, gate="head", seed=11)
    o_h, ht_h = _run(x)
    g_ch = np.repeat(x.g[:, :, None], x.d_k, axis=2)
    o_c, ht_c = kda_recurrence(x.q, x.k, x.v, g_ch, x.beta, x.h0, x.cu_seqlens, x.scale)
    np.testing.assert_array_equal(o_c, o_h)
    np.testing.assert_array_equal(ht_c, ht_h)


# ---------------------------------------------------------------------------------------
# Invariants: packing, grouped heads, scale, resumption, empty sequences
# ---------------------------------------------------------------------------------------

def test_packed_sequences_equal_separate_runs():
    x = _small(lengths=(19, 1, 40), H_k=1, H_v=2, d_k=8, d_v=6, h0=True, seed=12)
    o, ht = _run(x)
    for n in range(x.N):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        cu = np.array([0, e - s], np.int32)
        o1, ht1 = kda_recurrence(x.q[s:e], x.k[s:e], x.v[s:e], x.g[s:e], x.beta[s:e],
                                 x.h0[n:n + 1], cu, x.scale)
        np.testing.assert_array_equal(o[s:e], o1)
        np.testing.assert_array_equal(ht[n], ht1[0])


def test_grouped_heads_equal_repeated_key_heads():
    """"Gated DeltaNet" (GQA head map): value head h reads key head h // (H_v / H_k)."""
    x = _small(lengths=(30,), H_k=2, H_v=6, d_k=8, d_v=6, h0=True, seed=13)
    o, ht = _run(x)
    qr = np.repeat(x.q, 3, axis=1)
    kr = np.repeat(x.k, 3, axis=1)
    o2, ht2 = kda_recurrence(qr, kr, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(ht, ht2)


def test_scale_multiplies_output_only():
    x = _small(lengths=(25,), seed=14, h0=True)
    o1, ht1 = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, 1.0)
    o2, ht2 = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, 0.25)
    assert rel_l2(o2, 0.25 * o1) < 1e-15
    np.testing.assert_array_equal(ht1, ht2)


def test_resume_from_final_state():
    """The final state of [0, T1) is the initial state of [T1, T) ("Gated DeltaNet":
    the chunk path's final state feeds the recurrent path)."""
    x = _small(lengths=(50,), seed=15, h0=True)
    o, ht = _run(x)
    T1 = 23
    cu1 = np.array([0, T1], np.int32)
    cu2 = np.array([0, 50 - T1], np.int32)
    o1, ht1 = kda_recurrence(x.q[:T1], x.k[:T1], x.v[:T1], x.g[:T1], x.beta[:T1], x.h0, cu1, x.scale)
    o2, ht2 = kda_recurrence(x.q[T1:], x.k[T1:], x.v[T1:], x.g[T1:], x.beta[T1:],
                             ht1.astype(np.float32), cu2, x.scale)
    assert rel_l2(np.concatenate([o1, o2]), o) < 1e-6  # h0 hand-over is rounded to fp32
    assert rel_l2(ht2, ht) < 1e-6


def test_empty_sequence_keeps_initial_state():
    x = _small(lengths=(0, 5, 0), H_k=1, H_v=1, d_k=4, d_v=3, h0=True, seed=16, varlen=True)
    o, ht = _run(x)
    assert o.shape == (5, 1, 3)
    np.testing.assert_array_equal(ht[0], x.h0[0].astype(np.float64))
    np.testing.assert_array_equal(ht[2], x.h0[2].astype(np.float64))


def test_sampled_units_match_full_run():
    x = _small(lengths=(20, 31), H_k=2, H_v=4, d_k=8, d_v=6, h0=True, seed=17)
    o, ht = _run(x)
    res = kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale,
                         units=[(1, 3), (0, 0), (1, 1)])
    for (n, h), (ou, hu) in zip([(1, 3), (0, 0), (1, 1)], res):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        np.testing.assert_array_equal(ou, o[s:e, h])
        np.testing.assert_array_equal(hu, ht[n, h])
