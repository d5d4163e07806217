"""Chunkwise restatement of the gated delta rule in fp64 numpy — TEST INFRASTRUCTURE ONLY.

This is the oracle's second function: the same result as the token recurrence
(``kda_oracle.c``), reached through the per-chunk equations the pages derive. It exists
to pin the chunk algebra (cumulative gate with a reset per chunk, the decay-weighted
Gram matrix, the UT-transform triangular solve, the pseudo-values, the chunk output and
the chunk-to-chunk state step) against the definition, on small inputs.

Per chunk of n <= C tokens with entry state S (transposed layout, d_k x d_v), following
"TileLang 实战：KDA 从零到一–Kimi Delta Attention" §3.2 (reference B) and the standard
form of "RNN的复兴04:线性注意力并行计算DPLR" §5.3.5:

1. gamma_r = sum_{s <= r} g_s per channel, restarted at every chunk (§0 of the KDA page;
   "TileLang 实战：KDA 从零到一--标量衰减" §2.1 on the per-chunk reset);
2. M[c, i] = sum_d k_c[d] k_i[d] exp(gamma_c[d] - gamma_i[d]) for i < c, evaluated only
   where i < c (scalar-decay page §2.2: never build the full decay table and mask it);
3. the triangular system. Two pairings of beta are exact (KDA page §3.3, note 3):
   "row":  L = diag(beta) strict_lower(M),  T = (I + L)^-1,  A_hat = T diag(beta)
   "col":  L = strict_lower(M) diag(beta),  T = (I + L)^-1,  A_hat = diag(beta) T
   "mixed" takes the row L with the col A_hat; the KDA page reports that this mix is
   wrong (relative L2 ~1e-1 with random beta). It is kept so the tests can show that
   the pins detect it;
4. W = A_hat (K * exp(gamma)), U = A_hat V, pseudo-values V~ = U - W S;
5. A_qk[c, j] = sum_d q_c[d] k_j[d] exp(gamma_c[d] - gamma_j[d]) for j <= c;
   O = scale * ((Q * exp(gamma)) S + A_qk V~);
6. S <- Diag(exp(gamma_n)) S + (K * exp(gamma_n - gamma))^T V~, gamma_n the last row's.

The inverse is explicit (``numpy.linalg.inv``), as in reference B.
"""

from __future__ import annotations

import numpy as np


def naive_gram(Ka, Kb, gam_a, gam_b, strict: bool):
    """Decay-weighted Gram matrix, evaluated entry by entry on the causal side only.

    G[c, i] = sum_d Ka[c, d] Kb[i, d] exp(gam_a[c, d] - gam_b[i, d]) for i < c
    (``strict``) or i <= c, and 0 elsewhere.
    """
    n = Ka.shape[0]
    G = np.zeros((n, n), dtype=np.float64)
    for c in range(n):
        last = c if strict else c + 1
        for i in range(last):
            G[c, i] = np.dot(Ka[c] * np.exp(gam_a[c] - gam_b[i]), Kb[i])
    return G


def separable_gram(K, gam):
    """The separable form of the same matrix before masking: (K e^gamma)(K e^-gamma)^T.

    "TileLang 实战：KDA 从零到一–Kimi Delta Attention" §1.2: exp(gamma_c - gamma_i)
    factors into exp(gamma_c) * exp(-gamma_i) channel by channel.
    """
    return (K * np.exp(gam)) @ (K * np.exp(-gam)).T


def _chunk_step(Qc, Kc, Vc, gc, bc, S, scale, pairing):
    n = Kc.shape[0]
    gam = np.cumsum(gc, axis=0)
    gam_n = gam[-1]
    M = naive_gram(Kc, Kc, gam, gam, strict=True)
    I = np.eye(n)
    if pairing == "row":
        T = np.linalg.inv(I + bc[:, None] * M)
        A_hat = T * bc[None, :]
    elif pairing == "col":
        T = np.linalg.inv(I + M * bc[None, :])
        A_hat = bc[:, None] * T
    elif pairing == "mixed":
        T = np.linalg.inv(I + bc[:, None] * M)
        A_hat = bc[:, None] * T
    else:
        raise ValueError(f"unknown pairing {pairing!r}")
    W = A_hat @ (Kc * np.exp(gam))
    U = A_hat @ Vc
    Vt = U - W @ S
    Aqk = naive_gram(Qc, Kc, gam, gam, strict=False)
    O = scale * ((Qc * np.exp(gam)) @ S + Aqk @ Vt)
    S_next = np.exp(gam_n)[:, None] * S + (Kc * np.exp(gam_n[None, :] - gam)).T @ Vt
    return O, S_next


def kda_chunked(q, k, v, g, beta, h0, cu_seqlens, scale, C, pairing="row"):
    """Chunkwise fp64 restatement; same arguments and result as the full-mode recurrence.

    ``C`` is the chunk length; a sequence whose length is not a multiple of C ends in a
    shorter tail chunk. Returns ``(o [T, H_v, d_v], ht [N, H_v, d_k, d_v])``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    T, H_k, d_k = q.shape
    _, H_v, d_v = v.shape
    if g.ndim == 2:
        g = np.repeat(g[:, :, None], d_k, axis=2)
    if beta is None:
        raise ValueError("the chunked restatement covers the erase form (beta given)")
    beta = np.asarray(beta, dtype=np.float64)
    off = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(off) - 1
    o = np.zeros((T, H_v, d_v))
    ht = np.zeros((N, H_v, d_k, d_v))
    grp = H_v // H_k
    for n in range(N):
        for h in range(H_v):
            hk = h // grp
            S = np.zeros((d_k, d_v)) if h0 is None else np.asarray(h0[n, h], dtype=np.float64).copy()
            for s in range(off[n], off[n + 1], C):
                e = min(s + C, off[n + 1])
                O, S = _chunk_step(q[s:e, hk], k[s:e, hk], v[s:e, h], g[s:e, h], beta[s:e, h],
                                   S, scale, pairing)
                o[s:e, h] = O
            ht[n, h] = S
    return o, ht
