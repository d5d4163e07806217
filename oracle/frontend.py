"""Oracle for the fused front-end of the forward pass — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module. It shares no code with the CUDA path.

The front-end is the per-token preparation that the Gated DeltaNet model applies to its
projections before the recurrence, and that the recurrent and chunkwise kernels can do
in place when asked ("Gated DeltaNet", section "模型调用方式：Qwen3.5 GatedDeltaNet",
part "Short Conv、门控与 Head 映射"; section "Recurrent 算法代码解析", part "逐 Token
更新：衰减、残差与读出"; section "Chunk-wise 算法代码解析", part "累计衰减门"):

* q and k are divided, per token and key head, by sqrt(sum of their squares + 1e-6);
* beta is the logistic sigmoid of a logit b;
* the natural-log gate is g = -exp(A_log) * softplus(a + dt_bias), with A_log one number
  per value head; g is then negative, so the decay exp(g) lies in (0, 1).

Readings taken where the pages leave a choice open:

* the query scale multiplies the output after the normalisation (the recurrent kernel
  multiplies the normalised q by it);
* per-channel gate (Kimi Delta Attention): a is [T, H_v, d_k], A_log stays one number per
  value head and dt_bias has one entry per (value head, channel); per-head gate (the
  scalar Gated DeltaNet): a is [T, H_v] and dt_bias [H_v];
* every step here is done in float64; the prepared q, k, beta and g are then handed to
  the token recurrence, which reads its inputs as float32 (a relative change below 1e-7).
"""

from __future__ import annotations

import numpy as np

from .recurrence import kda_recurrence

L2NORM_EPS = 1e-6


def l2norm(x):
    """x / sqrt(sum(x^2) + 1e-6) over the last axis, in float64 ("Gated DeltaNet",
    "Recurrent 算法代码解析": the in-kernel q/k normalisation)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2NORM_EPS)


def sigmoid(b):
    """1 / (1 + exp(-b)) in float64, evaluated without overflow for large |b|."""
    b = np.asarray(b, dtype=np.float64)
    e = np.exp(-np.abs(b))
    return np.where(b >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softplus(x):
    """log(1 + exp(x)) in float64, as max(x, 0) + log1p(exp(-|x|)) (no overflow)."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def gate(a, A_log, dt_bias):
    """g = -exp(A_log) * softplus(a + dt_bias) ("Gated DeltaNet", the model's gate).

    a [T, H_v] with A_log, dt_bias [H_v]; or a [T, H_v, d_k] with A_log [H_v] and dt_bias
    [H_v, d_k] (or None for no bias)."""
    a = np.asarray(a, dtype=np.float64)
    A = np.asarray(A_log, dtype=np.float64)
    if a.ndim == 3:
        A = A[:, None]
    x = a if dt_bias is None else a + np.asarray(dt_bias, dtype=np.float64)
    return -np.exp(A) * softplus(x)


def prepare(q, k, b, a, *, qk_l2norm=True, beta_sigmoid=True, A_log=None, dt_bias=None):
    """The front-end: the q, k, beta and g that the recurrence consumes.

    ``b`` is passed through unchanged when ``beta_sigmoid`` is false (it is then beta
    itself, or None for the decay-only recurrence); ``a`` is passed through unchanged
    when ``A_log`` is None (it is then the log gate g itself)."""
    if qk_l2norm:
        q, k = l2norm(q), l2norm(k)
    beta = sigmoid(b) if (beta_sigmoid and b is not None) else b
    g = gate(a, A_log, dt_bias) if A_log is not None else a
    return q, k, beta, g


def kda_fused_recurrence(q, k, v, a, b, h0, cu_seqlens, scale, *, qk_l2norm=True,
                         beta_sigmoid=True, A_log=None, dt_bias=None, units=None, threads=0):
    """The front-end followed by the fp64 token recurrence (see :func:`kda_recurrence`)."""
    q, k, beta, g = prepare(q, k, b, a, qk_l2norm=qk_l2norm, beta_sigmoid=beta_sigmoid,
                            A_log=A_log, dt_bias=dt_bias)
    return kda_recurrence(q, k, v, g, beta, h0, cu_seqlens, scale, units=units, threads=threads)
