"""ctypes front end of the C oracle (``kda_oracle.c``) — TEST INFRASTRUCTURE ONLY.

Marshals numpy arrays into the C recurrence and reassembles its outputs. The C file
states the recurrence and cites the passages it follows.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, ctypes.c_double,
                                       P, I, P, P, P, I]
        lib.kda_oracle_fwd.restype = I
        lib.kda_oracle_default_threads.argtypes = []
        lib.kda_oracle_default_threads.restype = I
        _lib = lib
    return _lib


def oracle_threads() -> int:
    """Worker threads the oracle uses when asked for every core."""
    return int(_load().kda_oracle_default_threads())


def _f32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float32)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def kda_recurrence(q, k, v, g, beta, h0, cu_seqlens, scale, *, units=None, threads=0):
    """fp64 token recurrence of the gated delta rule (the oracle's definition).

    q, k [T, H_k, d_k]; v [T, H_v, d_v]; g [T, H_v, d_k] (per-channel gate) or [T, H_v]
    (scalar gate), natural log; beta [T, H_v] or None (decay-only recurrence);
    h0 [N, H_v, d_k, d_v] or None; cu_seqlens [N + 1] token offsets.

    With ``units=None`` every (sequence, value head) unit is run and the result is
    ``(o [T, H_v, d_v], ht [N, H_v, d_k, d_v])`` in float64. With ``units`` a list of
    ``(n, h)`` pairs, only those are run and the result is a list of
    ``(o_unit [len_n, d_v], ht_unit [d_k, d_v])``.
    """
    lib = _load()
    q, k, v, g = _f32(q), _f32(k), _f32(v), _f32(g)
    beta, h0 = _f32(beta), _f32(h0)
    T, H_k, d_k = q.shape
    _, H_v, d_v = v.shape
    if k.shape != q.shape or v.shape[0] != T or g.shape[0] != T:
        raise ValueError("inconsistent shapes")
    per_channel = 1 if g.ndim == 3 else 0
    seq_off = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = len(seq_off) - 1
    lens = np.diff(seq_off)

    full = units is None
    if full:
        ulist = [(n, h) for n in range(N) for h in range(H_v)]
    else:
        ulist = [(int(n), int(h)) for n, h in units]
    uid = np.array([n * H_v + h for n, h in ulist], dtype=np.int32)
    rows = np.array([lens[n] for n, _ in ulist], dtype=np.int64)
    o_row = np.zeros(len(ulist), dtype=np.int64)
    if len(ulist):
        o_row[1:] = np.cumsum(rows)[:-1]
    o = np.zeros((max(int(rows.sum()), 1), d_v), dtype=np.float64)
    ht = np.zeros((max(len(ulist), 1), d_k, d_v), dtype=np.float64)

    rc = lib.kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), per_channel, _ptr(beta), _ptr(h0),
                            _ptr(seq_off), N, H_k, H_v, d_k, d_v, float(scale), _ptr(uid),
                            len(ulist), _ptr(o_row), _ptr(o), _ptr(ht), int(threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with status {rc}")

    if not full:
        return [(o[o_row[i]:o_row[i] + rows[i]].copy(), ht[i].copy()) for i in range(len(ulist))]
    o_full = np.zeros((T, H_v, d_v), dtype=np.float64)
    ht_full = np.zeros((N, H_v, d_k, d_v), dtype=np.float64)
    for i, (n, h) in enumerate(ulist):
        o_full[seq_off[n]:seq_off[n + 1], h] = o[o_row[i]:o_row[i] + rows[i]]
        ht_full[n, h] = ht[i]
    return o_full, ht_full
