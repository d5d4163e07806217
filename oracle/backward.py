"""ctypes front end of the backward oracle (``kda_oracle_bwd.c``) — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module. The C file states the gradients and cites the passage it follows.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import recurrence

_fn = None


def _load():
    global _fn
    if _fn is None:
        lib = recurrence._load()
        P, I = ctypes.c_void_p, ctypes.c_int
        fn = lib.kda_oracle_bwd
        fn.argtypes = [P, P, P, P, I, P, P, P, P, P, I, I, I, I, I, ctypes.c_double, P, I, P,
                       P, P, P, P, P, P, I]
        fn.restype = I
        _fn = fn
    return _fn


def _f32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float32)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def kda_recurrence_bwd(q, k, v, g, beta, h0, do, dht, cu_seqlens, scale, *, units=None, threads=0):
    """Gradients of sum(do * o) + sum(dht * ht) through the token recurrence, in float64.

    Shapes as :func:`oracle.kda_recurrence`, plus do [T, H_v, d_v] and dht
    [N, H_v, d_k, d_v] (or None). With ``units=None`` every unit is run and the result is a
    dict with dq, dk [T, H_k, d_k] (summed over the value heads that share a key head), dv
    [T, H_v, d_v], dg (g's shape), dbeta [T, H_v] (None without beta) and dh0
    [N, H_v, d_k, d_v]. With ``units`` a list of (n, h) pairs, a list of per-unit dicts
    (rows of that sequence; dq and dk are the unit's own part).
    """
    fn = _load()
    q, k, v, g, beta, h0, do, dht = (_f32(x) for x in (q, k, v, g, beta, h0, do, dht))
    T, H_k, d_k = q.shape
    _, H_v, d_v = v.shape
    if k.shape != q.shape or do.shape != v.shape or g.shape[0] != T:
        raise ValueError("inconsistent shapes")
    per_channel = 1 if g.ndim == 3 else 0
    gd = d_k if per_channel else 1
    seq_off = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = len(seq_off) - 1
    lens = np.diff(seq_off)
    full = units is None
    ulist = [(n, h) for n in range(N) for h in range(H_v)] if full else [(int(n), int(h)) for n, h in units]
    uid = np.array([n * H_v + h for n, h in ulist], dtype=np.int32)
    rows = np.array([lens[n] for n, _ in ulist], dtype=np.int64)
    row = np.zeros(len(ulist), dtype=np.int64)
    if len(ulist):
        row[1:] = np.cumsum(rows)[:-1]
    R = int(rows.sum())
    out = {name: np.zeros((max(R, 1), w)) for name, w in
           (("dq", d_k), ("dk", d_k), ("dv", d_v), ("dg", gd), ("dbeta", 1))}
    dh0 = np.zeros((max(len(ulist), 1), d_k, d_v))
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), per_channel, _ptr(beta), _ptr(h0), _ptr(do), _ptr(dht),
            _ptr(seq_off), N, H_k, H_v, d_k, d_v, float(scale), _ptr(uid), len(ulist), _ptr(row),
            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
            _ptr(dh0), int(threads))
    if st != 0:
        raise RuntimeError(f"kda_oracle_bwd failed with status {st}")
    per_unit = []
    for i, (n, h) in enumerate(ulist):
        a, b = row[i], row[i] + rows[i]
        per_unit.append({"dq": out["dq"][a:b], "dk": out["dk"][a:b], "dv": out["dv"][a:b],
                         "dg": out["dg"][a:b] if per_channel else out["dg"][a:b, 0],
                         "dbeta": out["dbeta"][a:b, 0] if beta is not None else None, "dh0": dh0[i]})
    if not full:
        return per_unit
    grp = H_v // H_k
    res = {"dq": np.zeros((T, H_k, d_k)), "dk": np.zeros((T, H_k, d_k)), "dv": np.zeros((T, H_v, d_v)),
           "dg": np.zeros(g.shape, dtype=np.float64),
           "dbeta": np.zeros((T, H_v)) if beta is not None else None, "dh0": np.zeros((N, H_v, d_k, d_v))}
    for i, (n, h) in enumerate(ulist):
        s, e = seq_off[n], seq_off[n + 1]
        u = per_unit[i]
        res["dq"][s:e, h // grp] += u["dq"]
        res["dk"][s:e, h // grp] += u["dk"]
        res["dv"][s:e, h] = u["dv"]
        res["dg"][s:e, h] = u["dg"]
        if beta is not None:
            res["dbeta"][s:e, h] = u["dbeta"]
        res["dh0"][n, h] = u["dh0"]
    return res
