"""Seeded synthetic inputs for the chunkwise gated delta rule (KDA) forward pass.

Recipe (one ``numpy.random.default_rng(seed)`` stream, draws in this order):

1. sequence lengths (varlen workloads only): integers ~ U[len_lo, len_hi];
2. q [T, H_k, d_k] ~ N(0, 1) in fp32, L2-normalised per token and head (no epsilon);
3. k [T, H_k, d_k] likewise;
4. v [T, H_v, d_v] ~ N(0, 1) in fp32;
5. a ~ U[a_lo, 0.999] in fp64, one per (token, value head, channel) for the
   per-channel gate or one per (token, value head) for the scalar gate; g = log(a)
   rounded to fp32 (natural log, g < 0);
6. beta = sigmoid(b), b ~ N(0, 1), fp32, one per (token, value head);
7. h0 [N, H_v, d_k, d_v] ~ N(0, 0.1**2) in fp32 (sigma = 0.1), or no initial state.

Every tensor is drawn in blocks of ``_BLOCK`` tokens so that peak host memory stays
bounded; the block size is part of the recipe. q, k and v are then rounded to the
storage dtype (bf16 round-to-nearest-even, or kept in fp32); the returned float32
arrays hold exactly the values handed to the GPU.

The workloads follow the shapes and distributions that the KDA pages use for their
checks (Kimi Delta Attention page, section 3.4: L2-normalised q and k, a drawn from a
lower-bounded interval, beta in (0, 1)). No dataset is involved.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_BLOCK = 4096


@dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic workload."""

    name: str
    lengths: tuple  # per-sequence lengths; fixed-length batches repeat one value
    H_k: int
    H_v: int
    d_k: int
    d_v: int
    dtype: str = "bf16"  # storage dtype of q, k, v, o: "bf16" or "f32"
    gate: str = "channel"  # "channel" (g [T, H_v, d_k]) or "head" (g [T, H_v])
    a_lo: float = 0.9
    h0: bool = False
    varlen: bool = False  # packed with cu_seqlens (physical batch 1)
    len_range: tuple | None = None  # (lo, hi) for drawn lengths; overrides lengths
    n_seqs: int | None = None
    beta: bool = True  # False: no beta (the decay-only recurrence)

    @property
    def T(self) -> int:
        return self.lengths[0]


# The five workloads of the method's benchmark set, named by what they are.
WORKLOADS = {
    "kda_b1_t256_h1_d64_f32": Workload(
        "kda_b1_t256_h1_d64_f32", (256,), 1, 1, 64, 64, dtype="f32"),
    "gdn_b4_t4096_h16_d128_bf16": Workload(
        "gdn_b4_t4096_h16_d128_bf16", (4096,) * 4, 16, 16, 128, 128, gate="head"),
    "kda_b2_t8192_h32_d128_bf16": Workload(
        "kda_b2_t8192_h32_d128_bf16", (8192,) * 2, 32, 32, 128, 128, h0=True),
    "kda_gqa_b1_t32768_hk16_hv32_d128_bf16": Workload(
        "kda_gqa_b1_t32768_hk16_hv32_d128_bf16", (32768,), 16, 32, 128, 128),
    "kda_varlen16_t512to16384_h32_d128_bf16": Workload(
        "kda_varlen16_t512to16384_h32_d128_bf16", (), 32, 32, 128, 128, a_lo=0.8,
        h0=True, varlen=True, len_range=(512, 16384), n_seqs=16),
}

WORKLOAD_SEEDS = {name: i + 1 for i, name in enumerate(WORKLOADS)}

# Smaller cases of the same kernels for profiler captures (inputs still larger than L2),
# and the decay-only variant of the benchmark shape.
PROFILE_WORKLOADS = {
    "kda_decode_b256_t1_h32_d128_bf16": Workload(
        "kda_decode_b256_t1_h32_d128_bf16", (1,) * 256, 32, 32, 128, 128, h0=True),
    "kda_decayonly_b2_t8192_h32_d128_bf16": Workload(
        "kda_decayonly_b2_t8192_h32_d128_bf16", (8192,) * 2, 32, 32, 128, 128, h0=True, beta=False),
    "kda_b1_t8192_h32_d128_bf16": Workload(
        "kda_b1_t8192_h32_d128_bf16", (8192,), 32, 32, 128, 128, h0=True),
    # a short case of the backward for profiler captures (its scratch still exceeds L2)
    "kda_b1_t2048_h32_d128_bf16": Workload(
        "kda_b1_t2048_h32_d128_bf16", (2048,), 32, 32, 128, 128, h0=True),
    # the benchmark's 64 units (so the same ring depth and launch split) over half the tokens
    "kda_b2_t4096_h32_d128_bf16": Workload(
        "kda_b2_t4096_h32_d128_bf16", (4096,) * 2, 32, 32, 128, 128, h0=True),
}


@dataclass
class Inputs:
    """Host copies (float32 numpy) of one problem, exactly as handed to the GPU."""

    q: np.ndarray  # [T, H_k, d_k]
    k: np.ndarray  # [T, H_k, d_k]
    v: np.ndarray  # [T, H_v, d_v]
    g: np.ndarray  # [T, H_v, d_k] (channel gate) or [T, H_v] (scalar gate)
    beta: np.ndarray | None  # [T, H_v]
    h0: np.ndarray | None  # [N, H_v, d_k, d_v]
    cu_seqlens: np.ndarray  # int32 [N + 1]
    H_k: int
    H_v: int
    d_k: int
    d_v: int
    dtype: str
    gate: str
    scale: float
    varlen: bool
    meta: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def T_total(self) -> int:
        return int(self.cu_seqlens[-1])

    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype (bf16: round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    bits = x.view(np.uint32)
    nan = np.isnan(x)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    out = rounded.view(np.float32).copy()
    out[nan] = np.nan
    return out


def _normal_rows(rng, T, cols, dtype=np.float32):
    out = np.empty((T, cols), dtype=dtype)
    for s in range(0, T, _BLOCK):
        e = min(T, s + _BLOCK)
        out[s:e] = rng.standard_normal((e - s, cols), dtype=np.float32)
    return out


def _l2_normalise(x: np.ndarray, H: int, d: int) -> np.ndarray:
    x3 = x.reshape(-1, H, d)
    for s in range(0, x3.shape[0], _BLOCK):
        blk = x3[s:s + _BLOCK]
        nrm = np.sqrt(np.sum(blk * blk, axis=-1, dtype=np.float32), dtype=np.float32)
        blk /= nrm[..., None]
    return x3


def make_inputs(lengths, H_k, H_v, d_k, d_v, *, dtype="bf16", gate="channel", a_lo=0.9,
                h0=False, beta=True, varlen=None, seed=0, scale=None,
                len_range=None, n_seqs=None) -> Inputs:
    """Draw one problem following the recipe in the module docstring.

    ``lengths`` gives the sequence lengths (ignored when ``len_range`` is set, in which
    case ``n_seqs`` lengths are drawn first). ``varlen`` defaults to True when the
    lengths differ. ``beta=False`` leaves beta out (the decay-only recurrence).
    """
    rng = np.random.default_rng(seed)
    if len_range is not None:
        lo, hi = len_range
        lengths = tuple(int(x) for x in rng.integers(lo, hi + 1, size=n_seqs))
    lengths = tuple(int(x) for x in lengths)
    if varlen is None:
        varlen = len(set(lengths)) > 1
    if not varlen and len(set(lengths)) > 1:
        raise ValueError("fixed-length batches need equal lengths")
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])

    q = _l2_normalise(_normal_rows(rng, T, H_k * d_k), H_k, d_k)
    k = _l2_normalise(_normal_rows(rng, T, H_k * d_k), H_k, d_k)
    v = _normal_rows(rng, T, H_v * d_v).reshape(T, H_v, d_v)

    gcols = H_v * d_k if gate == "channel" else H_v
    g = np.empty((T, gcols), dtype=np.float32)
    for s in range(0, T, _BLOCK):
        e = min(T, s + _BLOCK)
        a = rng.uniform(a_lo, 0.999, size=(e - s, gcols))
        g[s:e] = np.log(a).astype(np.float32)
    g = g.reshape(T, H_v, d_k) if gate == "channel" else g.reshape(T, H_v)

    b = None
    if beta:
        logits = _normal_rows(rng, T, H_v)
        b = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)

    hinit = None
    if h0:
        hinit = (0.1 * rng.standard_normal((len(lengths), H_v, d_k, d_v), dtype=np.float32)).astype(np.float32)

    return Inputs(
        q=round_to_dtype(q, dtype), k=round_to_dtype(k, dtype), v=round_to_dtype(v, dtype),
        g=g, beta=b, h0=hinit, cu_seqlens=cu, H_k=H_k, H_v=H_v, d_k=d_k, d_v=d_v,
        dtype=dtype, gate=gate, scale=float(d_k ** -0.5 if scale is None else scale),
        varlen=bool(varlen), meta={"seed": seed, "a_lo": a_lo},
    )


@dataclass
class FrontendInputs(Inputs):
    """Raw inputs of the fused front-end, as handed to the GPU.

    Where the matching switch is on, ``q`` and ``k`` are not normalised, ``g`` holds the
    gate pre-activation a (not the log gate) and ``beta`` holds the logits b (not beta);
    ``A_log`` [H_v] and ``dt_bias`` ([H_v, d_k] per-channel, [H_v] per-head) are the
    gate's per-head parameters (None when the gate is given directly)."""

    A_log: np.ndarray | None = None
    dt_bias: np.ndarray | None = None
    qk_l2norm: bool = True
    beta_sigmoid: bool = True


def make_frontend_inputs(lengths, H_k, H_v, d_k, d_v, *, dtype="bf16", gate="channel", h0=False,
                         beta=True, varlen=None, seed=0, scale=None, qk_l2norm=True,
                         beta_sigmoid=True, gate_act=True, qk_std=1.0) -> FrontendInputs:
    """Raw inputs for the fused front-end (one ``default_rng(seed)`` stream, in order):

    1. sequence lengths as given;
    2. q, k [T, H_k, d_k] ~ N(0, qk_std**2) fp32 (normalised per token and head as in
       :func:`make_inputs` when ``qk_l2norm`` is off);
    3. v [T, H_v, d_v] ~ N(0, 1);
    4. A_log [H_v] = log(U[0.5, 1]); dt_bias ~ U[-5.6, -3.4], one per (value head,
       channel) or per value head; a ~ U[-1.2, 1.2] per (token, value head, channel) or
       (token, value head). Then a + dt_bias lies in [-6.8, -2.2], softplus of it in
       [1.1e-3, 0.105], and the per-token decay exp(g) in [0.90, 0.9994]: the
       lower-bounded range (at least 0.9) that the Kimi Delta Attention page requires of
       the gate. With ``gate_act`` off, g = log(U[0.9, 0.999]) directly instead;
    5. b [T, H_v] ~ N(0, 1) logits (beta = sigmoid(b) stored instead when
       ``beta_sigmoid`` is off; nothing when ``beta`` is off);
    6. h0 [N, H_v, d_k, d_v] ~ N(0, 0.1**2), or none.
    """
    rng = np.random.default_rng(seed)
    lengths = tuple(int(x) for x in lengths)
    if varlen is None:
        varlen = len(set(lengths)) > 1
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])

    q = (qk_std * _normal_rows(rng, T, H_k * d_k)).astype(np.float32)
    k = (qk_std * _normal_rows(rng, T, H_k * d_k)).astype(np.float32)
    if qk_l2norm:
        q, k = q.reshape(T, H_k, d_k), k.reshape(T, H_k, d_k)
    else:
        q, k = _l2_normalise(q, H_k, d_k), _l2_normalise(k, H_k, d_k)
    v = _normal_rows(rng, T, H_v * d_v).reshape(T, H_v, d_v)

    gshape = (T, H_v, d_k) if gate == "channel" else (T, H_v)
    A_log = dt_bias = None
    if gate_act:
        A_log = np.log(rng.uniform(0.5, 1.0, size=H_v)).astype(np.float32)
        dt_bias = rng.uniform(-5.6, -3.4, size=gshape[1:]).astype(np.float32)
        g = rng.uniform(-1.2, 1.2, size=gshape).astype(np.float32)
    else:
        g = np.log(rng.uniform(0.9, 0.999, size=gshape)).astype(np.float32)

    b = None
    if beta:
        b = _normal_rows(rng, T, H_v)
        if not beta_sigmoid:
            b = (1.0 / (1.0 + np.exp(-b.astype(np.float64)))).astype(np.float32)

    hinit = None
    if h0:
        hinit = (0.1 * rng.standard_normal((len(lengths), H_v, d_k, d_v), dtype=np.float32)).astype(np.float32)

    return FrontendInputs(
        q=round_to_dtype(q, dtype), k=round_to_dtype(k, dtype), v=round_to_dtype(v, dtype),
        g=g, beta=b, h0=hinit, cu_seqlens=cu, H_k=H_k, H_v=H_v, d_k=d_k, d_v=d_v,
        dtype=dtype, gate=gate, scale=float(d_k ** -0.5 if scale is None else scale),
        varlen=bool(varlen), meta={"seed": seed, "frontend": True},
        A_log=A_log, dt_bias=dt_bias, qk_l2norm=bool(qk_l2norm),
        beta_sigmoid=bool(beta_sigmoid and beta),
    )


def workload_inputs(name: str, seed: int | None = None) -> Inputs:
    """Inputs of one named workload (seed defaults to the workload's fixed seed)."""
    w = WORKLOADS[name] if name in WORKLOADS else PROFILE_WORKLOADS[name]
    s = WORKLOAD_SEEDS.get(name, 99) if seed is None else seed
    x = make_inputs(w.lengths, w.H_k, w.H_v, w.d_k, w.d_v, dtype=w.dtype, gate=w.gate,
                    a_lo=w.a_lo, h0=w.h0, beta=w.beta, varlen=w.varlen, seed=s,
                    len_range=w.len_range, n_seqs=w.n_seqs)
    x.meta["workload"] = name
    return x


def workload_frontend_inputs(name: str, seed: int | None = None) -> FrontendInputs:
    """Raw front-end inputs with the shape of one named workload (its gate mode, beta and
    h0 choices): every front-end part switched on."""
    w = WORKLOADS[name] if name in WORKLOADS else PROFILE_WORKLOADS[name]
    if w.len_range is not None:
        lengths = tuple(int(v) for v in np.random.default_rng(WORKLOAD_SEEDS.get(name, 99))
                        .integers(w.len_range[0], w.len_range[1] + 1, size=w.n_seqs))
    else:
        lengths = w.lengths
    s = WORKLOAD_SEEDS.get(name, 99) if seed is None else seed
    x = make_frontend_inputs(lengths, w.H_k, w.H_v, w.d_k, w.d_v, dtype=w.dtype, gate=w.gate, h0=w.h0,
                             beta=w.beta, varlen=w.varlen, seed=s)
    x.meta["workload"] = name
    return x
