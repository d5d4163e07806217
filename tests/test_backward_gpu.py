"""GPU parity of the backward pass (kda_chunk_bwd) against the fp64 backward oracle.

The library's contractions run on tf32 tensor cores with fp32 accumulation; everything
else is fp32. Tolerances (relative L2 over each whole gradient tensor):
  * fp32 inputs: operands split into two tf32 parts (three products each), fp32-grade:
    1e-5 on every gradient (about 1e-6 measured);
  * bf16 inputs: operands rounded to tf32 once (unit roundoff 2^-11 = 4.9e-4, so about
    1e-3 per product), through a few chained products per chunk (dT, the two products
    with T for dL, dKm, the reverse cumulative sum): 5e-3 on dg, dbeta and dh0; dq, dk, dv
    are rounded to bf16 outputs as well (about 1.7e-3 from that rounding alone): 5e-3.
"""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from kda_cases import to_device

pytestmark = pytest.mark.gpu

TOL_BF16_OUT = 5e-3   # every gradient, bf16 inputs
TOL_F32 = 1e-5        # every gradient, fp32 inputs


def _run(x, do, dht, want_dh0=True):
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_bwd

    d = to_device(x)
    dt = d["q"].dtype
    B = d["q"].shape[0]
    T = d["q"].shape[1]
    do_t = torch.from_numpy(np.ascontiguousarray(do)).reshape(B, T, x.H_v, x.d_v).to("cuda", dt).contiguous()
    dht_t = None if dht is None else torch.from_numpy(dht).cuda().contiguous()
    r = chunk_kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do_t, h0=d["h0"], dht=dht_t, scale=x.scale,
                      cu_seqlens=d["cu_seqlens"], want_dh0=want_dh0)
    torch.cuda.synchronize()
    names = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
    out = {}
    for name, t in zip(names, r):
        if t is None:
            out[name] = None
            continue
        a = t.float().cpu().numpy().astype(np.float64)
        if name in ("dq", "dk"):
            a = a.reshape(x.T_total, x.H_k, x.d_k)
        elif name == "dv":
            a = a.reshape(x.T_total, x.H_v, x.d_v)
        elif name == "dg":
            a = a.reshape(x.g.shape)
        elif name == "dbeta":
            a = a.reshape(x.T_total, x.H_v)
        out[name] = a
    return out


def _cotangents(x, seed, dht=True):
    rng = np.random.default_rng(seed)
    do = rng.standard_normal(x.v.shape).astype(np.float32)
    if x.dtype == "bf16":
        from inputs.synth import round_to_dtype

        do = round_to_dtype(do, "bf16").reshape(x.v.shape)
    dh = rng.standard_normal((x.N, x.H_v, x.d_k, x.d_v)).astype(np.float32) if dht else None
    return do, dh


def _check(x, tag, seed=0, dht=True):
    from oracle import kda_recurrence_bwd

    do, dh = _cotangents(x, seed, dht)
    got = _run(x, do, dh)
    ref = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dh, x.cu_seqlens, x.scale)
    worst = {}
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        if ref[name] is None:
            assert got[name] is None
            continue
        assert np.isfinite(got[name]).all(), name
        e = rel_l2(got[name], ref[name])
        worst[name] = e
        tol = TOL_BF16_OUT if x.dtype == "bf16" else TOL_F32
        assert e <= tol, (tag, name, e)
    print(tag, " ".join(f"{k}={v:.2e}" for k, v in worst.items()))


@pytest.mark.parametrize("gate", ["channel", "head"])
def test_bf16_d128_varlen_gqa(gate):
    x = make_inputs((1, 63, 64, 65, 200, 0), 2, 4, 128, 128, seed=301, h0=True, varlen=True, gate=gate)
    _check(x, f"bf16 {gate} varlen gqa")


def test_decay_only():
    x = make_inputs((130, 70), 2, 2, 128, 128, seed=302, h0=True, beta=False)
    _check(x, "decay-only")


@pytest.mark.parametrize("d_k,d_v", [(64, 64), (64, 128), (128, 64)])
def test_fp32_head_sizes(d_k, d_v):
    x = make_inputs((100, 37), 1, 2, d_k, d_v, seed=303, dtype="f32", h0=True)
    _check(x, f"f32 dk{d_k} dv{d_v}")


def test_no_initial_state_no_final_gradient():
    x = make_inputs((150,), 2, 2, 128, 128, seed=304, h0=False)
    _check(x, "no h0, no dht", dht=False)


def test_long_sequence_fixed_batch():
    x = make_inputs((1000, 1000), 2, 2, 128, 128, seed=305, h0=True)
    _check(x, "bf16 2 x 1000")


def test_repeat_is_bitwise_identical():
    """One value head per key head (dq, dk written directly, no atomics), per-channel gates,
    bf16, d = 128, packed sequences with ragged tails: two calls give the same bits in every
    gradient (no reduction in the path depends on scheduling)."""
    x = make_inputs((63, 64, 200), 2, 2, 128, 128, seed=307, h0=True, varlen=True)
    do, dh = _cotangents(x, 8)
    first = _run(x, do, dh)
    second = _run(x, do, dh)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.array_equal(first[name], second[name]), name


def test_benchmark_shape_sampled_units():
    """B = 2, T = 8192, H = 32, d = 128 (the benchmark's shape): every gradient of three
    units against the oracle (grouped heads do not occur here, so a unit's dq and dk are
    the whole gradient of its key head)."""
    from oracle import kda_recurrence_bwd

    x = make_inputs((8192, 8192), 32, 32, 128, 128, seed=306, h0=True)
    do, dh = _cotangents(x, 7)
    got = _run(x, do, dh)
    units = [(0, 3), (1, 30), (1, 0)]
    ref = kda_recurrence_bwd(x.q, x.k, x.v, x.g, x.beta, x.h0, do, dh, x.cu_seqlens, x.scale, units=units)
    T = 8192
    for (n, h), r in zip(units, ref):
        sl = slice(n * T, (n + 1) * T)
        errs = {"dq": rel_l2(got["dq"][sl, h], r["dq"]), "dk": rel_l2(got["dk"][sl, h], r["dk"]),
                "dv": rel_l2(got["dv"][sl, h], r["dv"]), "dg": rel_l2(got["dg"][sl, h], r["dg"]),
                "dbeta": rel_l2(got["dbeta"][sl, h], r["dbeta"]), "dh0": rel_l2(got["dh0"][n, h], r["dh0"])}
        print((n, h), " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
        for name, e in errs.items():
            assert e <= TOL_BF16_OUT, ((n, h), name, e)


@pytest.mark.parametrize("bad", [[0, 90, 60], [0, 90, 150]])
def test_malformed_cu_seqlens_raise_the_device_error(bad):
    """Decreasing offsets, or offsets past the packed length, are caught on the device: the
    sequence is skipped and the error bit raised (no access outside the tensors)."""
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_bwd, kda_get_device_error

    x = make_inputs((64, 36), 1, 1, 128, 128, seed=307, varlen=True)
    d = to_device(x)
    stream = torch.cuda.current_stream().cuda_stream
    assert kda_get_device_error(stream) == 0
    cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
    do = torch.zeros_like(d["v"])
    chunk_kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do, scale=x.scale, cu_seqlens=cu)
    assert kda_get_device_error(stream) == 1
    assert kda_get_device_error(stream) == 0


@pytest.mark.parametrize("case", ["gqa4_head_decay", "bf16_d64", "f32_head_varlen"])
def test_more_shapes(case):
    if case == "gqa4_head_decay":
        # four value heads per key head, scalar gate, no beta
        x = make_inputs((100, 29), 1, 4, 128, 128, seed=308, h0=True, gate="head", beta=False)
    elif case == "bf16_d64":
        x = make_inputs((170,), 2, 2, 64, 64, seed=309, h0=True)
    else:
        x = make_inputs((5, 64, 0, 140), 2, 2, 128, 64, seed=310, dtype="f32", h0=True, gate="head",
                        varlen=True)
    _check(x, case)


def test_backward_scratch_goes_back_to_the_device():
    """The backward's scratch (about 5.8 GB on the benchmark shape) comes from the library's
    pool and is freed on the stream; at the next synchronisation the pool gives back all
    but at most 64 MiB, so the device's free memory returns to within that of its value
    before the call."""
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_bwd

    B, T, H, D = 2, 8192, 32, 128
    gen = torch.Generator(device="cuda").manual_seed(11)
    q = torch.nn.functional.normalize(torch.randn(B, T, H, D, device="cuda", generator=gen), dim=-1).bfloat16()
    k = torch.nn.functional.normalize(torch.randn(B, T, H, D, device="cuda", generator=gen), dim=-1).bfloat16()
    v = torch.randn(B, T, H, D, device="cuda", generator=gen).bfloat16()
    g = torch.log(torch.empty(B, T, H, D, device="cuda").uniform_(0.9, 0.999, generator=gen))
    beta = torch.rand(B, T, H, device="cuda", generator=gen)
    do = torch.randn(B, T, H, D, device="cuda", generator=gen).bfloat16()
    r = chunk_kda_bwd(q, k, v, g, beta, do)  # torch's cache now holds blocks for the gradients
    del r
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    r = chunk_kda_bwd(q, k, v, g, beta, do)
    del r
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 <= (64 << 20) + (4 << 20), (free0, free1)
