"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Small cases span several 64-token chunks with ragged tails, grouped heads, both gate
modes, both dtypes, every (d_k, d_v) pair and the degenerate inputs (empty sequences,
one-token sequences, beta = 0). The tolerance is relative L2 over the whole o tensor and
over the whole ht tensor: 2e-2 for bf16 inputs with fp32 accumulation, 1e-5 for fp32.
"""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from kda_cases import TOL, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _check(x, tag="", **kw):
    o, ht = run_gpu(x, **kw)
    o_r, ht_r = run_oracle(x)
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    e_o, e_h = rel_l2(o, o_r), rel_l2(ht, ht_r)
    print(f"{tag} rel_l2 o={e_o:.3e} ht={e_h:.3e}")
    tol = TOL[x.dtype]
    assert e_o <= tol, (tag, e_o)
    assert e_h <= tol, (tag, e_h)
    return o, ht


@pytest.mark.parametrize("d_k,d_v", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_bf16_per_channel_ragged(d_k, d_v):
    x = make_inputs((200,), 2, 2, d_k, d_v, seed=101, h0=True)
    _check(x, f"bf16 dk{d_k} dv{d_v}")


def test_bf16_varlen_gqa_edge_lengths():
    x = make_inputs((1, 63, 64, 65, 130, 0, 7, 200), 2, 4, 128, 128, seed=102, h0=True, varlen=True,
                    a_lo=0.8)
    _check(x, "bf16 varlen gqa")


def test_bf16_per_head_gate_matches_broadcast_channel_gate():
    x = make_inputs((150, 150), 2, 2, 128, 128, seed=103, gate="head")
    o_h, ht_h = _check(x, "bf16 per-head gate")
    xb = make_inputs((150, 150), 2, 2, 128, 128, seed=103, gate="head")
    xb.g = np.ascontiguousarray(np.repeat(xb.g[:, :, None], 128, axis=2))
    xb.gate = "channel"
    o_c, ht_c = run_gpu(xb)
    assert rel_l2(o_c, o_h) < 1e-6 and rel_l2(ht_c, ht_h) < 1e-6


def test_bf16_strong_gates_and_no_initial_state():
    x = make_inputs((333,), 1, 2, 128, 128, seed=104, a_lo=0.8)
    _check(x, "bf16 a>=0.8")


def test_bf16_beta_zero_is_decay_of_h0():
    x = make_inputs((130,), 1, 1, 128, 128, seed=105, h0=True)
    x.beta[:] = 0.0
    _check(x, "bf16 beta=0")


@pytest.mark.parametrize("d", [64, 128])
def test_f32_path(d):
    x = make_inputs((256,), 1, 1, d, d, seed=106, dtype="f32")
    _check(x, f"f32 d{d}")
    y = make_inputs((70, 1, 129), 1, 2, d, d, seed=107, dtype="f32", h0=True, varlen=True,
                    gate="head")
    _check(y, f"f32 varlen d{d}")


def test_empty_batch_keeps_initial_state():
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    x = make_inputs((0,), 1, 2, 128, 128, seed=108, h0=True)
    d = to_device(x)
    o, ht = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale)
    torch.cuda.synchronize()
    assert o.numel() == 0
    np.testing.assert_array_equal(ht.cpu().numpy(), x.h0)


def test_deterministic_and_dv_halves_agree_across_kernels():
    """Two calls give bitwise-equal results. The two 64-wide d_v halves, run as calls of
    their own, go through another kernel (d_v = 64 selects the mma.sync kernel), so they are
    compared with the d = 128 result up to rounding; the bitwise slice invariance of one
    kernel is test_dv_slices_are_bitwise_invariant."""
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    x = make_inputs((190,), 2, 2, 128, 128, seed=109, h0=True)
    d = to_device(x)
    o1, h1 = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale)
    o2, h2 = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    # the two d_v halves run on their own ("TileLang 实战：KDA 从零到一–Kimi Delta Attention"
    # §3.4: slicing d_v introduces no dependence) give the same result up to rounding
    for s in (slice(0, 64), slice(64, 128)):
        vs = d["v"][..., s].contiguous()
        hs = d["h0"][..., s].contiguous()
        os_, hts = chunk_kda_fwd(d["q"], d["k"], vs, d["g"], d["beta"], h0=hs, scale=x.scale)
        torch.cuda.synchronize()
        assert rel_l2(os_.float().cpu().numpy(), o1[..., s].float().cpu().numpy()) < 1e-2
        assert rel_l2(hts.cpu().numpy(), h1[..., s].cpu().numpy()) < 1e-2


@pytest.mark.parametrize("dtype,d_k", [("bf16", 64), ("f32", 128)])
def test_dv_slices_are_bitwise_invariant(dtype, d_k):
    """Slicing d_v adds no dependence ("TileLang 实战：KDA 从零到一–Kimi Delta Attention",
    §3.4): the kernels that split d_v into 64-wide slices (one CTA each: the bf16 kernel at
    d_k = 64 and the fp32 kernel) give, for each slice of a d_v = 128 call, exactly the bits
    of a d_v = 64 call on that slice alone."""
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    x = make_inputs((200, 200), 1, 2, d_k, 128, seed=110, h0=True, dtype=dtype)
    d = to_device(x)
    o1, h1 = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale)
    for s in (slice(0, 64), slice(64, 128)):
        vs = d["v"][..., s].contiguous()
        hs = d["h0"][..., s].contiguous()
        os_, hts = chunk_kda_fwd(d["q"], d["k"], vs, d["g"], d["beta"], h0=hs, scale=x.scale)
        torch.cuda.synchronize()
        assert torch.equal(os_, o1[..., s].contiguous())
        assert torch.equal(hts, h1[..., s].contiguous())


def test_resume_from_final_state():
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    x = make_inputs((256,), 1, 1, 128, 128, seed=110, h0=True)
    d = to_device(x)
    o, ht = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale)
    T1 = 128  # a chunk boundary: the split run follows the same chunking
    cut = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
    o1, h1 = chunk_kda_fwd(cut(d["q"], 0, T1), cut(d["k"], 0, T1), cut(d["v"], 0, T1),
                           cut(d["g"], 0, T1), cut(d["beta"], 0, T1), h0=d["h0"], scale=x.scale)
    o2, h2 = chunk_kda_fwd(cut(d["q"], T1, 256), cut(d["k"], T1, 256), cut(d["v"], T1, 256),
                           cut(d["g"], T1, 256), cut(d["beta"], T1, 256), h0=h1, scale=x.scale)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o1, o2], dim=1), o) and torch.equal(h2, ht)


@pytest.mark.parametrize("one_cta", [False, True])
def test_malformed_cu_seqlens_raise_the_device_error(one_cta):
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd, kda_get_device_error

    x = make_inputs((64, 36), 1, 1, 128, 128, seed=111, varlen=True)
    d = to_device(x)
    stream = torch.cuda.current_stream().cuda_stream
    assert kda_get_device_error(stream) == 0
    bad = torch.tensor([0, 90, 60], dtype=torch.int32, device="cuda")  # decreasing
    chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x.scale, cu_seqlens=bad,
                  one_cta_per_unit=one_cta)
    assert kda_get_device_error(stream) == 1
    assert kda_get_device_error(stream) == 0  # the query clears it


# d_k = d_v = 128 in bf16 has two kernels: the persistent producer/consumer kernel (few
# units) and one CTA per unit (many units, or KDA_FLAG_ONE_CTA_PER_UNIT). Both are held
# to the oracle on the same inputs, and to each other.
@pytest.mark.parametrize("one_cta", [False, True])
@pytest.mark.parametrize("case", ["varlen_gqa", "head_gate", "long_ragged"])
def test_bf16_d128_both_kernels(case, one_cta):
    if case == "varlen_gqa":
        x = make_inputs((1, 63, 64, 65, 130, 0, 7, 200), 2, 4, 128, 128, seed=112, h0=True,
                        varlen=True)
    elif case == "head_gate":
        x = make_inputs((150, 150), 2, 2, 128, 128, seed=113, gate="head", h0=True)
    else:
        # 16 chunks per unit: the ring of chunk slots wraps several times
        x = make_inputs((1000, 1000), 1, 1, 128, 128, seed=114, h0=True)
    _check(x, f"{case} one_cta={one_cta}", one_cta_per_unit=one_cta)


def test_bf16_d128_persistent_many_jobs_per_producer():
    # 8 units x 64 chunks = 512 chunk jobs: every producer CTA takes several in a row, and
    # its two stages and the ring run many laps
    x = make_inputs((4096,), 8, 8, 128, 128, seed=116, h0=True)
    _check(x, "persistent, many jobs")


def test_bf16_d128_kernels_agree():
    x = make_inputs((500, 77, 321), 2, 4, 128, 128, seed=115, h0=True, varlen=True)
    o1, h1 = run_gpu(x)
    o2, h2 = run_gpu(x, one_cta_per_unit=True)
    o_r, h_r = run_oracle(x)
    e1, e2 = rel_l2(o1, o_r), rel_l2(o2, o_r)
    print(f"persistent o={e1:.3e} ht={rel_l2(h1, h_r):.3e}; one CTA per unit o={e2:.3e} "
          f"ht={rel_l2(h2, h_r):.3e}; between them o={rel_l2(o1, o2):.3e}")
    # the same products in bf16 with fp32 accumulation; the persistent kernel hands U^T
    # from producer to consumer in bf16, one more rounding of the size of a bf16 operand,
    # so the two differ by about the bf16 unit roundoff and are equally close to the oracle
    assert rel_l2(o1, o2) < 8e-3 and rel_l2(h1, h2) < 8e-3
    assert abs(e1 - e2) < 2e-3


# beta = NULL: the decay-only recurrence S <- Diag(a_t) S + k_t v_t^T, against the
# oracle's decay-only path, on every kernel and both gate modes
@pytest.mark.parametrize("case", ["d128", "d128_one_cta", "d64", "f32", "head_gate_varlen"])
def test_decay_only(case):
    kw = {}
    if case.startswith("d128"):
        x = make_inputs((300, 300), 2, 4, 128, 128, seed=140, h0=True, beta=False)
        kw = {"one_cta_per_unit": case.endswith("one_cta")}
    elif case == "d64":
        x = make_inputs((200,), 2, 2, 64, 64, seed=141, h0=True, beta=False)
    elif case == "f32":
        x = make_inputs((130, 70), 1, 2, 128, 128, seed=142, dtype="f32", varlen=True, beta=False)
    else:
        x = make_inputs((1, 64, 190), 2, 2, 128, 128, seed=143, gate="head", h0=True, varlen=True,
                        beta=False)
    assert x.beta is None
    _check(x, f"decay-only {case}", **kw)


def test_decay_only_benchmark_shape_sampled():
    from inputs import workload_inputs

    x = workload_inputs("kda_decayonly_b2_t8192_h32_d128_bf16")
    o, ht = run_gpu(x)
    units = [(0, 0), (1, 31), (0, 17)]
    res = run_oracle(x, units=units)
    for (n, h), (ou, hu) in zip(units, res):
        s, e = x.cu_seqlens[n], x.cu_seqlens[n + 1]
        eo, eh = rel_l2(o[s:e, h], ou), rel_l2(ht[n, h], hu)
        print(f"decay-only 2x8192x32: unit ({n}, {h}) rel_l2 o={eo:.3e} ht={eh:.3e}")
        assert eo <= TOL["bf16"] and eh <= TOL["bf16"]


def _guarded(shape, dtype, pattern):
    """A tensor of `shape` inside a larger buffer whose 4096-element head and tail hold a
    known bit pattern (the caller checks them after the call)."""
    import torch

    n = int(np.prod(shape))
    itype = torch.int16 if dtype == torch.bfloat16 else torch.int32
    buf = torch.full((4096 + n + 4096,), pattern, dtype=itype, device="cuda")
    return buf, buf[4096:4096 + n].view(dtype).view(*shape)


def _guards_intact(buf, n, pattern):
    return bool((buf[:4096] == pattern).all()) and bool((buf[4096 + n:] == pattern).all())


@pytest.mark.parametrize("case", ["persistent_varlen", "one_cta_varlen", "d64_ragged", "f32_ragged",
                                  "persistent_decay_only_ragged"])
def test_outputs_leave_their_neighbours_untouched(case):
    """o and ht are written inside their extents only: each sits between guard bands of a
    known pattern, checked after the call (packed sequences and ragged tails are where a
    stray write would land)."""
    import torch

    if case in ("persistent_varlen", "one_cta_varlen"):
        x = make_inputs((1, 63, 64, 65, 130, 0, 7, 200), 2, 4, 128, 128, seed=140, h0=True, varlen=True)
    elif case == "d64_ragged":
        x = make_inputs((201, 201), 1, 2, 64, 64, seed=141, h0=True)
    elif case == "f32_ragged":
        x = make_inputs((137, 137), 1, 1, 64, 128, seed=142, h0=True, dtype="f32")
    else:
        x = make_inputs((333,), 1, 2, 128, 128, seed=143, h0=True, beta=False)
    d = to_device(x)
    dt = d["q"].dtype
    o_pat = 0x7FA5 if dt == torch.bfloat16 else 0x7FC0DEAD
    h_pat = 0x7FC0BEEF
    o_buf, o = _guarded(d["v"].shape, dt, o_pat)
    h_buf, ht = _guarded((x.N, x.H_v, x.d_k, x.d_v), torch.float32, h_pat)
    o, ht = run_gpu(x, d, o=o, ht=ht, one_cta_per_unit=(case == "one_cta_varlen"))
    o_r, ht_r = run_oracle(x)
    assert rel_l2(o, o_r) <= TOL[x.dtype] and rel_l2(ht, ht_r) <= TOL[x.dtype]
    assert _guards_intact(o_buf, int(np.prod(d["v"].shape)), o_pat)
    assert _guards_intact(h_buf, x.N * x.H_v * x.d_k * x.d_v, h_pat)


@pytest.mark.parametrize("case", ["persistent", "one_cta", "d64", "f32", "recurrent"])
def test_no_final_state_requested(case):
    """ht = NULL (output_final_state=False): nothing is written for it and o still matches
    the oracle, on every forward kernel."""
    kw = {}
    if case in ("persistent", "one_cta"):
        x = make_inputs((300, 300), 2, 2, 128, 128, seed=150, h0=True)
        kw["one_cta_per_unit"] = case == "one_cta"
    elif case == "d64":
        x = make_inputs((250,), 1, 1, 64, 64, seed=151, h0=True)
    elif case == "f32":
        x = make_inputs((190,), 1, 1, 128, 64, seed=152, h0=True, dtype="f32")
    else:
        x = make_inputs((40,), 1, 2, 128, 128, seed=153, h0=True)
        kw["recurrent"] = True
    o, ht = run_gpu(x, output_final_state=False, **kw)
    assert ht is None
    o_r, _ = run_oracle(x)
    assert rel_l2(o, o_r) <= TOL[x.dtype]
