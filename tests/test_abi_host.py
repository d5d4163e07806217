"""The C-ABI library on the host: it loads, exports what include/kda.h declares, and
rejects bad arguments before touching the GPU (no compute call is made here)."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from chunkwise_gated_linear_gb300 import kda

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    L = kda.lib()
    names = _declared_functions()
    assert set(names) == set(kda.EXPORTED)
    for name in names:
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings():
    assert kda.status_string(kda.KDA_OK) == "KDA_OK"
    for st in (kda.KDA_ERR_INVALID_ARG, kda.KDA_ERR_UNSUPPORTED, kda.KDA_ERR_ALIGNMENT):
        assert kda.status_string(st).startswith("KDA_ERR_")
    assert "unknown" in kda.status_string(12345)


# Fake, 16-byte aligned addresses: every case below is rejected by the host checks,
# which run before any CUDA call, so nothing is dereferenced.
A = 1 << 20


def _call(**over):
    args = dict(q=A, k=A, v=A, g=A, beta=A, h0=0, o=A, ht=0, B=1, T=64, H_k=1, H_v=1, d_k=128,
                d_v=128, C=64, scale=1.0, cu_seqlens=0, stream=0)
    args.update(over)
    return kda.kda_chunk_fwd(**args)


@pytest.mark.parametrize("over,want", [
    (dict(q=0), kda.KDA_ERR_INVALID_ARG),
    (dict(k=0), kda.KDA_ERR_INVALID_ARG),
    (dict(v=0), kda.KDA_ERR_INVALID_ARG),
    (dict(g=0), kda.KDA_ERR_INVALID_ARG),
    (dict(o=0), kda.KDA_ERR_INVALID_ARG),
    (dict(B=0), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(H_k=0), kda.KDA_ERR_INVALID_ARG),
    (dict(H_k=3, H_v=4), kda.KDA_ERR_INVALID_ARG),
    (dict(d_k=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(d_v=256), kda.KDA_ERR_UNSUPPORTED),
    (dict(C=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(q=A + 8), kda.KDA_ERR_ALIGNMENT),
    (dict(o=A + 4), kda.KDA_ERR_ALIGNMENT),
    (dict(h0=A + 2), kda.KDA_ERR_ALIGNMENT),
    (dict(ht=A + 12), kda.KDA_ERR_ALIGNMENT),
])
def test_bad_arguments_are_rejected(over, want):
    assert _call(**over) == want


def test_ex_rejects_unknown_modes_and_flags():
    p = kda.kda_fwd_params(A, A, A, A, A, None, A, None, 1, 64, 1, 1, 128, 128, 64, 1.0, None,
                           kda.KDA_DTYPE_BF16, kda.KDA_GATE_PER_CHANNEL, 8)
    assert kda.kda_chunk_fwd_ex(p, 0) == kda.KDA_ERR_INVALID_ARG
    p.flags = kda.KDA_FLAG_ONE_CTA_PER_UNIT | kda.KDA_FLAG_UNFUSED_FRONTEND | kda.KDA_FLAG_DEBUG_SHORT_WAITS | 16
    assert kda.kda_chunk_fwd_ex(p, 0) == kda.KDA_ERR_INVALID_ARG
    p.flags = 0
    p.dtype = 7
    assert kda.kda_chunk_fwd_ex(p, 0) == kda.KDA_ERR_UNSUPPORTED
    p.dtype = kda.KDA_DTYPE_F32
    p.gate_mode = 5
    assert kda.kda_chunk_fwd_ex(p, 0) == kda.KDA_ERR_UNSUPPORTED
    assert kda.lib().kda_chunk_fwd_ex(None, None) == kda.KDA_ERR_INVALID_ARG


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    # checked on the host before any CUDA call: more than 16 units, or d != 128
    args = dict(q=A, k=A, v=A, g=A, beta=A, h0=0, o=A, ht=0, B=1, T=64, H_k=1, H_v=17, d_k=128,
                d_v=128, C=64, scale=1.0, cu_seqlens=0, stream=0)
    assert kda.kda_chunk_fwd_noalloc(**args) == kda.KDA_ERR_UNSUPPORTED
    args.update(B=2, H_v=16)  # 32 units
    assert kda.kda_chunk_fwd_noalloc(**args) == kda.KDA_ERR_UNSUPPORTED
    args.update(B=1, H_v=4, d_k=64)
    assert kda.kda_chunk_fwd_noalloc(**args) == kda.KDA_ERR_UNSUPPORTED
    args.update(d_k=128, q=0)
    assert kda.kda_chunk_fwd_noalloc(**args) == kda.KDA_ERR_INVALID_ARG


def test_fused_front_end_rejections():
    # all checked on the host before any CUDA call
    p = kda.kda_fwd_params(A, A, A, A, A, None, A, None, 1, 64, 1, 1, 128, 128, 64, 1.0, None,
                           kda.KDA_DTYPE_BF16, kda.KDA_GATE_PER_CHANNEL, 0)
    for fn in (kda.kda_chunk_fwd_fused, kda.kda_recurrent_fwd_fused):
        # dt_bias without A_log
        assert fn(p, kda.kda_frontend(0, 0, None, A), 0) == kda.KDA_ERR_INVALID_ARG
        # misaligned gate parameters
        assert fn(p, kda.kda_frontend(0, 0, A + 4, None), 0) == kda.KDA_ERR_ALIGNMENT
        assert fn(p, kda.kda_frontend(0, 0, A, A + 8), 0) == kda.KDA_ERR_ALIGNMENT
        # beta logits without beta
        p.beta = None
        assert fn(p, kda.kda_frontend(0, 1, None, None), 0) == kda.KDA_ERR_INVALID_ARG
        p.beta = A
        # the base checks still apply
        p.d_k = 96
        assert fn(p, kda.kda_frontend(1, 1, A, A), 0) == kda.KDA_ERR_UNSUPPORTED
        p.d_k = 128
    assert kda.lib().kda_chunk_fwd_fused(None, None, None) == kda.KDA_ERR_INVALID_ARG


def test_backward_rejections():
    # all checked on the host before any CUDA call
    def params(**over):
        p = kda.kda_bwd_params(A, A, A, A, A, None, A, None, A, A, A, A, A, None, 1, 64, 1, 1, 128, 128,
                               64, 1.0, None, kda.KDA_DTYPE_BF16, kda.KDA_GATE_PER_CHANNEL, 0)
        for key, val in over.items():
            setattr(p, key, val)
        return p

    assert kda.kda_chunk_bwd(params(flags=1), 0) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_chunk_bwd(params(dO=None), 0) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_chunk_bwd(params(dq=None), 0) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_chunk_bwd(params(dbeta=None), 0) == kda.KDA_ERR_INVALID_ARG   # beta without dbeta
    assert kda.kda_chunk_bwd(params(beta=None), 0) == kda.KDA_ERR_INVALID_ARG    # dbeta without beta
    assert kda.kda_chunk_bwd(params(dO=A + 4), 0) == kda.KDA_ERR_ALIGNMENT
    assert kda.kda_chunk_bwd(params(dh0=A + 8), 0) == kda.KDA_ERR_ALIGNMENT
    assert kda.kda_chunk_bwd(params(d_k=96), 0) == kda.KDA_ERR_UNSUPPORTED
    assert kda.kda_chunk_bwd(params(C=32), 0) == kda.KDA_ERR_UNSUPPORTED
    assert kda.lib().kda_chunk_bwd(None, None) == kda.KDA_ERR_INVALID_ARG
