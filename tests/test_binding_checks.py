"""The Python binding's argument checks (host only, no GPU): every tensor's shape and dtype
is checked before anything reaches the library, whose kernels cannot check a raw pointer's
extent. CPU tensors of the right shapes get as far as the device check."""

from __future__ import annotations

import pytest

torch = pytest.importorskip("torch")


def _fwd_args(B=1, T=70, H=2, D=128, dtype=torch.bfloat16):
    q = torch.zeros(B, T, H, D, dtype=dtype)
    k = torch.zeros(B, T, H, D, dtype=dtype)
    v = torch.zeros(B, T, H, D, dtype=dtype)
    g = torch.zeros(B, T, H, D, dtype=torch.float32)
    beta = torch.zeros(B, T, H, dtype=torch.float32)
    return q, k, v, g, beta


def test_forward_well_formed_reaches_the_device_check():
    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    q, k, v, g, beta = _fwd_args()
    h0 = torch.zeros(1, 2, 128, 128)
    o = torch.zeros(1, 70, 2, 128, dtype=torch.bfloat16)
    ht = torch.zeros(1, 2, 128, 128)
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        chunk_kda_fwd(q, k, v, g, beta, h0=h0, o=o, ht=ht)


@pytest.mark.parametrize("what", ["h0", "o_shape", "o_dtype", "ht", "cu_dtype", "cu_dim", "beta"])
def test_forward_rejects_malformed_arguments(what):
    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    q, k, v, g, beta = _fwd_args()
    kw = {}
    if what == "h0":
        kw["h0"] = torch.zeros(1, 2, 128, 64)
    elif what == "o_shape":
        kw["o"] = torch.zeros(1, 70, 2, 64, dtype=torch.bfloat16)
    elif what == "o_dtype":
        kw["o"] = torch.zeros(1, 70, 2, 128, dtype=torch.float32)
    elif what == "ht":
        kw["ht"] = torch.zeros(2, 2, 128, 128)
    elif what == "cu_dtype":
        kw["cu_seqlens"] = torch.tensor([0, 30, 70], dtype=torch.int64)
    elif what == "cu_dim":
        kw["cu_seqlens"] = torch.tensor([[0, 30, 70]], dtype=torch.int32)
    else:
        beta = torch.zeros(1, 70, 3)
    with pytest.raises((ValueError, TypeError)) as ei:
        chunk_kda_fwd(q, k, v, g, beta, **kw)
    assert "CUDA" not in str(ei.value)


def test_forward_ht_is_ignored_without_final_state():
    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    q, k, v, g, beta = _fwd_args()
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        chunk_kda_fwd(q, k, v, g, beta, ht=torch.zeros(3), output_final_state=False)


def test_backward_well_formed_reaches_the_device_check():
    from chunkwise_gated_linear_gb300 import chunk_kda_bwd

    q, k, v, g, beta = _fwd_args()
    do = torch.zeros_like(v)
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        chunk_kda_bwd(q, k, v, g, beta, do, h0=torch.zeros(1, 2, 128, 128), dht=torch.zeros(1, 2, 128, 128))


@pytest.mark.parametrize("what", ["g_dtype", "beta_shape", "beta_dtype", "h0", "dht", "cu_dtype", "do"])
def test_backward_rejects_malformed_arguments(what):
    from chunkwise_gated_linear_gb300 import chunk_kda_bwd

    q, k, v, g, beta = _fwd_args()
    do = torch.zeros_like(v)
    kw = {}
    if what == "g_dtype":
        g = g.to(torch.bfloat16)
    elif what == "beta_shape":
        beta = torch.zeros(1, 70, 3)
    elif what == "beta_dtype":
        beta = beta.to(torch.bfloat16)
    elif what == "h0":
        kw["h0"] = torch.zeros(1, 2, 64, 128)
    elif what == "dht":
        kw["dht"] = torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16)
    elif what == "cu_dtype":
        kw["cu_seqlens"] = torch.tensor([0, 30, 70], dtype=torch.int64)
    else:
        do = torch.zeros(1, 70, 2, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, TypeError)) as ei:
        chunk_kda_bwd(q, k, v, g, beta, do, **kw)
    assert "CUDA" not in str(ei.value)
