"""Helpers shared by the GPU tests: move seeded inputs to the device, run the library
through its Python binding, and run the oracle on the same values."""

from __future__ import annotations

import numpy as np

from inputs import Inputs

TOL = {"bf16": 2e-2, "f32": 1e-5}  # relative L2 on o and on ht, vs the fp64 oracle


def to_device(x: Inputs, device="cuda"):
    """Torch tensors laid out as the ABI wants them (fixed batches [B, T, ...], packed
    sequences [1, T_total, ...] with cu_seqlens)."""
    import torch

    dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    if x.varlen:
        B, T = 1, x.T_total
    else:
        B = x.N
        T = x.T_total // max(B, 1)

    def tens(a, dtype):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.reshape(B, T, *a.shape[1:]).to(device=device, dtype=dtype).contiguous()

    d = {
        "q": tens(x.q, dt), "k": tens(x.k, dt), "v": tens(x.v, dt),
        "g": tens(x.g, torch.float32), "beta": None if x.beta is None else tens(x.beta, torch.float32),
        "h0": None if x.h0 is None else torch.from_numpy(x.h0).to(device).contiguous(),
        "cu_seqlens": torch.from_numpy(x.cu_seqlens.astype(np.int32)).to(device) if x.varlen else None,
    }
    return d


def run_gpu(x: Inputs, d=None, **kw):
    """(o [T_total, H_v, d_v] float64, ht [N, H_v, d_k, d_v] float64) from the library."""
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    if d is None:
        d = to_device(x)
    o, ht = chunk_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], scale=x.scale,
                          cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    o = o.float().cpu().numpy().reshape(x.T_total, x.H_v, x.d_v).astype(np.float64)
    ht = None if ht is None else ht.cpu().numpy().astype(np.float64)
    return o, ht


def run_oracle(x: Inputs, units=None):
    from oracle import kda_recurrence

    return kda_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale, units=units)


def run_gpu_fe(x, d=None, **kw):
    """run_gpu for front-end inputs (:class:`inputs.FrontendInputs`): the raw q, k, a and b
    go in with the front-end switched on as the inputs say."""
    import torch

    if d is None:
        d = to_device(x)
    dev = d["q"].device
    A_log = None if x.A_log is None else torch.from_numpy(x.A_log).to(dev).contiguous()
    dt_bias = None if x.dt_bias is None else torch.from_numpy(x.dt_bias).to(dev).contiguous()
    return run_gpu(x, d, qk_l2norm=x.qk_l2norm, beta_sigmoid=x.beta_sigmoid, A_log=A_log,
                   dt_bias=dt_bias, **kw)


def run_oracle_fe(x, units=None):
    from oracle import kda_fused_recurrence

    return kda_fused_recurrence(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, x.scale,
                                qk_l2norm=x.qk_l2norm, beta_sigmoid=x.beta_sigmoid, A_log=x.A_log,
                                dt_bias=x.dt_bias, units=units)
