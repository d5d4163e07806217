"""Chunkwise forward pass of the gated delta rule with a per-channel gate (Kimi Delta
Attention) for GB300 (sm_103a): a C-ABI CUDA library (``include/kda.h``,
``lib/libkda.so``) and its thin Python binding (:mod:`.kda`)."""

from .kda import (  # noqa: F401
    KdaError,
    chunk_kda_bwd,
    chunk_kda_fwd,
    kda_bwd_params,
    kda_chunk_bwd,
    kda_chunk_fwd,
    kda_chunk_fwd_ex,
    kda_chunk_fwd_f32,
    kda_chunk_fwd_fused,
    kda_chunk_fwd_noalloc,
    kda_frontend,
    kda_fwd_params,
    kda_get_device_error,
    kda_recurrent_fwd,
    kda_recurrent_fwd_ex,
    kda_recurrent_fwd_fused,
    lib,
    status_string,
)
