"""The forward's failure path on the GPU, driven without any fault.

A test-only flag (KDA_FLAG_DEBUG_SHORT_WAITS) gives the one-CTA-per-unit kernel's bounded
waits a limit of about a thousand SM cycles, far shorter than a chunk takes to arrive, so
that they run out. The kernel then drains its copies and tensor-core work, frees its tensor
memory and returns, and the call reports KDA_DEVICE_ERR_TIMEOUT through
kda_get_device_error. The next ordinary call on the same stream must match the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from kda_cases import TOL, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def test_short_waits_raise_the_timeout_and_the_next_call_is_correct():
    import torch

    from chunkwise_gated_linear_gb300 import kda as K

    stream = torch.cuda.current_stream().cuda_stream
    x = make_inputs((512, 512), 2, 2, 128, 128, seed=301, h0=True)
    d = to_device(x)
    K.kda_get_device_error(stream)  # clear bits left by earlier calls
    o = torch.empty(d["v"].shape, dtype=torch.bfloat16, device="cuda")
    ht = torch.empty((x.N, x.H_v, 128, 128), dtype=torch.float32, device="cuda")
    T = x.T_total // x.N
    p = K.kda_fwd_params(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                         d["beta"].data_ptr(), d["h0"].data_ptr(), o.data_ptr(), ht.data_ptr(), x.N, T,
                         x.H_k, x.H_v, 128, 128, 64, x.scale, None, K.KDA_DTYPE_BF16,
                         K.KDA_GATE_PER_CHANNEL, K.KDA_FLAG_DEBUG_SHORT_WAITS)
    assert K.kda_chunk_fwd_ex(p, stream) == K.KDA_OK
    assert K.kda_get_device_error(stream) & K.KDA_DEVICE_ERR_TIMEOUT
    assert K.kda_get_device_error(stream) == 0  # read once, then cleared

    # the device and the stream are still usable: an ordinary call, then the oracle
    for one_cta in (True, False):
        o2, ht2 = run_gpu(x, d, one_cta_per_unit=one_cta)
        o_r, ht_r = run_oracle(x)
        assert rel_l2(o2, o_r) <= TOL["bf16"] and rel_l2(ht2, ht_r) <= TOL["bf16"]
    assert K.kda_get_device_error(stream) == 0

