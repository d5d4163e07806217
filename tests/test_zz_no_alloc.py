"""kda_chunk_fwd_noalloc (scratch in a fixed device array, nothing allocated) against
kda_chunk_fwd on the same inputs, on two consecutive calls with different inputs (the
second call finds the array as the first left it), with and without beta, h0 and ht; and
the property the entry point exists for: a call allocates no device memory."""

from __future__ import annotations

import os
import subprocess
import sys

import pytest

from inputs import make_inputs
from kda_cases import to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _call(fn, d, x, o, ht, stream, use_h0=True):
    B = 1 if x.varlen else x.N
    T = x.T_total // B
    ptr = lambda t: 0 if t is None else t.data_ptr()  # noqa: E731
    st = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
            ptr(d["beta"]), ptr(d["h0"]) if use_h0 else 0, o.data_ptr(),
            ptr(ht), x.N, T, x.H_k, x.H_v, x.d_k, x.d_v, 64, x.scale, ptr(d["cu_seqlens"]), stream)
    return st


@pytest.mark.parametrize("variant", ["beta_h0_ht", "decay_only", "no_h0_no_ht"])
def test_noalloc_matches_kda_chunk_fwd_on_two_calls(variant):
    import torch

    from chunkwise_gated_linear_gb300 import kda

    stream = torch.cuda.current_stream().cuda_stream
    beta = variant != "decay_only"
    cases = [make_inputs((700, 1, 300, 1029), 2, 4, 128, 128, seed=130, h0=True, varlen=True, beta=beta),
             make_inputs((1500, 1500), 1, 2, 128, 128, seed=131, h0=True, beta=beta)]
    for x in cases:
        d = to_device(x)
        outs = []
        for fn in (kda.kda_chunk_fwd, kda.kda_chunk_fwd_noalloc):
            o = torch.full(d["v"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            ht = None
            if variant != "no_h0_no_ht":
                ht = torch.full((x.N, x.H_v, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
            assert _call(fn, d, x, o, ht, stream, use_h0=variant != "no_h0_no_ht") == kda.KDA_OK
            torch.cuda.synchronize()
            outs.append((o, ht))
        assert kda.kda_get_device_error(stream) == 0
        # the same kernel on the same inputs: bitwise equal
        assert torch.equal(outs[0][0], outs[1][0])
        assert not torch.isnan(outs[1][0].float()).any()
        if outs[0][1] is not None:
            assert torch.equal(outs[0][1], outs[1][1])


_PROBE = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from chunkwise_gated_linear_gb300 import kda
from inputs import make_inputs
from kda_cases import to_device
x = make_inputs((1500, 1500), 1, 2, 128, 128, seed=131, h0=True)
d = to_device(x)
o = torch.empty(d["v"].shape, dtype=torch.bfloat16, device="cuda")
ht = torch.empty((x.N, x.H_v, 128, 128), dtype=torch.float32, device="cuda")
s = torch.cuda.current_stream().cuda_stream
def call(fn):
    st = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(), d["beta"].data_ptr(),
            d["h0"].data_ptr(), o.data_ptr(), ht.data_ptr(), x.N, 1500, 1, 2, 128, 128, 64, x.scale, 0, s)
    assert st == 0, st
    torch.cuda.synchronize()
# the first call loads the kernel's code and its fixed array (part of the library's
# footprint, loaded once); the measurement starts after it
call(kda.kda_chunk_fwd_noalloc)
free0 = torch.cuda.mem_get_info()[0]
fn = kda.kda_chunk_fwd_noalloc if sys.argv[2] == "noalloc" else kda.kda_chunk_fwd
call(fn)
call(fn)
print("USED", free0 - torch.cuda.mem_get_info()[0])
"""


def _used(mode):
    r = subprocess.run([sys.executable, "-c", _PROBE, ROOT, mode], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return int([ln for ln in r.stdout.split("\n") if ln.startswith("USED")][0].split()[1])


def test_noalloc_allocates_nothing():
    """In a fresh process, after a first call has loaded the kernel and its fixed array, two
    more calls of kda_chunk_fwd_noalloc leave the device's free memory exactly as it was; the
    same measurement does see the pool scratch of kda_chunk_fwd (so it would catch a call
    that allocated)."""
    assert _used("noalloc") == 0
    assert _used("pool") > 0
