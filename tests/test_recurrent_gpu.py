"""GPU parity of the recurrent (token-by-token) entry point against the fp64 oracle, and
prefill -> decode continuity: the chunkwise pass over a prefix, then the recurrent step
over the next tokens from its final state (updated in place), equals one pass over the
whole sequence."""

from __future__ import annotations

import numpy as np
import pytest

from conftest import rel_l2
from inputs import make_inputs
from kda_cases import TOL, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["bf16_d128_varlen_gqa", "bf16_d64", "f32_d128", "head_gate",
                                  "decay_only", "dk64_dv128"])
def test_recurrent_matches_oracle(case):
    if case == "bf16_d128_varlen_gqa":
        x = make_inputs((1, 17, 64, 130), 2, 4, 128, 128, seed=150, h0=True, varlen=True)
    elif case == "bf16_d64":
        x = make_inputs((90,), 2, 2, 64, 64, seed=151, h0=True)
    elif case == "f32_d128":
        x = make_inputs((70, 70), 1, 2, 128, 128, seed=152, dtype="f32", h0=True)
    elif case == "head_gate":
        x = make_inputs((100,), 2, 2, 128, 128, seed=153, gate="head", h0=True)
    elif case == "decay_only":
        x = make_inputs((100,), 1, 2, 128, 128, seed=154, h0=True, beta=False)
    else:
        x = make_inputs((80,), 1, 1, 64, 128, seed=155, h0=True)
    o, ht = run_gpu(x, recurrent=True)
    o_r, ht_r = run_oracle(x)
    e_o, e_h = rel_l2(o, o_r), rel_l2(ht, ht_r)
    print(f"recurrent {case}: rel_l2 o={e_o:.3e} ht={e_h:.3e}")
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    assert e_o <= TOL[x.dtype] and e_h <= TOL[x.dtype]


def test_prefill_then_decode_in_place():
    import torch

    from chunkwise_gated_linear_gb300 import chunk_kda_fwd

    T1, T2 = 320, 6
    x = make_inputs((T1 + T2,), 2, 4, 128, 128, seed=156, h0=True)
    d = to_device(x)
    cut = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
    # prefill: the chunkwise pass over the first T1 tokens
    o1, state = chunk_kda_fwd(cut(d["q"], 0, T1), cut(d["k"], 0, T1), cut(d["v"], 0, T1),
                              cut(d["g"], 0, T1), cut(d["beta"], 0, T1), h0=d["h0"], scale=x.scale)
    # decode: one token at a time, the state updated in place (ht is h0)
    outs = []
    for t in range(T1, T1 + T2):
        ot, _ = chunk_kda_fwd(cut(d["q"], t, t + 1), cut(d["k"], t, t + 1), cut(d["v"], t, t + 1),
                              cut(d["g"], t, t + 1), cut(d["beta"], t, t + 1), h0=state, ht=state,
                              scale=x.scale, recurrent=True)
        outs.append(ot)
    torch.cuda.synchronize()
    o_r, ht_r = run_oracle(x)
    o_r = o_r.reshape(x.N, T1 + T2, x.H_v, x.d_v)
    got = torch.cat([o1] + outs, dim=1).float().cpu().numpy()
    e_pre = rel_l2(got[:, :T1], o_r[:, :T1])
    e_dec = rel_l2(got[:, T1:], o_r[:, T1:])
    e_h = rel_l2(state.cpu().numpy().astype(np.float64), ht_r)
    print(f"prefill o={e_pre:.3e}, decoded o={e_dec:.3e}, final state={e_h:.3e}")
    assert e_pre <= TOL["bf16"] and e_dec <= TOL["bf16"] and e_h <= TOL["bf16"]
