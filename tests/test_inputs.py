"""The seeded input generator: determinism, shapes, value ranges, dtype exactness."""

from __future__ import annotations

import numpy as np

from inputs import WORKLOADS, make_inputs
from inputs.synth import round_to_dtype


def test_deterministic_for_a_seed():
    a = make_inputs((40, 7), 2, 4, 16, 8, seed=5, h0=True)
    b = make_inputs((40, 7), 2, 4, 16, 8, seed=5, h0=True)
    for f in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    c = make_inputs((40, 7), 2, 4, 16, 8, seed=6, h0=True)
    assert not np.array_equal(a.q, c.q)


def test_shapes_ranges_and_normalisation():
    x = make_inputs((100,), 2, 4, 16, 8, seed=1, a_lo=0.8, dtype="f32")
    assert x.q.shape == (100, 2, 16) and x.v.shape == (100, 4, 8) and x.g.shape == (100, 4, 16)
    assert x.beta.shape == (100, 4) and x.h0 is None and not x.varlen
    a = np.exp(x.g.astype(np.float64))
    assert a.min() >= 0.8 - 1e-6 and a.max() <= 0.999 + 1e-6
    assert (x.beta > 0).all() and (x.beta < 1).all()
    np.testing.assert_allclose(np.linalg.norm(x.q, axis=-1), 1.0, rtol=1e-5)
    np.testing.assert_allclose(np.linalg.norm(x.k, axis=-1), 1.0, rtol=1e-5)
    assert abs(x.scale - 16 ** -0.5) < 1e-12
    s = make_inputs((100,), 2, 4, 16, 8, seed=1, gate="head")
    assert s.g.shape == (100, 4)


def test_bf16_rounding_is_nearest_even_and_exact():
    vals = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 1e-30, 0.0], np.float32)
    r = round_to_dtype(vals, "bf16")
    assert (r.view(np.uint32) & 0xFFFF).max() == 0  # representable in bf16
    assert r[1] == 1.0  # tie 1 + 2^-8 rounds to even (1.0)
    assert r[2] == np.float32(1.0078125)  # above the tie rounds up
    x = make_inputs((10,), 1, 1, 8, 8, seed=2)
    for t in (x.q, x.k, x.v):
        assert (t.view(np.uint32) & 0xFFFF).max() == 0


def test_varlen_lengths_are_drawn_in_range():
    w = WORKLOADS["kda_varlen16_t512to16384_h32_d128_bf16"]
    rng = np.random.default_rng(5)
    lens = rng.integers(w.len_range[0], w.len_range[1] + 1, size=w.n_seqs)
    assert lens.min() >= 512 and lens.max() <= 16384
    x = make_inputs((), 1, 1, 8, 8, seed=5, len_range=(3, 9), n_seqs=4)
    assert x.varlen and x.N == 4 and (np.diff(x.cu_seqlens) >= 3).all()
