"""Pins of the oracle's SwiGLU forward/backward -- CPU only."""
import math

import numpy as np

import oracle


def _bits(a):
    a = np.asarray(a, np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _val(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 2.0], np.float32)
    u = np.array([3.0, 1.0, 1.0, 1.0, 1.0, 0.5], np.float32)
    h = oracle.swiglu_fwd(np.concatenate([_bits(g), _bits(u)]).reshape(1, -1))[0]
    assert h[0] == 0.0                                            # silu(0) = 0
    assert h[1] == np.float32(1.0 / (1.0 + math.exp(-1.0)))       # silu(1) = sigmoid(1)
    assert h[2] == np.float32(-1.0 / (1.0 + math.e))              # silu(-1)
    assert abs(h[3] - 20.0) < 1e-6 and abs(h[4]) < 1e-7           # saturating ends
    assert h[5] == np.float32(2.0 / (1.0 + math.exp(-2.0)) * 0.5)


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(0)
    R, I = 4, 16
    a = _bits(rng.standard_normal((R, 2 * I)))
    dh = _bits(rng.standard_normal((R, I)))
    dH = oracle.swiglu_bwd(dh, a).astype(np.float64)
    g, u, d = _val(a[:, :I]), _val(a[:, I:]), _val(dh)
    silu = lambda z: z / (1.0 + np.exp(-z))
    eps = 1e-6
    num_dg = d * u * (silu(g + eps) - silu(g - eps)) / (2 * eps)
    assert np.allclose(dH[:, :I], num_dg, rtol=1e-5, atol=1e-6)
    # the up-gradient is the forward with the output gradient in place of up
    fwd_with_d = oracle.swiglu_fwd(np.concatenate([a[:, :I], dh], axis=1)).astype(np.float64)
    assert np.array_equal(dH[:, I:], fwd_with_d)
