"""Pins of the oracle's combine (unpermute / weighted merge) forward and backward -- CPU only."""
import numpy as np
import pytest

import oracle


def _bits(v):
    f = np.asarray(v, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def _val(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(T, k, E_rows_per, H, seed, integer=True):
    rng = np.random.default_rng(seed)
    R = T * k
    perm = rng.permutation(R).astype(np.int32)
    dst_of = perm.reshape(T, k)
    if integer:
        Y = rng.integers(-8, 9, size=(R, H)).astype(np.float32)
        gate = rng.integers(-4, 5, size=(T, k)).astype(np.float32)
        dOut = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    else:
        Y = rng.standard_normal((R, H)).astype(np.float32)
        gate = rng.random((T, k)).astype(np.float32)
        dOut = rng.standard_normal((T, H)).astype(np.float32)
    Yb = (Y.view(np.uint32) >> 16).astype(np.uint16)
    dOb = (dOut.view(np.uint32) >> 16).astype(np.uint16)
    return Yb, gate, dst_of, dOb


def test_top1_unit_gate_is_inverse_permutation():
    Yb, _, dst_of, _ = _case(50, 1, 1, 64, 0, integer=False)
    out = oracle.combine_fwd(Yb, np.ones((50, 1), np.float32), dst_of)
    assert np.array_equal(out, Yb[dst_of[:, 0]])


def test_power_of_two_gate_scaling_is_exact():
    Yb, gate, dst_of, _ = _case(20, 4, 1, 32, 1, integer=False)
    a = oracle.combine_fwd(Yb, gate, dst_of)
    b = oracle.combine_fwd(Yb, gate * 4.0, dst_of)
    assert np.array_equal(_val(b), 4.0 * _val(a))


def test_adjoint_identity_exact():
    # integer data: every sum is exact, so <combine(Y), dOut> == <Y, combine_bwd_dY(dOut)>
    Yb, gate, dst_of, dOb = _case(16, 3, 1, 40, 2)
    out = _val(oracle.combine_fwd(Yb, gate, dst_of))
    dY, _ = oracle.combine_bwd(dOb, Yb, gate, dst_of)
    lhs = np.sum(out * _val(dOb))
    rhs = np.sum(_val(Yb) * _val(dY))
    assert lhs == rhs


def test_dgate_is_derivative_of_forward():
    # combine is linear in the gates: the change of <out[t], dOut[t]> when gate[t][j] grows by 1
    Yb, gate, dst_of, dOb = _case(6, 4, 1, 24, 3)
    _, dgate = oracle.combine_bwd(dOb, Yb, gate, dst_of)
    base = _val(oracle.combine_fwd(Yb, gate, dst_of))
    for t in range(6):
        for j in range(4):
            g2 = gate.copy()
            g2[t, j] += 1.0
            moved = _val(oracle.combine_fwd(Yb, g2, dst_of))
            assert np.sum((moved[t] - base[t]) * _val(dOb[t])) == dgate[t, j]


def test_dropped_slots():
    Yb, gate, dst_of, dOb = _case(5, 2, 1, 16, 4)
    dst_of = dst_of.copy()
    dst_of[2, 1] = -1
    out = oracle.combine_fwd(Yb, gate, dst_of)
    want = np.float64(gate[2, 0]) * _val(Yb[dst_of[2, 0]])        # exact small integers
    assert np.array_equal(_val(out[2]), want)
    dY, dgate = oracle.combine_bwd(dOb, Yb, gate, dst_of)
    assert dgate[2, 1] == 0.0
