"""The near-tie checker used by the fused-SwiGLU parity tests, on the CPU: differences that
an fp32 perturbation within the stated bound can cause pass; a code or a scale byte that no
such perturbation explains fails.  The "kernel" here is the oracle applied to perturbed
values, so every planted mistake lives on the CPU side."""
import numpy as np
import pytest

import oracle
from near_tie import check_blocks, swiglu_bounds


def _quant(v):
    q, sf = oracle.quantize_rowwise_ex(np.asarray(v, np.float32))
    return q, sf


def _values(rng, rows=64, n=256):
    v = rng.standard_normal((rows, n)) * np.exp2(rng.integers(-6, 6, (rows, 1)))
    return v.astype(np.float32).astype(np.float64)


def test_perturbation_within_the_bound_is_explained():
    rng = np.random.default_rng(1)
    v = _values(rng)
    rel = 2.0 ** -12                                        # a deliberately coarse bound
    w = (v * (1 + rel * rng.uniform(-1, 1, v.shape))).astype(np.float32)
    q, sf = _quant(w)
    n_codes, n_scales = check_blocks(v, rel * np.abs(v) * 1.01, q, sf)
    assert n_codes > 0                                      # the perturbation did move some codes


def test_scale_flip_at_a_power_of_two_is_explained():
    v = np.full((1, 32), 0.5)
    v[0, 7] = 2.0 ** 3 * (1 - 2.0 ** -20)                  # block maximum just below 8
    w = v.copy()
    w[0, 7] = 8.0                                           # the "kernel" rounds it up: scale one higher
    q, sf = _quant(w)
    check_blocks(v, 2.0 ** -18 * np.abs(v), q, sf)
    with pytest.raises(AssertionError):
        check_blocks(v, 2.0 ** -24 * np.abs(v), q, sf)       # too far for this bound


def test_misrounded_code_fails():
    rng = np.random.default_rng(2)
    v = _values(rng)
    q, sf = _quant(v)
    q = q.copy()
    r, c = 5, 77
    assert q[r, c] & 0x7F not in (0, 0x7E)
    q[r, c] += 1                                             # one step up, far from any tie
    y = oracle.e4m3_decode(q[r:r + 1, c])
    with pytest.raises(AssertionError):
        check_blocks(v, 2.0 ** -20 * np.abs(v), q, sf)
    assert np.isfinite(y).all()


def test_wrong_scale_fails():
    rng = np.random.default_rng(3)
    v = _values(rng)
    q, sf = _quant(v)
    sf = sf.copy()
    sf[3, 2] += 1
    with pytest.raises(AssertionError):
        check_blocks(v, 2.0 ** -20 * np.abs(v), q, sf)


def test_swapped_columns_fail():
    # a staging-tile indexing mistake: two columns of the kernel's output exchanged
    rng = np.random.default_rng(4)
    v = _values(rng)
    q, sf = _quant(v)
    q = q.copy()
    q[:, [10, 11]] = q[:, [11, 10]]
    with pytest.raises(AssertionError):
        check_blocks(v, 2.0 ** -20 * np.abs(v), q, sf)


def test_swiglu_bounds_cover_fp32_evaluation():
    # the bounds hold for a plain fp32 evaluation of the same expressions (libm exp, IEEE
    # division): a weaker check than the kernel's own arithmetic, but a check of the formulas
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(20000) * 4).astype(np.float32)
    u = rng.standard_normal(20000).astype(np.float32)
    d = (rng.standard_normal(20000) * 1e-2).astype(np.float32)
    s32 = (np.float32(1) / (np.float32(1) + np.exp(-g))).astype(np.float32)
    h32 = g * s32 * u
    du32 = d * (g * s32)
    dg32 = d * u * (s32 * (np.float32(1) + g * (np.float32(1) - s32)))
    G, U, D = g.astype(np.float64), u.astype(np.float64), d.astype(np.float64)
    s = 1 / (1 + np.exp(-G))
    assert np.all(np.abs(h32 - G * s * U) <= swiglu_bounds(G, U))
    b_dg, b_du = swiglu_bounds(G, U, D)
    assert np.all(np.abs(du32 - D * G * s) <= b_du)
    assert np.all(np.abs(dg32 - D * U * s * (1 + G * (1 - s))) <= b_dg)
