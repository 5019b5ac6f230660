"""Pins of the oracle's fp64 GEMM over dequantized MX operands -- CPU only."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _exact(qa, sfa, qb, sfb):
    """Exact rational C = deq(A) deq(B)^T from the E4M3 / E8M0 definitions (no floating point)."""
    def e4m3(c):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))
        return -v if s else v

    def deq(q, sf):
        return [[e4m3(int(q[r, k])) * Fraction(2) ** (int(sf[r, k // 32]) - 127) for k in range(q.shape[1])]
                for r in range(q.shape[0])]
    A, B = deq(qa, sfa), deq(qb, sfb)
    return [[sum(a * b for a, b in zip(A[m], B[n])) for n in range(len(B))] for m in range(len(A))], A, B


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38   # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 32, 0), (3, 5, 64, 1), (8, 8, 128, 2), (2, 7, 96, 3)])
def test_gemm_against_exact_rationals(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa, qb = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    sfa = rng.integers(117, 138, size=(M, K // 32), dtype=np.uint8)
    sfb = rng.integers(117, 138, size=(N, K // 32), dtype=np.uint8)
    got = oracle.gemm_nt(qa, sfa, qb, sfb)
    exact, A, B = _exact(qa, sfa, qb, sfb)
    for m in range(M):
        for n in range(N):
            bound = sum(abs(a * b) for a, b in zip(A[m], B[n])) * Fraction(K) * Fraction(2) ** -52
            assert abs(Fraction(got[m, n]) - exact[m][n]) <= bound, (m, n)


def test_gemm_exact_when_representable():
    # codes restricted to small integers, scales to 2^0: every partial sum is an
    # exact small integer, so fp64 must reproduce the exact sum bit for bit.
    rng = np.random.default_rng(5)
    M, N, K = 6, 4, 128
    ints = np.array([0x00, 0x38, 0x40, 0x44, 0x48, 0xB8, 0xC0, 0xC4, 0xC8], np.uint8)   # 0, +-1, +-2, +-3, +-4
    qa = rng.choice(ints, size=(M, K)).astype(np.uint8)
    qb = rng.choice(ints, size=(N, K)).astype(np.uint8)
    sfa = np.full((M, K // 32), 127, np.uint8)
    sfb = np.full((N, K // 32), 127, np.uint8)
    got = oracle.gemm_nt(qa, sfa, qb, sfb)
    exact, _, _ = _exact(qa, sfa, qb, sfb)
    assert all(Fraction(got[m, n]) == exact[m][n] for m in range(M) for n in range(N))


def test_gemm_identity_b_returns_dequantized_a():
    rng = np.random.default_rng(6)
    M, K = 5, 64
    qa = _rand_codes(rng, (M, K))
    sfa = rng.integers(100, 150, size=(M, K // 32), dtype=np.uint8)
    qb = np.zeros((K, K), np.uint8)
    np.fill_diagonal(qb, 0x38)                         # 1.0
    sfb = np.full((K, K // 32), 127, np.uint8)         # scale 2^0
    got = oracle.gemm_nt(qa, sfa, qb, sfb)
    want = oracle.e4m3_decode(qa.reshape(-1)).reshape(M, K) * np.exp2(np.repeat(sfa.astype(np.float64) - 127, 32, axis=1))
    assert np.array_equal(got, want)


def test_gemm_transposition_and_scale_linearity():
    rng = np.random.default_rng(7)
    M, N, K = 4, 6, 64
    qa, qb = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    sfa = rng.integers(120, 135, size=(M, K // 32), dtype=np.uint8)
    sfb = rng.integers(120, 135, size=(N, K // 32), dtype=np.uint8)
    c = oracle.gemm_nt(qa, sfa, qb, sfb)
    ct = oracle.gemm_nt(qb, sfb, qa, sfa)
    assert np.allclose(c, ct.T, rtol=1e-13, atol=0)
    # raising every scale of A's row 0 by one doubles that output row exactly
    sfa2 = sfa.copy()
    sfa2[0] += 1
    c2 = oracle.gemm_nt(qa, sfa2, qb, sfb)
    assert np.array_equal(c2[0], 2 * c[0]) and np.array_equal(c2[1:], c[1:])


def test_bf16_rounding():
    assert list(oracle.to_bf16_bits([1.0, -2.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 0.0])) == [0x3F80, 0xC000, 0x3F80, 0x3F82, 0x0000]
