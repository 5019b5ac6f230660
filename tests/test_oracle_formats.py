"""Pins of the oracle's element formats (E4M3, E8M0, bf16) -- CPU only."""
import math
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def test_encoders_agree_exhaustively():
    # every finite bf16 value times 2^s: the definitional RNE encoder must equal the
    # brute-force nearest-code search; s spans the shifts the MX rule can apply
    # (bf16 exponents -133..127, element window up to 2^9) plus margin.
    bad, bits, shift = oracle.check_encoders(-20, 20)
    assert bad == 0, f"encoder mismatch, first at bf16 0x{bits:04x} * 2^{shift}"


@pytest.mark.parametrize("lo,hi", [(-140, -100), (100, 140)])
def test_encoders_agree_far_shifts(lo, hi):
    bad, bits, shift = oracle.check_encoders(lo, hi)
    assert bad == 0, f"encoder mismatch, first at bf16 0x{bits:04x} * 2^{shift}"


def test_decode_encode_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254                      # only S.1111.111 is NaN
    assert set(codes[~finite]) == {0x7F, 0xFF}
    re = oracle.e4m3_encode(vals[finite])
    assert np.array_equal(re, codes[finite])        # -0 keeps its sign: 0x80
    assert vals[finite].max() == 448.0 and vals[finite].min() == -448.0


def test_decode_is_monotone_on_positive_codes():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)


def test_golden_e4m3_values():
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for code_hex, val in rows:
        code = int(code_hex, 16)
        v = float(val)
        dec = oracle.e4m3_decode([code])[0]
        assert dec == v and math.copysign(1, dec) == math.copysign(1, v), code_hex
        assert oracle.e4m3_encode([v])[0] == code, code_hex


def test_saturation_and_nan():
    enc = oracle.e4m3_encode([449.0, 463.99, 464.0, 1e30, -1e30, math.inf, -math.inf, math.nan])
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]


def test_e8m0_decode():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_decode(255))


def test_bf16_decode_matches_numpy():
    bits = np.arange(0, 0x10000, 97, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns widen with a warning
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_to_double(bits)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all((ref == got) | both_nan)
