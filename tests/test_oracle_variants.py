"""Pins of the oracle's scale-rule (floor / RCEIL) and fp32-input variants -- CPU only."""
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN
from test_oracle_quant import _parse_blocks  # noqa: F401  (same fixture format)


def _parse(path):
    blocks, cur = [], None
    for ln in open(path):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        key, _, rest = ln.partition(" ")
        if key == "block":
            cur = dict(name=rest.strip(), inp={}, out={}, sf=None)
            blocks.append(cur)
        elif key in ("in", "out"):
            d = cur["inp" if key == "in" else "out"]
            for tok in rest.split():
                pos, val = tok.split(":")
                for i in (range(32) if pos == "*" else [int(pos)]):
                    d[i] = int(val, 16)
        elif key == "sf":
            cur["sf"] = int(rest, 16)
    return blocks


@pytest.mark.parametrize("blk", _parse(os.path.join(GOLDEN, "mx_blocks_rceil.txt")), ids=lambda b: b["name"])
def test_golden_rceil_blocks(blk):
    bits = np.zeros(32, np.uint16)
    for i, v in blk["inp"].items():
        bits[i] = v
    want = np.zeros(32, np.uint8)
    for i, v in blk["out"].items():
        want[i] = v
    sf, q = oracle.mx_block_rule(oracle.bf16_to_double(bits), oracle.RULE_RCEIL)
    assert sf == blk["sf"] and np.array_equal(q, want)
    q2, sf2 = oracle.quantize_rowwise_ex(bits.reshape(1, 32), oracle.RULE_RCEIL)
    assert sf2[0, 0] == blk["sf"] and np.array_equal(q2[0], want)


def test_rceil_never_saturates_and_relates_to_floor():
    rng = np.random.default_rng(0)
    for _ in range(500):
        x = (rng.standard_normal(32) * 2.0 ** rng.integers(-40, 40)).astype(np.float32).astype(np.float64)
        amax = np.max(np.abs(x))
        sr, qr = oracle.mx_block_rule(x, oracle.RULE_RCEIL)
        sf, _ = oracle.mx_block_rule(x, oracle.RULE_FLOOR)
        X = 2.0 ** (sr - 127)
        assert 224 * X < amax <= 448 * X
        m = amax / 2.0 ** np.floor(np.log2(amax))          # mantissa in [1, 2), exact for binary floats
        assert sr == sf + (1 if m > 1.75 else 0)
        # no saturation: every element is within half an E4M3 step of x / X
        deq = oracle.e4m3_decode(qr) * X
        e = np.floor(np.log2(np.maximum(np.abs(x) / X, 2.0 ** -6)))
        assert np.all(np.abs(deq - x) <= 2.0 ** (e - 4) * X * (1 + 1e-12))


def test_fp32_input_matches_bf16_path_on_bf16_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 96)) * np.exp(rng.standard_normal((64, 1)) * 3)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)          # the same values as fp32
    for rule in (oracle.RULE_FLOOR, oracle.RULE_RCEIL):
        assert all(np.array_equal(a, b) for a, b in zip(oracle.quantize_rowwise_ex(xb, rule),
                                                        oracle.quantize_rowwise_ex(xf, rule)))
        off = np.array([0, 64], np.int32)
        assert all(np.array_equal(a, b) for a, b in zip(oracle.quantize_colwise_seg_ex(xb, off, [0, 128], 128, rule),
                                                        oracle.quantize_colwise_seg_ex(xf, off, [0, 128], 128, rule)))
    # the floor-rule bf16 path through the _ex entry equals the original entry
    assert all(np.array_equal(a, b) for a, b in zip(oracle.quantize_rowwise_ex(xb), oracle.quantize_rowwise(xb)))


def test_fp32_hand_worked():
    # 1 + 2^-10 is not a bf16 value: amax -> s = -8; (1 + 2^-10) * 256 = 256.25 rounds to 256 -> 0x78
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1.0 + 2.0 ** -10
    x[0, 1] = 3.0 * 2.0 ** -9          # * 256 = 1.5 -> 1.5 exactly (0_0111_100 = 0x3C)
    q, sf = oracle.quantize_rowwise_ex(x)
    assert sf[0, 0] == 0x77 and q[0, 0] == 0x78 and q[0, 1] == 0x3C and np.all(q[0, 2:] == 0)
