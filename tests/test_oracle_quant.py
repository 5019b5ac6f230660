"""Pins of the oracle's MX quantization (block rule, rowwise, columnwise, scale layout) -- CPU only."""
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _parse_blocks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "mx_blocks.txt")) as f:
        for ln in f:
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
                    if pos == "*":
                        for i in range(32):
                            d[i] = int(val, 16)
                    else:
                        d[int(pos)] = int(val, 16)
            elif key == "sf":
                cur["sf"] = int(rest, 16)
    return blocks


@pytest.mark.parametrize("blk", _parse_blocks(), ids=lambda b: b["name"])
def test_golden_blocks(blk):
    bits = np.zeros(32, np.uint16)
    for i, v in blk["inp"].items():
        bits[i] = v
    want_q = np.zeros(32, np.uint8)
    for i, v in blk["out"].items():
        want_q[i] = v
    # through the block rule
    sf, q = oracle.mx_block(oracle.bf16_to_double(bits))
    assert sf == blk["sf"]
    assert np.array_equal(q, want_q), (q, want_q)
    # through the rowwise quantizer, as one row of a [1 x 32] tensor
    q2, sf2 = oracle.quantize_rowwise(bits.reshape(1, 32))
    assert sf2[0, 0] == blk["sf"] and np.array_equal(q2[0], want_q)


def _bf16(vals):
    f = np.asarray(vals, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def test_powers_of_two_roundtrip():
    rng = np.random.default_rng(0)
    for _ in range(200):
        top = int(rng.integers(-120, 120))
        # exponents within 2^17 of the amax: top-8 .. top-17 land in [2^-9, 2^8] after scaling
        ex = top - rng.integers(0, 18, size=32)
        ex[0] = top
        sign = rng.choice([-1.0, 1.0], size=32)
        vals = sign * np.ldexp(1.0, ex)
        sf, q = oracle.mx_block(vals)
        assert sf == top - 8 + 127
        deq = oracle.e4m3_decode(q) * 2.0 ** (sf - 127)
        assert np.array_equal(deq, vals)


def test_three_bit_mantissas_roundtrip():
    rng = np.random.default_rng(1)
    for _ in range(200):
        top = int(rng.integers(-100, 100))
        m = rng.integers(8, 16, size=32)            # 1.mmm with 3 fraction bits
        ex = top - rng.integers(0, 15, size=32)      # stays in the normal window of E4M3
        m[0], ex[0] = 8, top
        m[ex == top] = np.minimum(m[ex == top], 14)   # 1.875 * 2^8 = 480 would saturate
        vals = m / 8.0 * np.ldexp(1.0, ex)
        sf, q = oracle.mx_block(vals)
        deq = oracle.e4m3_decode(q) * 2.0 ** (sf - 127)
        amax_e = int(np.floor(np.log2(np.max(np.abs(vals)))))
        assert sf == amax_e - 8 + 127
        assert np.array_equal(deq, vals)


@pytest.mark.parametrize("c", [1.0, -3.0, 0.15625, 300.0, 2.0 ** -100, 1.5 * 2.0 ** -14, -1.9921875])
def test_constant_block(c):
    cb = float(np.float32(c))
    bits = _bf16([cb] * 32) if np.float32(cb).view(np.uint32) & 0xFFFF == 0 else None
    if bits is None:
        pytest.skip("not a bf16 value")
    sf, q = oracle.mx_block(oracle.bf16_to_double(bits))
    e = int(np.floor(np.log2(abs(cb))))
    assert sf == e + 119
    expect = oracle.e4m3_encode([cb * 2.0 ** (8 - e)])[0]
    assert np.all(q == expect)


def test_block_invariants_random():
    rng = np.random.default_rng(2)
    for trial in range(300):
        scale = 2.0 ** rng.integers(-60, 60)
        x = (rng.standard_normal(32) * scale).astype(np.float32)
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)      # truncate to bf16
        xv = oracle.bf16_to_double(bits)
        sf, q = oracle.mx_block(xv)
        X = 2.0 ** (sf - 127)
        deq = oracle.e4m3_decode(q) * X
        assert np.all(np.abs(deq) <= 448 * X)
        i = int(np.argmax(np.abs(xv)))
        assert 256 * X <= abs(deq[i]) <= 448 * X
        # monotone within a block
        order = np.argsort(xv, kind="stable")
        assert np.all(np.diff(deq[order]) >= 0)
        # one rounding: |x - deq| <= half an E4M3 step at x's binade, or saturation
        err = np.abs(xv - deq)
        e = np.floor(np.log2(np.maximum(np.abs(xv) / X, 2.0 ** -6)))
        half_ulp = 2.0 ** (e - 4) * X
        assert np.all((err <= half_ulp * (1 + 1e-12)) | (np.abs(xv) > 448 * X))


def test_colwise_is_rowwise_of_transpose():
    rng = np.random.default_rng(3)
    rows, cols = 256, 96
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.standard_normal((rows, 1)))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    qc, sfc = oracle.quantize_colwise_seg(bits, [0, rows], [0, rows], rows)
    qr, sfr = oracle.quantize_rowwise(np.ascontiguousarray(bits.T))
    assert np.array_equal(qc, qr) and np.array_equal(sfc, sfr)


def test_colwise_segments_match_per_segment_transpose():
    rng = np.random.default_rng(4)
    counts = [0, 5, 128, 131, 0, 40]
    cols = 64
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    poff = np.concatenate([[0], np.cumsum([(c + 127) // 128 * 128 for c in counts])]).astype(np.int32)
    R = int(off[-1])
    x = rng.standard_normal((R, cols)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    ld = int(poff[-1]) + 128
    qc, sfc = oracle.quantize_colwise_seg(bits, off, poff, ld)
    for g, te in enumerate(counts):
        pad = (te + 127) // 128 * 128
        seg = np.zeros((pad, cols), np.uint16)
        seg[:te] = bits[off[g]:off[g] + te]
        if pad == 0:
            continue
        qr, sfr = oracle.quantize_rowwise(np.ascontiguousarray(seg.T))
        assert np.array_equal(qc[:, poff[g]:poff[g] + pad], qr)
        assert np.array_equal(sfc[:, poff[g] // 32:(poff[g] + pad) // 32], sfr)
        # zero padding: codes 0, and fully padded blocks take scale 0x00
        assert np.all(qc[:, poff[g] + te:poff[g] + pad] == 0)
        nb_real = (te + 31) // 32
        assert np.all(sfc[:, poff[g] // 32 + nb_real:(poff[g] + pad) // 32] == 0)


def test_place_sf_rows():
    sf = np.arange(10 * 3, dtype=np.uint8).reshape(10, 3) + 1
    off = [0, 3, 3, 10]
    poff = [0, 128, 128, 256]
    out = oracle.place_sf_rows(sf, off, poff)
    assert out.shape == (256, 3)
    assert np.array_equal(out[0:3], sf[0:3]) and np.all(out[3:128] == 0)
    assert np.array_equal(out[128:135], sf[3:10]) and np.all(out[135:] == 0)


def test_golden_sf_layout():
    rows, kb = 256, 8
    sf = np.zeros((rows, kb), np.uint8)
    with open(os.path.join(GOLDEN, "sf_layout.txt")) as f:
        pts = [tuple(int(t) for t in ln.split()) for ln in f if ln.strip() and not ln.startswith("#")]
    for i, (r, c, _) in enumerate(pts):
        sf[r, c] = i + 1
    sw = oracle.sf_to_tcgen05(sf)
    for i, (r, c, o) in enumerate(pts):
        assert sw[o] == i + 1, (r, c, o)


@pytest.mark.parametrize("rows,kb", [(1, 1), (128, 4), (130, 7), (300, 224), (5, 2)])
def test_sf_layout_bijective_and_padded(rows, kb):
    rng = np.random.default_rng(rows * 1000 + kb)
    sf = rng.integers(1, 255, size=(rows, kb), dtype=np.uint8)
    sw = oracle.sf_to_tcgen05(sf)
    assert sw.size == ((rows + 127) // 128 * 128) * ((kb + 3) // 4 * 4)
    assert np.array_equal(oracle.sf_from_tcgen05(sw, rows, kb), sf)
    assert np.count_nonzero(sw) == rows * kb          # padding is zero, nothing overwritten
