"""GPU quantizer vs the CPU oracle: bit-exact codes and scale bytes (layout included)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import bits, check_dev_err, dev, from_bits, np_, offsets  # noqa: F401

pytestmark = pytest.mark.gpu


def _randbits(shape, seed, spread=4.0):
    g = synth.generator(seed)
    x = torch.randn(*shape, generator=g) * torch.exp(spread * torch.randn(shape[0], 1, generator=g))
    return bits(x.to(torch.bfloat16))


def _check_row(xb, out):
    rows, cols = xb.shape
    oq, osf = oracle.quantize_rowwise(xb)
    assert np.array_equal(np_(out["q_row"]), oq), "rowwise codes differ"
    want = oracle.sf_to_tcgen05(osf)
    got = np_(out["sf_row"])
    assert np.array_equal(got[: want.size], want), "rowwise scales differ"


def _check_col(xb, out, off=None, poff=None):
    rows, cols = xb.shape
    if off is None:
        off, poff = np.array([0, rows], np.int32), np.array([0, (rows + 127) // 128 * 128], np.int32)
    ld = out["ld_col"]
    P = int(poff[-1])
    oq, osf = oracle.quantize_colwise_seg(xb, off, poff, ld)
    assert np.array_equal(np_(out["q_col"])[:, :P], oq[:, :P]), "columnwise codes differ"
    got_sf = oracle.sf_from_tcgen05(np_(out["sf_col"]), cols, ld // 32)
    assert np.array_equal(got_sf[:, : P // 32], osf[:, : P // 32]), "columnwise scales differ"


@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 96), (512, 256), (300, 7168), (129, 4096), (77, 160)])
def test_rowwise(dev, rows, cols):
    xb = _randbits((rows, cols), rows * 7 + cols)
    out = mx.quantize_alloc(from_bits(xb, dev), mx.MX_ROWWISE)
    torch.cuda.synchronize()
    _check_row(xb, out)


@pytest.mark.parametrize("rows,cols", [(32, 32), (256, 96), (130, 160), (1000, 256)])
def test_colwise(dev, rows, cols):
    xb = _randbits((rows, cols), rows * 11 + cols)
    out = mx.quantize_alloc(from_bits(xb, dev), mx.MX_COLWISE)
    torch.cuda.synchronize()
    _check_col(xb, out)


@pytest.mark.parametrize("rows,cols", [(384, 256), (200, 96)])
def test_fused_equals_separate(dev, rows, cols):
    xb = _randbits((rows, cols), rows + cols)
    x = from_bits(xb, dev)
    both = mx.quantize_alloc(x, mx.MX_ROWWISE | mx.MX_COLWISE)
    torch.cuda.synchronize()
    _check_row(xb, both)
    _check_col(xb, both)


@pytest.mark.parametrize("counts,cols", [([0, 5, 128, 131, 0, 40], 64), ([300, 1, 0, 257], 160), ([0, 0, 0, 33], 32)])
def test_segmented(dev, counts, cols):
    off, poff = offsets(counts)
    R = int(off[-1])
    xb = _randbits((R, cols), R + cols)
    x = from_bits(xb, dev)
    err = mx.new_dev_err(dev)
    out = mx.quantize_alloc(x, mx.MX_ROWWISE | mx.MX_COLWISE, torch.from_numpy(off).to(dev),
                            torch.from_numpy(poff).to(dev), dev_err=err)
    check_dev_err(err)
    oq, osf = oracle.quantize_rowwise(xb)
    assert np.array_equal(np_(out["q_row"]), oq)
    want = oracle.sf_to_tcgen05(oracle.place_sf_rows(osf, off, poff))
    assert np.array_equal(np_(out["sf_row"])[: want.size], want), "segmented rowwise scales differ"
    _check_col(xb, out, off, poff)


def test_all_bf16_values_in_varied_blocks(dev):
    # every finite bf16 pattern appears; blocks hold 31 neighbouring magnitudes plus
    # a leading element 0..24 binades above them, so every scale, subnormal E4M3
    # outputs, ties, saturation and signed zeros are all exercised
    allb = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    fin = allb[(allb & 0x7F80) != 0x7F80]
    order = np.argsort(fin & 0x7FFF, kind="stable")
    v = fin[order]
    v = v[: (v.size // 31) * 31].reshape(-1, 31)
    rng = np.random.default_rng(9)
    top = (v & 0x7FFF).max(axis=1).astype(np.int64)
    shift = rng.integers(0, 25, size=top.shape)
    lead = np.minimum(top + (shift << 7), 0x7F7F).astype(np.uint16)
    lead |= (rng.integers(0, 2, size=top.shape) << 15).astype(np.uint16)
    blk = np.concatenate([lead[:, None], v], axis=1)
    rng.shuffle(blk, axis=1)
    xb = blk[: (blk.shape[0] // 4) * 4].reshape(-1, 128)
    out = mx.quantize_alloc(from_bits(xb, dev), mx.MX_ROWWISE | mx.MX_COLWISE)
    torch.cuda.synchronize()
    _check_row(xb, out)
    _check_col(xb, out)


def test_nan_and_inf_blocks(dev):
    xb = _randbits((128, 64), 5)
    xb[3, 5] = 0x7FC0    # NaN in block (3, 0)
    xb[7, 40] = 0xFF80   # -Inf in block (7, 1)
    out = mx.quantize_alloc(from_bits(xb, dev), mx.MX_ROWWISE)
    torch.cuda.synchronize()
    _check_row(xb, out)
    q = np_(out["q_row"])
    assert np.all(q[3, :32] == 0x7F) and np.all(q[7, 32:] == 0x7F)


def test_nan_and_inf_full_tiles_both_forms(dev):
    # full 128 x 128 tiles (the 256-bit-load path, whose NaN/Inf blocks take a NaN scale)
    xb = _randbits((256, 256), 6)
    xb[3, 5] = 0x7FC0      # NaN: rowwise block (3, 0), columnwise block (5, 0)
    xb[7, 40] = 0xFF80     # -Inf: rowwise block (7, 1), columnwise block (40, 0)
    xb[200, 255] = 0x7F80  # +Inf: rowwise block (200, 7), columnwise block (255, 6)
    xb[130, 64] = 0xFFC1   # negative-signed NaN pattern
    out = mx.quantize_alloc(from_bits(xb, dev), mx.MX_ROWWISE | mx.MX_COLWISE)
    torch.cuda.synchronize()
    _check_row(xb, out)
    _check_col(xb, out)
    q = np_(out["q_row"])
    assert np.all(q[3, :32] == 0x7F) and np.all(q[7, 32:64] == 0x7F) and np.all(q[130, 64:96] == 0x7F)


@pytest.mark.parametrize("mode", [mx.MX_ROWWISE, mx.MX_ROWWISE | mx.MX_COLWISE])
def test_input_16_byte_aligned_only(dev, mode):
    # x 16-byte but not 32-byte aligned: every tile takes the general path
    rows, cols = 300, 384
    xb = _randbits((rows, cols), 17)
    buf = torch.empty(rows * cols + 8, dtype=torch.bfloat16, device=dev)
    assert buf.data_ptr() % 32 == 0
    x = buf[8:].view(rows, cols)
    x.copy_(from_bits(xb, dev))
    assert x.data_ptr() % 32 == 16
    out = mx.quantize_alloc(x, mode)
    torch.cuda.synchronize()
    _check_row(xb, out)
    if mode & mx.MX_COLWISE:
        _check_col(xb, out)


def _gather_case(name):
    g = synth.generator(31)
    if name == "tiny_top1":
        T, K, E, ids = 512, 256, 4, synth.uniform_ids(512, 4, 1, g)
    elif name == "skewed_zipf":
        d = synth.skewed(with_weights=False)
        T, K, E, ids = d["T"], 256, d["E"], d["ids"]
    elif name == "many_experts":
        # E = 1024 (the limit), 40 of them routed: the segment search spans 32 rounds of offsets,
        # and experts with more than 128 rows give full tiles next to ragged ones
        T, K, E = 1600, 256, 1024
        busy = torch.randperm(E, generator=g)[:40]
        ids = torch.stack([busy[torch.randperm(40, generator=g)[:4]] for _ in range(T)]).to(torch.int32)
    else:
        T, K, E, ids = 300, 160, 7, synth.uniform_ids(300, 7, 3, g)
    x = synth.randn_bf16((T, K), g) * torch.exp(torch.randn(T, 1, generator=g)).to(torch.bfloat16)
    return T, K, E, ids, x.to(torch.bfloat16)


@pytest.mark.parametrize("name", ["tiny_top1", "skewed_zipf", "ragged", "many_experts"])
def test_gather_quantize_is_quantize_of_gathered(dev, name):
    # quantize-on-gather == quantize(gather(x, src_row)) with the experts as segments
    T, K, E, ids, x = _gather_case(name)
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(ids.to(dev), E, dev_err=err)
    R = ids.numel()
    pb = mx.mx_padded_rows_bound(R, E)
    q_row = torch.empty(R, K, dtype=torch.uint8, device=dev)
    sf_row = torch.empty(mx.mx_sf_bytes(pb, K // 32), dtype=torch.uint8, device=dev)
    q_col = torch.empty(K, pb, dtype=torch.uint8, device=dev)
    sf_col = torch.empty(mx.mx_sf_bytes(K, pb // 32), dtype=torch.uint8, device=dev)
    mx.mxfp8_gather_quantize(x.to(dev), T, K, mx.MX_ROWWISE | mx.MX_COLWISE, pm["src_row"], pm["off"], pm["poff"],
                             E, R, pb, q_row, sf_row, q_col, sf_col, err)
    check_dev_err(err)
    p = oracle.permute(ids.numpy(), E)
    xg = oracle.gather_rows(bits(x), p["src_row"])
    oq, osf = oracle.quantize_rowwise(xg)
    assert np.array_equal(np_(q_row), oq)
    want = oracle.sf_to_tcgen05(oracle.place_sf_rows(osf, p["off"], p["poff"]))
    assert np.array_equal(np_(sf_row)[: want.size], want)
    P = int(p["poff"][-1])
    cq, csf = oracle.quantize_colwise_seg(xg, p["off"], p["poff"], pb)
    assert np.array_equal(np_(q_col)[:, :P], cq[:, :P])
    got = oracle.sf_from_tcgen05(np_(sf_col), K, pb // 32)
    assert np.array_equal(got[:, : P // 32], csf[:, : P // 32])


def test_gather_quantize_flags_out_of_range_rows(dev):
    T, K, E = 64, 64, 2
    x = synth.randn_bf16((T, K), synth.generator(3)).to(dev)
    off = torch.tensor([0, 2, 3], dtype=torch.int32, device=dev)
    poff = torch.tensor([0, 128, 256], dtype=torch.int32, device=dev)
    src = torch.tensor([5, 70, 1], dtype=torch.int32, device=dev)    # 70 is out of range
    pb = mx.mx_padded_rows_bound(3, E)
    q_row = torch.empty(3, K, dtype=torch.uint8, device=dev)
    sf_row = torch.empty(mx.mx_sf_bytes(pb, K // 32), dtype=torch.uint8, device=dev)
    err = mx.new_dev_err(dev)
    mx.mxfp8_gather_quantize(x, T, K, mx.MX_ROWWISE, src, off, poff, E, 3, 0, q_row, sf_row, None, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) & mx.MX_DEVERR_BAD_SEGMENTS
    assert np.all(np_(q_row)[1] == 0)                                  # the bad row reads as zeros
    oq, _ = oracle.quantize_rowwise(bits(x.cpu())[[5, 1]])
    assert np.array_equal(np_(q_row)[[0, 2]], oq)


def _check_ex(x_np, out, rule, off=None, poff=None):
    rows, cols = x_np.shape
    if off is None:
        off, poff = np.array([0, rows], np.int32), np.array([0, (rows + 127) // 128 * 128], np.int32)
    if out.get("q_row") is not None:
        oq, osf = oracle.quantize_rowwise_ex(x_np, rule)
        assert np.array_equal(np_(out["q_row"]), oq), "rowwise codes differ"
        want = oracle.sf_to_tcgen05(oracle.place_sf_rows(osf, off, poff))
        assert np.array_equal(np_(out["sf_row"])[: want.size], want), "rowwise scales differ"
    if out.get("q_col") is not None:
        ld = out["ld_col"]
        P = int(poff[-1])
        cq, csf = oracle.quantize_colwise_seg_ex(x_np, off, poff, ld, rule)
        assert np.array_equal(np_(out["q_col"])[:, :P], cq[:, :P]), "columnwise codes differ"
        got = oracle.sf_from_tcgen05(np_(out["sf_col"]), cols, ld // 32)
        assert np.array_equal(got[:, : P // 32], csf[:, : P // 32]), "columnwise scales differ"


@pytest.mark.parametrize("mode", [mx.MX_ROWWISE, mx.MX_COLWISE, mx.MX_ROWWISE | mx.MX_COLWISE])
@pytest.mark.parametrize("rows,cols", [(130, 96), (300, 256)])
def test_rceil_bf16(dev, mode, rows, cols):
    xb = _randbits((rows, cols), rows + 3 * cols, spread=6.0)
    out = mx.quantize_alloc(from_bits(xb, dev), mode, scale_rule=mx.MX_SCALE_RCEIL)
    torch.cuda.synchronize()
    _check_ex(xb, out, oracle.RULE_RCEIL)


@pytest.mark.parametrize("rule", [oracle.RULE_FLOOR, oracle.RULE_RCEIL])
@pytest.mark.parametrize("mode", [mx.MX_ROWWISE, mx.MX_COLWISE, mx.MX_ROWWISE | mx.MX_COLWISE])
@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 96), (256, 512), (77, 160)])
def test_fp32_input(dev, rule, mode, rows, cols):
    g = synth.generator(rows * 13 + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp(3.0 * torch.randn(rows, 1, generator=g))
    x[0, 0] = 1.0 + 2.0 ** -10          # not a bf16 value
    out = mx.quantize_alloc(x.to(dev), mode, scale_rule=rule)
    torch.cuda.synchronize()
    _check_ex(x.numpy(), out, rule)


@pytest.mark.parametrize("rule", [oracle.RULE_FLOOR, oracle.RULE_RCEIL])
def test_fp32_full_tiles_with_special_values(dev, rule):
    # whole 128 x 128 tiles of fp32 input (the full-tile column pass) with NaN, +-Inf, zero
    # blocks and a huge dynamic range, both forms from one read, over expert segments
    counts = [256, 128, 384]
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(4321)
    x = torch.randn(R, 384, generator=g) * torch.exp(4.0 * torch.randn(R, 1, generator=g))
    x[5, 7] = float("nan")
    x[200, 140] = float("inf")
    x[300, 300] = float("-inf")
    x[128:160, 256:288] = 0.0
    x[400, 33] = 3.0e38
    err = mx.new_dev_err(dev)
    out = mx.quantize_alloc(x.to(dev), mx.MX_ROWWISE | mx.MX_COLWISE, torch.from_numpy(off).to(dev),
                            torch.from_numpy(poff).to(dev), dev_err=err, scale_rule=rule)
    check_dev_err(err)
    _check_ex(x.numpy(), out, rule, off, poff)


def test_fp32_input_segmented(dev):
    counts = [0, 5, 128, 131, 0, 40]
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(77)
    x = torch.randn(R, 64, generator=g) * torch.exp(torch.randn(R, 1, generator=g))
    err = mx.new_dev_err(dev)
    out = mx.quantize_alloc(x.to(dev), mx.MX_ROWWISE | mx.MX_COLWISE, torch.from_numpy(off).to(dev),
                            torch.from_numpy(poff).to(dev), dev_err=err)
    check_dev_err(err)
    _check_ex(x.numpy(), out, oracle.RULE_FLOOR, off, poff)
