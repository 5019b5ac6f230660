"""Blocked code layout (E4M3 codes in 128 x 128 blocks of 16 KiB, block (i, j) at
(i * cols / 128 + j) * 16384, each block row-major).

1. The quantizer's blocked outputs (mode bits MX_ROWWISE_BLK / MX_COLWISE_BLK) are its
   row-major outputs rearranged block by block, byte for byte, with the same scales --
   on the 256-bit-load path, the 16-byte path (input not 32-byte aligned), fp32 input and
   columnwise segments with padding positions.
2. The grouped GEMMs reading blocked B operands (MX_GEMM_B_BLOCKED) give the row-major
   path's outputs bit for bit (same codes, same scales, same MMAs): forward on both tile
   shapes, dgrad, wgrad, the SwiGLU forward, and the public *_ex calls.  The row-major path
   is pinned to the oracle in test_gpu_gemm.py / test_gpu_gemm_swiglu.py."""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, ROW_B, check_dev_err, dev, np_, offsets  # noqa: F401

pytestmark = pytest.mark.gpu

RC = mx.MX_ROWWISE | mx.MX_COLWISE
RB, CB = mx.MX_ROWWISE_BLK, mx.MX_COLWISE_BLK


def _unblock(q_flat, rows, cols):
    """Blocked bytes -> the row-major [rows x cols] matrix (the header's layout definition)."""
    return q_flat.reshape(rows // 128, cols // 128, 128, 128).permute(0, 2, 1, 3).reshape(rows, cols)


def _rand(shape, seed, std=1.0, dtype=torch.bfloat16):
    t = synth.randn_bf16(shape, synth.generator(seed), std=std)
    return t if dtype == torch.bfloat16 else t.float()


def _offset_copy(x, elems):
    """x in a buffer that starts `elems` elements past an allocation (16 bytes: not 32-byte aligned)."""
    buf = torch.empty(x.numel() + elems, dtype=x.dtype, device=x.device)
    y = buf[elems:].view(x.shape)
    y.copy_(x)
    return y


@pytest.mark.parametrize("rows,cols,dtype,misalign", [
    (256, 384, torch.bfloat16, False),
    (384, 256, torch.bfloat16, True),
    (128, 512, torch.float32, False),
])
@pytest.mark.parametrize("mode", [RC | RB | CB, RC | RB | CB | mx.MX_ROWWISE_X4 | mx.MX_COLWISE_X4,
                                  mx.MX_ROWWISE | RB, mx.MX_COLWISE | CB, RC | CB])
def test_quantize_blocked_is_row_major_rearranged(dev, rows, cols, dtype, misalign, mode):
    x = _rand((rows, cols), rows * 7 + cols, dtype=dtype).to(dev)
    if misalign:
        x = _offset_copy(x, 16 // x.element_size())
        assert x.data_ptr() % 32 == 16
    err = mx.new_dev_err(dev)
    std = mode & ~(RB | CB)
    a = mx.quantize_alloc(x, std, dev_err=err)
    b = mx.quantize_alloc(x, mode, dev_err=err)
    check_dev_err(err)
    if mode & mx.MX_ROWWISE:
        got = _unblock(b["q_row"].reshape(-1), rows, cols) if mode & RB else b["q_row"]
        assert torch.equal(got, a["q_row"])
        assert torch.equal(b["sf_row"], a["sf_row"])
    if mode & mx.MX_COLWISE:
        ld = a["ld_col"]
        got = _unblock(b["q_col"].reshape(-1), cols, ld) if mode & CB else b["q_col"]
        assert torch.equal(got, a["q_col"])
        assert torch.equal(b["sf_col"], a["sf_col"])


@pytest.mark.parametrize("counts,cols", [([0, 37, 128, 300, 1], 256), ([129, 0, 255, 64], 384)])
def test_quantize_blocked_columnwise_segments(dev, counts, cols):
    # columnwise over expert segments: the blocked codes of every position below poff[E]
    # (data and zero padding) are the row-major ones; the scales written are the same bytes
    E = len(counts)
    off, poff = offsets(counts)
    R, P = int(off[-1]), int(poff[-1])
    x = _rand((R, cols), 4242 + R).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    a = mx.quantize_alloc(x, RC, offd, poffd, dev_err=err)
    b = mx.quantize_alloc(x, RC | CB, offd, poffd, dev_err=err)
    check_dev_err(err)
    ld = a["ld_col"]
    assert torch.equal(b["q_row"], a["q_row"])
    nsf = P * cols // 32   # scale rows past poff[E] are not written
    assert torch.equal(b["sf_row"][:nsf], a["sf_row"][:nsf])
    got = _unblock(b["q_col"].reshape(-1), cols, ld)
    assert torch.equal(got[:, :P], a["q_col"][:, :P])
    atoms = lambda t: np_(t).reshape(cols // 128, ld // 128, 512)[:, :P // 128]
    assert np.array_equal(atoms(b["sf_col"]), atoms(a["sf_col"]))


def _passes(dev, xp, w, dy, off, poff, E, N, K, blocked, flags=0, ctas_per_mma=0, cluster_pairs=0):
    """Forward, dgrad and wgrad through the internal test entry, B operands row-major or blocked."""
    R = xp.shape[0]
    x4 = not (flags & mx.MX_GEMM_B_SCALES_X1)
    row_b = (ROW_B if x4 else mx.MX_ROWWISE) | (RB if blocked else 0)
    col_b = (COL_B if x4 else mx.MX_COLWISE) | (CB if blocked else 0)
    fl = flags | (mx.MX_GEMM_B_BLOCKED if blocked else 0)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb = mx.quantize_alloc(w.reshape(E * N, K).to(dev), row_b, dev_err=err)
    C = torch.full((max(R, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    run = lambda *a: mx.testing_grouped_gemm(*a, err, flags=fl, ctas_per_mma=ctas_per_mma,
                                             cluster_pairs=cluster_pairs)
    assert run(mx.MX_TESTING_FWD, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K, 0,
               C) == 0
    qd = mx.quantize_alloc(dy.to(dev), RC, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=dev)
    qw = mx.quantize_alloc(w.reshape(E * N, K).to(dev), col_b, woff, woff, dev_err=err, ld_col=E * N)
    dX = torch.full((max(R, 1), K), float("nan"), dtype=torch.bfloat16, device=dev)
    assert run(mx.MX_TESTING_DGRAD, qd["q_row"], qd["sf_row"], qw["q_col"], qw["sf_col"], offd, poffd, E, R, K, N, 0,
               dX) == 0
    qx = mx.quantize_alloc(xp.to(dev), col_b, offd, poffd, dev_err=err)
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    assert run(mx.MX_TESTING_WGRAD, qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, 0, N, K,
               qd["ld_col"], dW) == 0
    check_dev_err(err)
    return C[:R], dX[:R], dW


@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("flags", [0, mx.MX_GEMM_B_SCALES_X1])
@pytest.mark.parametrize("counts,N,K", [([0, 37, 128, 300, 1], 384, 384), ([1000, 3, 260], 256, 512)])
def test_gemm_blocked_b_matches_row_major(dev, counts, N, K, flags, ctas):
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 61 + R), _rand((E, N, K), 62 + R), _rand((R, N), 63 + R, std=1e-2)
    ref = _passes(dev, xp, w, dy, off, poff, E, N, K, False, flags, ctas)
    got = _passes(dev, xp, w, dy, off, poff, E, N, K, True, flags, ctas)
    for name, g, r in zip(("fwd", "dgrad"), got[:2], ref[:2]):
        assert torch.equal(g.view(torch.int16), r.view(torch.int16)), name
    assert torch.equal(got[2].view(torch.int32), ref[2].view(torch.int32)), "wgrad"


@pytest.mark.parametrize("ctas", [1, 2])
def test_blocked_b_in_clusters(dev, ctas):
    # blocked B operands inside the multicast clusters (internal option cluster_pairs = 2; with
    # blocked B each CTA copies its whole B tile itself): bit-identical to row-major B without
    # clusters
    counts, N, K = [0, 37, 128, 300, 1], 640, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 81 + R), _rand((E, N, K), 82 + R), _rand((R, N), 83 + R, std=1e-2)
    ref = _passes(dev, xp, w, dy, off, poff, E, N, K, False, 0, ctas, cluster_pairs=1)
    got = _passes(dev, xp, w, dy, off, poff, E, N, K, True, 0, ctas, cluster_pairs=2)
    for name, g, r in zip(("fwd", "dgrad"), got[:2], ref[:2]):
        assert torch.equal(g.view(torch.int16), r.view(torch.int16)), name
    assert torch.equal(got[2].view(torch.int32), ref[2].view(torch.int32)), "wgrad"


def test_public_calls_read_blocked_b(dev):
    # the public *_ex calls with MX_GEMM_B_BLOCKED on many small experts (single-CTA tiles):
    # forward, dgrad and wgrad equal the default calls on row-major B
    E, N, K = 24, 256, 384
    counts = [int(c) for c in np.random.default_rng(7).integers(0, 300, E)]
    counts[3] = 0
    off, poff = offsets(counts)
    R = int(off[-1])
    xp, w, dy = _rand((R, K), 71), _rand((E * N, K), 72), _rand((R, N), 73, std=1e-2)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), RC, offd, poffd, dev_err=err)
    qd = mx.quantize_alloc(dy.to(dev), RC, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=dev)
    out = {}
    for blk in (False, True):
        fl = mx.MX_GEMM_B_BLOCKED if blk else 0
        qb = mx.quantize_alloc(w.to(dev), ROW_B | (RB if blk else 0), dev_err=err)
        qw = mx.quantize_alloc(w.to(dev), COL_B | (CB if blk else 0), woff, woff, dev_err=err, ld_col=E * N)
        qx = mx.quantize_alloc(xp.to(dev), COL_B | (CB if blk else 0), offd, poffd, dev_err=err)
        C = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(R, K, dtype=torch.bfloat16, device=dev)
        dW = torch.empty(E, N, K, dtype=torch.float32, device=dev)
        mx.grouped_gemm_mxfp8_fwd_ex(qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K,
                                     C, fl, err)
        mx.grouped_gemm_mxfp8_dgrad_ex(qd["q_row"], qd["sf_row"], qw["q_col"], qw["sf_col"], offd, poffd, E, R, K, N,
                                       dX, fl, err)
        mx.grouped_gemm_mxfp8_wgrad_ex(qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, N, K,
                                       qd["ld_col"], dW, fl, err)
        check_dev_err(err)
        out[blk] = (C.view(torch.int16), dX.view(torch.int16), dW.view(torch.int32))
    for name, g, r in zip(("fwd", "dgrad", "wgrad"), out[True], out[False]):
        assert torch.equal(g, r), name


def test_swiglu_gemm_reads_blocked_w1(dev):
    # grouped_gemm_mxfp8_fwd_swiglu_ex with MX_GEMM_B_BLOCKED (the pair's CTAs stage blocked gate
    # and up rows) gives the default call's out1, codes and scales byte for byte
    counts, I, K = [0, 37, 300, 129], 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R, P = int(off[-1]), int(poff[-1])
    g = synth.generator(5252)
    x = synth.randn_bf16((R, K), g).to(dev)
    w1 = synth.randn_bf16((E * 2 * I, K), g, std=K ** -0.5).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    qa = mx.quantize_alloc(x, mx.MX_ROWWISE, offd, poffd, dev_err=err)
    res = []
    for blk in (False, True):
        qw = mx.quantize_alloc(w1, ROW_B | (RB if blk else 0), dev_err=err)
        o = dict(out1=torch.full((R, 2 * I), float("nan"), dtype=torch.bfloat16, device=dev),
                 q_row=torch.zeros(R, I, dtype=torch.uint8, device=dev),
                 sf_row=torch.zeros(mx.mx_sf_bytes(pb, I // 32), dtype=torch.uint8, device=dev),
                 q_col=torch.zeros(I, pb, dtype=torch.uint8, device=dev),
                 sf_col=torch.zeros(mx.mx_sf_bytes(I, pb // 32), dtype=torch.uint8, device=dev))
        mx.grouped_gemm_mxfp8_fwd_swiglu_ex(qa["q_row"], qa["sf_row"], qw["q_row"], qw["sf_row"], offd, poffd, E, R,
                                            I, K, o["out1"], o["q_row"], o["sf_row"], o["q_col"], o["sf_col"], pb, RC,
                                            mx.MX_GEMM_B_BLOCKED if blk else 0, err)
        check_dev_err(err)
        res.append(o)
    a, b = res
    assert torch.equal(a["out1"].view(torch.int16), b["out1"].view(torch.int16))
    assert torch.equal(a["q_row"], b["q_row"])
    assert torch.equal(a["q_col"][:, :P], b["q_col"][:, :P])
    assert torch.equal(a["sf_row"], b["sf_row"])
    assert torch.equal(a["sf_col"], b["sf_col"])


@pytest.mark.parametrize("dtype,rule", [(torch.bfloat16, mx.MX_SCALE_RCEIL), (torch.float32, mx.MX_SCALE_FLOOR)])
def test_quantize_blocked_columnwise_ragged_rows(dev, dtype, rule):
    # columnwise blocked codes of 200 rows (positions 200..255 of the last block are written as
    # zero codes), under the ceiling scale rule and from fp32 input: the row-major bytes rearranged
    rows, cols = 200, 384
    x = _rand((rows, cols), 777, dtype=dtype).to(dev)
    err = mx.new_dev_err(dev)
    a = mx.quantize_alloc(x, mx.MX_COLWISE, dev_err=err, scale_rule=rule)
    b = mx.quantize_alloc(x, mx.MX_COLWISE | CB, dev_err=err, scale_rule=rule)
    check_dev_err(err)
    ld = a["ld_col"]
    assert ld == 256
    assert torch.equal(_unblock(b["q_col"].reshape(-1), cols, ld), a["q_col"])
    assert torch.equal(b["sf_col"], a["sf_col"])
    assert not torch.any(a["q_col"][:, rows:])
