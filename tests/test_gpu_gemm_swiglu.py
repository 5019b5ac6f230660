"""GEMM1 with SwiGLU and MXFP8 quantization in its epilogue (grouped_gemm_mxfp8_fwd_swiglu).

1. Bit-exact against the two-call path it fuses -- grouped_gemm_mxfp8_fwd then
   mxfp8_swiglu_quantize, each pinned to the oracle in its own test file: the same
   accumulation, the same fp32 SwiGLU expression on the same bf16 values and the same
   scale rule, so out1, both code forms and both scale forms must agree byte for byte.
2. Against the oracle directly, on operands for which the GEMM is exact: out1 equal to the
   oracle's bf16 GEMM output bit for bit, and h's codes and scales equal to the oracle's
   quantization of its SwiGLU of that output except where the kernel's fp32 SwiGLU error
   bound explains a difference (near_tie)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import ROW_B, bits, check_dev_err, dev, np_, offsets, sf_x4_first  # noqa: F401
from swiglu_check import check_swiglu_outputs

pytestmark = pytest.mark.gpu

RC = mx.MX_ROWWISE | mx.MX_COLWISE


def _bufs(R, I, pb, ld, device, mode=RC):
    srow = mx.mx_sf_bytes_x4 if mode & mx.MX_ROWWISE_X4 else mx.mx_sf_bytes
    scol = mx.mx_sf_bytes_x4 if mode & mx.MX_COLWISE_X4 else mx.mx_sf_bytes
    return dict(out1=torch.full((max(R, 1), 2 * I), float("nan"), dtype=torch.bfloat16, device=device),
                q_row=torch.zeros(max(R, 1), I, dtype=torch.uint8, device=device),
                sf_row=torch.zeros(srow(pb, I // 32), dtype=torch.uint8, device=device),
                q_col=torch.zeros(I, ld, dtype=torch.uint8, device=device),
                sf_col=torch.zeros(scol(I, ld // 32), dtype=torch.uint8, device=device))


def _plain(buf, x4):
    return sf_x4_first(buf) if x4 else np_(buf)


@pytest.mark.parametrize("counts,I,K,mode", [
    ([0, 37, 300, 129, 1], 256, 384, RC | mx.MX_COLWISE_X4),
    ([513], 128, 256, RC),
    ([128, 0, 0, 255, 64, 7], 384, 128, RC | mx.MX_ROWWISE_X4 | mx.MX_COLWISE_X4),
])
def test_fused_equals_two_calls(dev, counts, I, K, mode):
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(R + I + K)
    x = synth.randn_bf16((R, K), g).to(dev)
    w1 = synth.randn_bf16((E * 2 * I, K), g, std=K ** -0.5).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    qa = mx.quantize_alloc(x, mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qw = mx.quantize_alloc(w1, ROW_B, dev_err=err)
    fu = _bufs(R, I, pb, pb, dev, mode)
    mx.grouped_gemm_mxfp8_fwd_swiglu(qa["q_row"], qa["sf_row"], qw["q_row"], qw["sf_row"], offd, poffd, E, R, I, K,
                                     fu["out1"], fu["q_row"], fu["sf_row"], fu["q_col"], fu["sf_col"], pb, mode, err)
    sp = _bufs(R, I, pb, pb, dev, mode)
    mx.grouped_gemm_mxfp8_fwd(qa["q_row"], qa["sf_row"], qw["q_row"], qw["sf_row"], offd, poffd, E, R, 2 * I, K,
                              sp["out1"], err)
    mx.mxfp8_swiglu_quantize(sp["out1"], R, I, mode, offd, poffd, E, pb, sp["q_row"], sp["sf_row"], sp["q_col"],
                             sp["sf_col"], err)
    check_dev_err(err)
    P = int(poff[-1])
    assert np.array_equal(bits(fu["out1"][:R]), bits(sp["out1"][:R]))
    assert np.array_equal(np_(fu["q_row"][:R]), np_(sp["q_row"][:R]))
    assert np.array_equal(np_(fu["q_col"][:, :P]), np_(sp["q_col"][:, :P]))
    rx4, cx4 = bool(mode & mx.MX_ROWWISE_X4), bool(mode & mx.MX_COLWISE_X4)
    sf_f = oracle.sf_from_tcgen05(_plain(fu["sf_row"], rx4), pb, I // 32)[:P]
    sf_s = oracle.sf_from_tcgen05(_plain(sp["sf_row"], rx4), pb, I // 32)[:P]
    assert np.array_equal(sf_f, sf_s)
    cf = oracle.sf_from_tcgen05(_plain(fu["sf_col"], cx4), I, pb // 32)[:, :P // 32]
    cs = oracle.sf_from_tcgen05(_plain(sp["sf_col"], cx4), I, pb // 32)[:, :P // 32]
    assert np.array_equal(cf, cs)


def _grid_bf16(shape, rng, step):
    """Integers in [-3, 3] times a power of two: every 32-element block quantizes exactly (the
    block scale is a power of two and the codes hold k * 128 or k * 256 exactly)."""
    k = rng.integers(-3, 4, size=shape)
    return torch.from_numpy((k * step).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("mode", [RC, RC | mx.MX_COLWISE_X4])
def test_fused_against_oracle_exact_operands(dev, mode):
    # Operands on a small integer grid make the GEMM exact: every product and partial sum is a
    # multiple of 2^-7 below 2^10, so the fp32 accumulation in tensor memory and the oracle's
    # fp64 sum are the same number and both round it to the same bf16.  So out1 must equal the
    # oracle bit for bit, and h is checked against the oracle's SwiGLU of that same out1 with
    # differences allowed only where the kernel's fp32 SwiGLU error bound explains them.
    counts = [0, 37, 300, 129, 1]
    I, K = 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    rng = np.random.default_rng(4242)
    x = _grid_bf16((R, K), rng, 2.0 ** -3)
    w1 = _grid_bf16((E * 2 * I, K), rng, 2.0 ** -4)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    qa = mx.quantize_alloc(x.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qw = mx.quantize_alloc(w1.to(dev), ROW_B, dev_err=err)
    fu = _bufs(R, I, pb, pb, dev, mode)
    mx.grouped_gemm_mxfp8_fwd_swiglu(qa["q_row"], qa["sf_row"], qw["q_row"], qw["sf_row"], offd, poffd, E, R, I, K,
                                     fu["out1"], fu["q_row"], fu["sf_row"], fu["q_col"], fu["sf_col"], pb, mode, err)
    check_dev_err(err)
    aq, asf = oracle.quantize_rowwise(bits(x))
    wq, wsf = oracle.quantize_rowwise(bits(w1))
    a1 = np.zeros((R, 2 * I))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            a1[r0:r1] = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], wq[e * 2 * I:(e + 1) * 2 * I],
                                       wsf[e * 2 * I:(e + 1) * 2 * I])
    assert np.all(a1 * 2.0 ** 7 == np.round(a1 * 2.0 ** 7)) and np.abs(a1).max() < 2.0 ** 10
    a1_bits = oracle.to_bf16_bits(a1).reshape(a1.shape)
    assert np.array_equal(bits(fu["out1"][:R]), a1_bits), "exact GEMM: out1 must match the oracle bit for bit"
    flips = check_swiglu_outputs(False, a1_bits, None, off, poff, fu["q_row"], fu["sf_row"], fu["q_col"],
                                 fu["sf_col"], x4=(False, bool(mode & mx.MX_COLWISE_X4)))
    print("explained near-tie differences (codes, scales) rowwise / columnwise:", flips)


def test_fused_takes_one_copy_w1_scales(dev):
    # grouped_gemm_mxfp8_fwd_swiglu_ex with MX_GEMM_B_SCALES_X1 reads SFW1 in the plain layout and
    # gives the same bytes as the default call on the four-copy layout
    counts, I, K = [0, 37, 300, 129], 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(5151)
    x = synth.randn_bf16((R, K), g).to(dev)
    w1 = synth.randn_bf16((E * 2 * I, K), g, std=K ** -0.5).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    qa = mx.quantize_alloc(x, mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qw1 = mx.quantize_alloc(w1, mx.MX_ROWWISE, dev_err=err)
    qw4 = mx.quantize_alloc(w1, ROW_B, dev_err=err)
    a, b = _bufs(R, I, pb, pb, dev), _bufs(R, I, pb, pb, dev)
    mx.grouped_gemm_mxfp8_fwd_swiglu_ex(qa["q_row"], qa["sf_row"], qw1["q_row"], qw1["sf_row"], offd, poffd, E, R, I,
                                        K, a["out1"], a["q_row"], a["sf_row"], a["q_col"], a["sf_col"], pb, RC,
                                        mx.MX_GEMM_B_SCALES_X1, err)
    mx.grouped_gemm_mxfp8_fwd_swiglu(qa["q_row"], qa["sf_row"], qw4["q_row"], qw4["sf_row"], offd, poffd, E, R, I, K,
                                     b["out1"], b["q_row"], b["sf_row"], b["q_col"], b["sf_col"], pb, RC, err)
    check_dev_err(err)
    P = int(poff[-1])
    assert np.array_equal(bits(a["out1"][:R]), bits(b["out1"][:R]))
    assert np.array_equal(np_(a["q_row"][:R]), np_(b["q_row"][:R]))
    assert np.array_equal(np_(a["q_col"][:, :P]), np_(b["q_col"][:, :P]))
    assert np.array_equal(np_(a["sf_row"]), np_(b["sf_row"]))
    assert np.array_equal(np_(a["sf_col"]), np_(b["sf_col"]))
