"""GEMM1 with SwiGLU and MXFP8 quantization in its epilogue (grouped_gemm_mxfp8_fwd_swiglu).

1. Bit-exact against the two-call path it fuses -- grouped_gemm_mxfp8_fwd then
   mxfp8_swiglu_quantize, each pinned to the oracle in its own test file: the same
   accumulation, the same fp32 SwiGLU expression on the same bf16 values and the same
   scale rule, so out1, both code forms and both scale forms must agree byte for byte.
2. Against the oracle directly: out1 within 2e-2 x rms of the oracle's fp64 GEMM, and the
   dequantized h within one E4M3 step (or the per-GEMM bound) of the oracle's SwiGLU of
   its own bf16 GEMM output."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import ROW_B, TOL, bits, check_dev_err, dev, np_, offsets, rel_err, sf_x4_first  # noqa: F401

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


def test_fused_against_oracle(dev):
    counts = [0, 37, 300, 129, 1]
    I, K = 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(4242)
    x = synth.randn_bf16((R, K), g)
    w1 = synth.randn_bf16((E * 2 * I, K), g, std=K ** -0.5)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err = mx.new_dev_err(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    qa = mx.quantize_alloc(x.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qw = mx.quantize_alloc(w1.to(dev), ROW_B, dev_err=err)
    fu = _bufs(R, I, pb, pb, dev)
    mx.grouped_gemm_mxfp8_fwd_swiglu(qa["q_row"], qa["sf_row"], qw["q_row"], qw["sf_row"], offd, poffd, E, R, I, K,
                                     fu["out1"], fu["q_row"], fu["sf_row"], fu["q_col"], fu["sf_col"], pb, RC, err)
    check_dev_err(err)
    aq, asf = oracle.quantize_rowwise(bits(x))
    wq, wsf = oracle.quantize_rowwise(bits(w1))
    a1 = np.zeros((R, 2 * I))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            a1[r0:r1] = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], wq[e * 2 * I:(e + 1) * 2 * I],
                                       wsf[e * 2 * I:(e + 1) * 2 * I])
    got1 = (bits(fu["out1"][:R]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert rel_err(got1, a1) <= TOL
    h32 = oracle.swiglu_fwd(oracle.to_bf16_bits(a1).reshape(a1.shape))
    hq, hsf = oracle.quantize_rowwise_ex(h32)
    sf_rm = oracle.sf_from_tcgen05(np_(fu["sf_row"]), pb, I // 32)
    rows_pad = np.concatenate([np.arange(poff[e], poff[e] + counts[e]) for e in range(E)]).astype(np.int64)

    def deq(q, sf):
        return oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape) * np.exp2(
            np.repeat(sf.astype(np.float64) - 127, 32, axis=1))

    dg, dr = deq(np_(fu["q_row"][:R]), sf_rm[rows_pad]), deq(hq, oracle.place_sf_rows(hsf, off, poff)[rows_pad])
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(dr), 2.0 ** -126))) - 3)
    rms = float(np.sqrt(np.mean(dr ** 2)))
    # one E4M3 step where the two fp32 SwiGLU values straddle a rounding boundary, plus the
    # GEMM-level bound for the bf16 inputs of SwiGLU (one GEMM stage)
    assert np.all(np.abs(dg - dr) <= np.maximum(step, 2 ** -9 * np.abs(dr)) + 2 * TOL * rms)
    assert np.linalg.norm(dg - dr) <= TOL * np.linalg.norm(dr)
