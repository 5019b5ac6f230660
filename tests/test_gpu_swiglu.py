"""Fused SwiGLU + MXFP8 quantization (forward and backward) on the GPU vs the oracle.

Both sides decide each E4M3 code and scale from an fp32 SwiGLU value (the kernel's
precision).  The GPU forms that value with expf and fp32 arithmetic, the oracle in double
rounded once to fp32; the two fp32 values can differ in their last bits, so a value lying
within that distance of an E4M3 rounding boundary may take the neighbouring code.  The
test therefore requires: every dequantized element within one E4M3 step of the oracle's,
and at most 1e-4 of the codes (and 1e-3 of the scales) different."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import check_dev_err, dev, np_, offsets  # noqa: F401
from gpu_util import bits

pytestmark = pytest.mark.gpu


def _deq(q, sf_rm):
    v = oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape)
    return v * np.exp2(np.repeat(sf_rm.astype(np.float64) - 127, 32, axis=1))


def _close(q_gpu, sf_gpu_rm, q_ref, sf_ref_rm):
    dg, dr = _deq(q_gpu, sf_gpu_rm), _deq(q_ref, sf_ref_rm)
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(dr), 1e-300))) - 3)   # one E4M3 step at |ref|
    scale_step = np.exp2(np.repeat(sf_ref_rm.astype(np.float64) - 127 - 9, 32, axis=1))
    assert np.all(np.abs(dg - dr) <= np.maximum(step, scale_step) * (1 + 1e-9))
    assert np.mean(q_gpu != q_ref) <= 1e-4
    assert np.mean(sf_gpu_rm != sf_ref_rm) <= 1e-3


@pytest.mark.parametrize("counts,I", [([512], 128), ([0, 37, 300, 129], 256)])
def test_swiglu_fwd_and_bwd(dev, counts, I):
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(R + I)
    a = synth.randn_bf16((R, 2 * I), g, std=3.0)
    dh = synth.randn_bf16((R, I), g, std=1e-2)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    E = len(counts)
    pb = mx.mx_padded_rows_bound(R, E)
    err = mx.new_dev_err(dev)
    RC = mx.MX_ROWWISE | mx.MX_COLWISE
    for bwd in (False, True):
        cols = 2 * I if bwd else I
        q_row = torch.empty(R, cols, dtype=torch.uint8, device=dev)
        sf_row = torch.empty(mx.mx_sf_bytes(pb, cols // 32), dtype=torch.uint8, device=dev)
        q_col = torch.empty(cols, pb, dtype=torch.uint8, device=dev)
        sf_col = torch.empty(mx.mx_sf_bytes(cols, pb // 32), dtype=torch.uint8, device=dev)
        if bwd:
            mx.mxfp8_swiglu_bwd_quantize(dh.to(dev), a.to(dev), R, I, RC, offd, poffd, E, pb, q_row, sf_row, q_col,
                                         sf_col, err)
            ref32 = oracle.swiglu_bwd(bits(dh), bits(a))
        else:
            mx.mxfp8_swiglu_quantize(a.to(dev), R, I, RC, offd, poffd, E, pb, q_row, sf_row, q_col, sf_col, err)
            ref32 = oracle.swiglu_fwd(bits(a))
        check_dev_err(err)
        oq, osf = oracle.quantize_rowwise_ex(ref32)
        P = int(poff[-1])
        sf_rm = oracle.sf_from_tcgen05(np_(sf_row), P, cols // 32)
        sf_ref = oracle.place_sf_rows(osf, off, poff)
        # rowwise: data rows dense, scale rows at padded positions
        rows_pad = np.concatenate([np.arange(poff[e], poff[e] + counts[e]) for e in range(E)]).astype(np.int64)
        _close(np_(q_row), sf_rm[rows_pad], oq, sf_ref[rows_pad])
        cq, csf = oracle.quantize_colwise_seg_ex(ref32, off, poff, pb)
        got_sf = oracle.sf_from_tcgen05(np_(sf_col), cols, pb // 32)
        _close(np_(q_col)[:, :P], got_sf[:, : P // 32], cq[:, :P], csf[:, : P // 32])
