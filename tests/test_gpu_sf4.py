"""Scale arrays in the four-copy layout (mode bits MX_ROWWISE_X4 / MX_COLWISE_X4): every
quantizing call must write the same codes as without the bits, and each 512-byte scale atom
four times, each copy equal to the plain layout's atom (which the other parity tests pin to
the oracle).  The grouped GEMMs read their B operands' scales in this layout."""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import check_dev_err, dev, np_, offsets, sf_x4_first  # noqa: F401

pytestmark = pytest.mark.gpu

RC = mx.MX_ROWWISE | mx.MX_COLWISE
X4 = mx.MX_ROWWISE_X4 | mx.MX_COLWISE_X4


def _bufs(rows, cols, pb, ld, mode, device):
    srow = mx.mx_sf_bytes_x4 if mode & mx.MX_ROWWISE_X4 else mx.mx_sf_bytes
    scol = mx.mx_sf_bytes_x4 if mode & mx.MX_COLWISE_X4 else mx.mx_sf_bytes
    return dict(q_row=torch.full((max(rows, 1), cols), 0xAB, dtype=torch.uint8, device=device),
                sf_row=torch.full((srow(pb, cols // 32),), 0xAB, dtype=torch.uint8, device=device),
                q_col=torch.full((cols, ld), 0xAB, dtype=torch.uint8, device=device),
                sf_col=torch.full((scol(cols, ld // 32),), 0xAB, dtype=torch.uint8, device=device))


def _same(plain, x4, mode):
    assert np.array_equal(np_(plain["q_row"]), np_(x4["q_row"]))
    assert np.array_equal(np_(plain["q_col"]), np_(x4["q_col"]))
    row = sf_x4_first(x4["sf_row"]) if mode & mx.MX_ROWWISE_X4 else np_(x4["sf_row"])
    col = sf_x4_first(x4["sf_col"]) if mode & mx.MX_COLWISE_X4 else np_(x4["sf_col"])
    assert np.array_equal(np_(plain["sf_row"]), row)
    assert np.array_equal(np_(plain["sf_col"]), col)


@pytest.mark.parametrize("xmode", [mx.MX_ROWWISE_X4, mx.MX_COLWISE_X4, X4])
@pytest.mark.parametrize("dtype,rule", [(torch.bfloat16, mx.MX_SCALE_FLOOR), (torch.bfloat16, mx.MX_SCALE_RCEIL),
                                        (torch.float32, mx.MX_SCALE_FLOOR)])
def test_quantize_x4(dev, xmode, dtype, rule):
    counts = [0, 37, 300, 129, 1]
    off, poff = offsets(counts)
    R, K, E = int(off[-1]), 160, len(counts)
    g = synth.generator(77)
    x = (torch.randn(R, K, generator=g) * torch.exp(2 * torch.randn(R, 1, generator=g))).to(dtype).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    err = mx.new_dev_err(dev)
    dt = mx.MX_DTYPE_F32 if dtype == torch.float32 else mx.MX_DTYPE_BF16
    out = {}
    for mode in (RC, RC | xmode):
        b = _bufs(R, K, pb, pb, mode, dev)
        mx.mxfp8_quantize_ex(x, dt, rule, R, K, mode, offd, poffd, E, pb, b["q_row"], b["sf_row"], b["q_col"],
                             b["sf_col"], err)
        out[mode] = b
    check_dev_err(err)
    _same(out[RC], out[RC | xmode], RC | xmode)


def test_gather_quantize_x4(dev):
    T, K, E, k = 300, 256, 7, 3
    g = synth.generator(78)
    ids = synth.uniform_ids(T, E, k, g)
    x = synth.randn_bf16((T, K), g).to(dev)
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(ids.to(dev), E, dev_err=err)
    R = T * k
    pb = mx.mx_padded_rows_bound(R, E)
    out = {}
    for mode in (RC, RC | mx.MX_COLWISE_X4):
        b = _bufs(R, K, pb, pb, mode, dev)
        mx.mxfp8_gather_quantize(x, T, K, mode, pm["src_row"], pm["off"], pm["poff"], E, R, pb, b["q_row"],
                                 b["sf_row"], b["q_col"], b["sf_col"], err)
        out[mode] = b
    check_dev_err(err)
    _same(out[RC], out[RC | mx.MX_COLWISE_X4], RC | mx.MX_COLWISE_X4)


@pytest.mark.parametrize("bwd", [False, True])
@pytest.mark.parametrize("xmode", [mx.MX_COLWISE_X4, X4])
def test_swiglu_x4(dev, bwd, xmode):
    counts = [0, 37, 300, 129]
    off, poff = offsets(counts)
    R, I, E = int(off[-1]), 256, len(counts)
    g = synth.generator(79)
    a = synth.randn_bf16((R, 2 * I), g, std=3.0).to(dev)
    dh = synth.randn_bf16((R, I), g, std=1e-2).to(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    pb = mx.mx_padded_rows_bound(R, E)
    cols = 2 * I if bwd else I
    err = mx.new_dev_err(dev)
    out = {}
    for mode in (RC, RC | xmode):
        b = _bufs(R, cols, pb, pb, mode, dev)
        if bwd:
            mx.mxfp8_swiglu_bwd_quantize(dh, a, R, I, mode, offd, poffd, E, pb, b["q_row"], b["sf_row"], b["q_col"],
                                         b["sf_col"], err)
        else:
            mx.mxfp8_swiglu_quantize(a, R, I, mode, offd, poffd, E, pb, b["q_row"], b["sf_row"], b["q_col"],
                                     b["sf_col"], err)
        out[mode] = b
    check_dev_err(err)
    _same(out[RC], out[RC | xmode], RC | xmode)
