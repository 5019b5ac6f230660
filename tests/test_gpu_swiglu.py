"""Fused SwiGLU + MXFP8 quantization (forward and backward) on the GPU vs the oracle.

Both sides decide each E4M3 code and scale byte from an fp32 SwiGLU value (the kernel's
precision).  The kernel forms it on the special-function unit and in fp32, the oracle in
double rounded once to fp32, so the two fp32 values differ by at most a bound that follows
from the kernel's arithmetic (near_tie.swiglu_bounds).  Every code or scale byte that differs
from the oracle's must be explained by that bound: the oracle's value lies within it of the
rounding midpoint between the two codes (or its block maximum within it of the power of two
between the two scales).  Any other difference fails."""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import check_dev_err, dev, offsets  # noqa: F401
from gpu_util import bits
from swiglu_check import check_swiglu_outputs

pytestmark = pytest.mark.gpu


_MANY = [0] * 1024          # E = 1024, three experts routed (the segment search spans 32 rounds)
_MANY[17], _MANY[600], _MANY[1023] = 300, 129, 5


@pytest.mark.parametrize("counts,I,std", [([512], 128, 3.0), ([0, 37, 300, 129], 256, 3.0), ([700, 1, 333], 384, 1.0),
                                          (_MANY, 128, 1.0),
                                          # the MoE FFN intermediate size: every column tile of the step
                                          ([300, 0, 64, 193], 2048, 1.0)])
def test_swiglu_fwd_and_bwd(dev, counts, I, std):
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(R + I)
    a = synth.randn_bf16((R, 2 * I), g, std=std)
    dh = synth.randn_bf16((R, I), g, std=1e-2)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    E = len(counts)
    pb = mx.mx_padded_rows_bound(R, E)
    err = mx.new_dev_err(dev)
    RC = mx.MX_ROWWISE | mx.MX_COLWISE
    flips = {}
    for bwd in (False, True):
        cols = 2 * I if bwd else I
        q_row = torch.empty(R, cols, dtype=torch.uint8, device=dev)
        sf_row = torch.empty(mx.mx_sf_bytes(pb, cols // 32), dtype=torch.uint8, device=dev)
        q_col = torch.empty(cols, pb, dtype=torch.uint8, device=dev)
        sf_col = torch.empty(mx.mx_sf_bytes(cols, pb // 32), dtype=torch.uint8, device=dev)
        if bwd:
            mx.mxfp8_swiglu_bwd_quantize(dh.to(dev), a.to(dev), R, I, RC, offd, poffd, E, pb, q_row, sf_row, q_col,
                                         sf_col, err)
        else:
            mx.mxfp8_swiglu_quantize(a.to(dev), R, I, RC, offd, poffd, E, pb, q_row, sf_row, q_col, sf_col, err)
        check_dev_err(err)
        flips["bwd" if bwd else "fwd"] = check_swiglu_outputs(bwd, bits(a), bits(dh), off, poff, q_row, sf_row,
                                                              q_col, sf_col)
    print("explained near-tie differences (codes, scales) rowwise / columnwise:", flips)


def test_swiglu_special_values(dev):
    """Gate values with |g| >= 64 (the kernels' exact path for the sigmoid's e^-|g| step, which
    keeps subnormal results) mixed into blocks of ordinary values, next to warps that take the
    flushed path; and NaN / Inf in gate, up and dh, which turn their blocks into NaN blocks
    (scale byte 0xFF, codes 0x7F) on both sides."""
    counts, I = [128, 96], 128
    off, poff = offsets(counts)
    R = int(off[-1])
    gen = synth.generator(4242)
    a = synth.randn_bf16((R, 2 * I), gen, std=1.0).clone()
    dh = synth.randn_bf16((R, I), gen, std=1e-2).clone()
    big = torch.rand(32, 8, generator=gen) * 56.0 + 64.0
    sign = torch.where(torch.rand(32, 8, generator=gen) < 0.5, -1.0, 1.0)
    a[:32, :8] = (big * sign).to(torch.bfloat16)                    # |g| in [64, 120)
    a[140:150, 40] = -100.0                                         # e^-|g| subnormal, second expert
    nan, inf = float("nan"), float("inf")
    a[40, 5] = nan                                                  # gate NaN
    a[42, I + 70] = inf                                             # up +Inf
    a[43, 3] = -inf                                                 # gate -Inf: silu = NaN
    a[45, 100] = inf                                                # gate +Inf
    a[150, I + 17] = -inf                                           # up -Inf, second expert
    dh[44, 9] = inf                                                 # dh +Inf (backward only)
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
        else:
            mx.mxfp8_swiglu_quantize(a.to(dev), R, I, RC, offd, poffd, E, pb, q_row, sf_row, q_col, sf_col, err)
        check_dev_err(err)
        with np.errstate(invalid="ignore", over="ignore"):
            check_swiglu_outputs(bwd, bits(a), bits(dh), off, poff, q_row, sf_row, q_col, sf_col)
        q = q_row.cpu()
        # the NaN blocks: gate NaN at (40, 5) -> rowwise block 0 of row 40 all NaN codes
        assert bool((q[40, :32] == 0x7F).all())
