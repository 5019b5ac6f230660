"""Grouped GEMMs at full MoE sizes, in the launch configuration the benchmark uses, vs the
oracle on sampled outputs.

* Skewed small groups (T=4096 tokens, top-8 of E=128 experts with Zipf(1.2) popularity and
  four experts without tokens, hidden 4096, intermediate 1536): GEMM1 forward, its dgrad
  and its wgrad.  Empty experts must get exactly zero weight gradients.
* Backward of the T=16384, top-8 of 32 FFN (hidden 7168, intermediate 2048): dgrad and
  wgrad of the down projection.

A sampled output element needs only its own rows and columns of the operands: a rowwise
scale block depends on its row alone and a columnwise block on its column alone (within
the expert's segment), so the oracle quantizes just those slices, in fp64 GEMMs over the
dequantized codes.  Tolerance: max|gpu - oracle| <= 2e-2 x rms(oracle) per expert."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, ROW_B, TOL, bits, check_dev_err, dev, np_, rel_err  # noqa: F401

pytestmark = pytest.mark.gpu


def _pick(rng, lo, hi, n):
    """Sorted unique sample of [lo, hi) holding both ends."""
    if hi - lo <= n:
        return np.arange(lo, hi)
    return np.unique(np.concatenate([[lo, hi - 1], rng.integers(lo, hi, n)]))


def _rows(t, idx):
    return t[torch.from_numpy(np.asarray(idx, np.int64)).to(t.device)]


def _cols_of_rows(t, rows, cols):
    """t[rows][:, cols] as bf16 bits (rows, cols: index arrays or slices)."""
    sub = t[rows] if isinstance(rows, slice) else _rows(t, rows)
    return bits(sub[:, torch.from_numpy(np.asarray(cols, np.int64)).to(t.device)])


def _colwise_one_segment(b):
    """Columnwise codes/scales of a [rows x c] bf16-bits block taken as one expert segment."""
    n = b.shape[0]
    ld = (n + 127) // 128 * 128
    return oracle.quantize_colwise_seg(b, np.array([0, n], np.int32), np.array([0, ld], np.int32), ld)


def test_skewed_small_groups_fwd_dgrad_wgrad(dev):
    d = synth.skewed(device="cuda")
    T, E, k, H, I2 = d["T"], d["E"], d["k"], d["hidden"], 2 * d["inter"]
    R = T * k
    dH = synth.randn_bf16((R, I2), synth.generator(7001, "cuda"), std=1e-2, device="cuda")
    w1 = d["w1"].view(E * I2, H)
    err = mx.new_dev_err(dev)
    qx = mx.quantize_alloc(d["x"], mx.MX_ROWWISE, dev_err=err)
    pm = mx.permute_alloc(d["ids"], E, qx["q_row"], qx["sf_row"], dev_err=err)
    offd, poffd = pm["off"], pm["poff"]
    # forward: C = x_perm W1_e^T
    qw = mx.quantize_alloc(w1, ROW_B, dev_err=err)
    C = torch.empty(R, I2, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(pm["q"], pm["sf"], qw["q_row"], qw["sf_row"], offd, poffd, E, R, I2, H, C, err)
    # dgrad: dX = dH W1_e (contraction over the I2 rows of W1_e)
    qdh = mx.quantize_alloc(dH, mx.MX_ROWWISE | mx.MX_COLWISE, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * I2, I2, dtype=torch.int32, device=dev)
    qwc = mx.quantize_alloc(w1, COL_B, woff, woff, dev_err=err, ld_col=E * I2)
    dX = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_dgrad(qdh["q_row"], qdh["sf_row"], qwc["q_col"], qwc["sf_col"], offd, poffd, E, R, H, I2,
                                dX, err)
    # wgrad: dW1_e = dH_e^T x_perm_e (contraction over the expert's tokens)
    xp = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    mx.moe_gather_rows(d["x"], H * 2, pm["src_row"], R, xp)
    qxc = mx.quantize_alloc(xp, COL_B, offd, poffd, dev_err=err)
    assert qxc["ld_col"] == qdh["ld_col"]
    dW = torch.full((E, I2, H), float("nan"), dtype=torch.float32, device=dev)
    mx.grouped_gemm_mxfp8_wgrad(qdh["q_col"], qdh["sf_col"], qxc["q_col"], qxc["sf_col"], offd, poffd, E, I2, H,
                                qdh["ld_col"], dW, err)
    check_dev_err(err)

    off, src = np_(offd), np_(pm["src_row"])
    counts = np.diff(off)
    empty = np.nonzero(counts == 0)[0]
    assert len(empty) >= 3 and np.any(counts % 128 != 0)
    for e in empty:
        assert int(torch.count_nonzero(dW[e]).item()) == 0, "empty expert %d must get a zero gradient" % e
    xb = bits(d["x"])
    rng = np.random.default_rng(5)
    worst = {"fwd": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    for e in np.nonzero(counts)[0]:
        r0, r1 = int(off[e]), int(off[e + 1])
        rows = _pick(rng, r0, r1, 3)
        w1e = d["w1"][e]
        # forward
        cols = _pick(rng, 0, I2, 12)
        aq, asf = oracle.quantize_rowwise(xb[src[rows]])
        bq, bsf = oracle.quantize_rowwise(bits(_rows(w1e, cols)))
        got = _cols_of_rows(C, rows, cols)
        worst["fwd"] = max(worst["fwd"], rel_err((got.astype(np.uint32) << 16).view(np.float32).astype(np.float64),
                                                 oracle.gemm_nt(aq, asf, bq, bsf)))
        # dgrad
        jc = _pick(rng, 0, H, 12)
        aq, asf = oracle.quantize_rowwise(bits(_rows(dH, rows)))
        cq, csf = _colwise_one_segment(_cols_of_rows(w1e, slice(None), jc))
        got = _cols_of_rows(dX, rows, jc)
        worst["dgrad"] = max(worst["dgrad"], rel_err((got.astype(np.uint32) << 16).view(np.float32).astype(np.float64),
                                                     oracle.gemm_nt(aq, asf, cq, csf)))
        # wgrad
        ic, jc = _pick(rng, 0, I2, 6), _pick(rng, 0, H, 6)
        dq, dsf = _colwise_one_segment(_cols_of_rows(dH, slice(r0, r1), ic))
        xq, xsf = _colwise_one_segment(xb[src[r0:r1]][:, jc])
        got = dW[e][torch.from_numpy(ic).to(dev)][:, torch.from_numpy(jc).to(dev)].cpu().numpy().astype(np.float64)
        worst["wgrad"] = max(worst["wgrad"], rel_err(got, oracle.gemm_nt(dq, dsf, xq, xsf)))
    assert max(worst.values()) <= TOL, worst


def test_ffn_down_projection_backward_full_size(dev):
    d = synth.ffn(device="cuda")
    T, E, k, H, I = d["T"], d["E"], d["k"], d["hidden"], d["inter"]
    R = T * k
    dY = synth.ffn_bwd(device="cuda", R=R, hidden=H, inter=I)["dy"]     # expert-ordered down-projection grads
    h = d["h"]                                                          # expert-ordered down-projection input
    w2 = d["w2"].view(E * H, I)
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(d["ids"], E, dev_err=err)
    offd, poffd = pm["off"], pm["poff"]
    qdy = mx.quantize_alloc(dY, mx.MX_ROWWISE | mx.MX_COLWISE, offd, poffd, dev_err=err)
    woff = torch.arange(0, (E + 1) * H, H, dtype=torch.int32, device=dev)
    qwc = mx.quantize_alloc(w2, COL_B, woff, woff, dev_err=err, ld_col=E * H)
    dh = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_dgrad(qdy["q_row"], qdy["sf_row"], qwc["q_col"], qwc["sf_col"], offd, poffd, E, R, I, H,
                                dh, err)
    qhc = mx.quantize_alloc(h, COL_B, offd, poffd, dev_err=err)
    dW = torch.empty(E, H, I, dtype=torch.float32, device=dev)
    mx.grouped_gemm_mxfp8_wgrad(qdy["q_col"], qdy["sf_col"], qhc["q_col"], qhc["sf_col"], offd, poffd, E, H, I,
                                qdy["ld_col"], dW, err)
    check_dev_err(err)

    off = np_(offd)
    rng = np.random.default_rng(6)
    worst = {"dgrad": 0.0, "wgrad": 0.0}
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        assert r1 > r0
        w2e = d["w2"][e]
        rows, jc = _pick(rng, r0, r1, 3), _pick(rng, 0, I, 24)
        aq, asf = oracle.quantize_rowwise(bits(_rows(dY, rows)))
        cq, csf = _colwise_one_segment(_cols_of_rows(w2e, slice(None), jc))
        got = _cols_of_rows(dh, rows, jc)
        worst["dgrad"] = max(worst["dgrad"], rel_err((got.astype(np.uint32) << 16).view(np.float32).astype(np.float64),
                                                     oracle.gemm_nt(aq, asf, cq, csf)))
        ic, jc = _pick(rng, 0, H, 6), _pick(rng, 0, I, 6)
        dq, dsf = _colwise_one_segment(_cols_of_rows(dY, slice(r0, r1), ic))
        hq, hsf = _colwise_one_segment(_cols_of_rows(h, slice(r0, r1), jc))
        got = dW[e][torch.from_numpy(ic).to(dev)][:, torch.from_numpy(jc).to(dev)].cpu().numpy().astype(np.float64)
        worst["wgrad"] = max(worst["wgrad"], rel_err(got, oracle.gemm_nt(dq, dsf, hq, hsf)))
    assert max(worst.values()) <= TOL, worst
