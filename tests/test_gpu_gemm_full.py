"""Grouped GEMMs at full MoE sizes, in the launch configuration the benchmark uses, vs the
oracle on sampled outputs.

* Skewed small groups (T=4096 tokens, top-8 of E=128 experts with Zipf(1.2) popularity and
  four experts without tokens, hidden 4096, intermediate 1536): GEMM1 forward, its dgrad
  and its wgrad.  Empty experts must get exactly zero weight gradients.
* All six GEMMs of the T=16384, top-8 of 32 FFN (hidden 7168, intermediate 2048): both
  forward GEMMs, both dgrads and both wgrads; per expert the first 2, the last 2 and 28
  seeded random output rows, over the full output width.

A sampled output element needs only its own rows and columns of the operands: a rowwise
scale block depends on its row alone and a columnwise block on its column alone (within
the expert's segment), so the oracle quantizes just those slices, in fp64 GEMMs over the
dequantized codes.  Tolerance: max|gpu - oracle| <= 2e-2 x rms(oracle) per expert."""
import os
from concurrent.futures import ThreadPoolExecutor

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


def _sample_rows(rng, lo, hi, n_rand=28):
    """The first 2, the last 2 and n_rand seeded random rows of [lo, hi) (sorted, unique)."""
    if hi - lo <= 4 + n_rand:
        return np.arange(lo, hi)
    return np.unique(np.concatenate([[lo, lo + 1, hi - 2, hi - 1], rng.integers(lo, hi, n_rand)]))


def _bf16_vals(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_ffn_six_gemms_full_size_sampled(dev):
    """All six grouped GEMMs of the MoE FFN layer (T=16384, top-8 of E=32, hidden 7168,
    intermediate 2048) at full size, launched as the benchmark launches them, each on its own
    seeded bf16 inputs.  Per expert the first 2, the last 2 and 28 seeded random output rows
    are checked over their full width against the oracle's fp64 GEMM of its own quantization
    (per expert: max|gpu - oracle| <= 2e-2 x rms(oracle))."""
    d = synth.ffn(device="cuda")
    bw = synth.ffn_bwd(device="cuda")
    T, E, k, H, I = d["T"], d["E"], d["k"], d["hidden"], d["inter"]
    I2, R = 2 * I, T * k
    err = mx.new_dev_err(dev)
    RC = mx.MX_ROWWISE | mx.MX_COLWISE
    pm = mx.permute_alloc(d["ids"], E, dev_err=err)
    offd, poffd = pm["off"], pm["poff"]
    pb = mx.mx_padded_rows_bound(R, E)
    # operands exactly as the layer quantizes them (B operands' scales in the four-copy layout)
    a1 = dict(q_row=torch.empty(R, H, dtype=torch.uint8, device=dev),
              sf_row=torch.empty(mx.mx_sf_bytes(pb, H // 32), dtype=torch.uint8, device=dev),
              q_col=torch.empty(H, pb, dtype=torch.uint8, device=dev),
              sf_col=torch.empty(mx.mx_sf_bytes_x4(H, pb // 32), dtype=torch.uint8, device=dev))
    mx.mxfp8_gather_quantize(d["x"], T, H, mx.MX_ROWWISE | COL_B, pm["src_row"], offd, poffd, E, R, pb,
                             a1["q_row"], a1["sf_row"], a1["q_col"], a1["sf_col"], err)
    w1seg = torch.arange(0, (E + 1) * I2, I2, dtype=torch.int32, device=dev)
    w2seg = torch.arange(0, (E + 1) * H, H, dtype=torch.int32, device=dev)
    qw1 = mx.quantize_alloc(d["w1"].view(E * I2, H), ROW_B | COL_B, w1seg, w1seg, dev_err=err, ld_col=E * I2)
    qw2 = mx.quantize_alloc(d["w2"].view(E * H, I), ROW_B | COL_B, w2seg, w2seg, dev_err=err, ld_col=E * H)
    qh = mx.quantize_alloc(d["h"], mx.MX_ROWWISE | COL_B, offd, poffd, dev_err=err)
    qdy = mx.quantize_alloc(bw["dy"], RC, offd, poffd, dev_err=err)
    qdh = mx.quantize_alloc(bw["dh"], RC, offd, poffd, dev_err=err)
    out = {}
    out["fwd1"] = torch.empty(R, I2, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(a1["q_row"], a1["sf_row"], qw1["q_row"], qw1["sf_row"], offd, poffd, E, R, I2, H,
                              out["fwd1"], err)
    out["fwd2"] = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(qh["q_row"], qh["sf_row"], qw2["q_row"], qw2["sf_row"], offd, poffd, E, R, H, I,
                              out["fwd2"], err)
    out["dgrad2"] = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_dgrad(qdy["q_row"], qdy["sf_row"], qw2["q_col"], qw2["sf_col"], offd, poffd, E, R, I, H,
                                out["dgrad2"], err)
    out["wgrad2"] = torch.empty(E, H, I, dtype=torch.float32, device=dev)
    mx.grouped_gemm_mxfp8_wgrad(qdy["q_col"], qdy["sf_col"], qh["q_col"], qh["sf_col"], offd, poffd, E, H, I, pb,
                                out["wgrad2"], err)
    out["dgrad1"] = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_dgrad(qdh["q_row"], qdh["sf_row"], qw1["q_col"], qw1["sf_col"], offd, poffd, E, R, H, I2,
                                out["dgrad1"], err)
    out["wgrad1"] = torch.empty(E, I2, H, dtype=torch.float32, device=dev)
    mx.grouped_gemm_mxfp8_wgrad(qdh["q_col"], qdh["sf_col"], a1["q_col"], a1["sf_col"], offd, poffd, E, I2, H, pb,
                                out["wgrad1"], err)
    check_dev_err(err)

    p = oracle.permute(d["ids"].cpu().numpy(), E)
    off, src = p["off"], p["src_row"]
    assert np.array_equal(np_(offd), off)
    rng = np.random.default_rng(2024)
    rows = {e: _sample_rows(rng, int(off[e]), int(off[e + 1])) for e in range(E)}
    wrows2 = {e: _sample_rows(rng, 0, H) for e in range(E)}          # dW2[e] rows (of H)
    wrows1 = {e: _sample_rows(rng, 0, I2) for e in range(E)}         # dW1[e] rows (of 2I)
    # the sampled rows of every output, brought to the host once
    got = {}
    for name in ("fwd1", "fwd2", "dgrad2", "dgrad1"):
        idx = torch.from_numpy(np.concatenate([rows[e] for e in range(E)])).to(dev)
        got[name] = _bf16_vals(bits(out[name][idx]))
    got["wgrad2"] = np.concatenate([np_(out["wgrad2"][e][torch.from_numpy(wrows2[e]).to(dev)]) for e in range(E)])
    got["wgrad1"] = np.concatenate([np_(out["wgrad1"][e][torch.from_numpy(wrows1[e]).to(dev)]) for e in range(E)])
    starts = np.concatenate([[0], np.cumsum([len(rows[e]) for e in range(E)])])
    wst2 = np.concatenate([[0], np.cumsum([len(wrows2[e]) for e in range(E)])])
    wst1 = np.concatenate([[0], np.cumsum([len(wrows1[e]) for e in range(E)])])
    xb, hb, dyb, dhb = bits(d["x"]), bits(d["h"]), bits(bw["dy"]), bits(bw["dh"])
    w1b, w2b = bits(d["w1"]), bits(d["w2"])

    def expert(e):
        r0, r1 = int(off[e]), int(off[e + 1])
        rr = rows[e]
        sl = slice(starts[e], starts[e + 1])
        res = {}
        aq, asf = oracle.quantize_rowwise(xb[src[rr]])
        bq, bsf = oracle.quantize_rowwise(w1b[e])
        res["fwd1"] = rel_err(got["fwd1"][sl], oracle.gemm_nt(aq, asf, bq, bsf))
        aq, asf = oracle.quantize_rowwise(hb[rr])
        bq, bsf = oracle.quantize_rowwise(w2b[e])
        res["fwd2"] = rel_err(got["fwd2"][sl], oracle.gemm_nt(aq, asf, bq, bsf))
        aq, asf = oracle.quantize_rowwise(dyb[rr])
        cq, csf = _colwise_one_segment(w2b[e])                   # W2_e [H x I] -> [I x H] over H
        res["dgrad2"] = rel_err(got["dgrad2"][sl], oracle.gemm_nt(aq, asf, cq, csf))
        aq, asf = oracle.quantize_rowwise(dhb[rr])
        cq, csf = _colwise_one_segment(w1b[e])                   # W1_e [2I x H] -> [H x 2I] over 2I
        res["dgrad1"] = rel_err(got["dgrad1"][sl], oracle.gemm_nt(aq, asf, cq, csf))
        dq, dsf = _colwise_one_segment(np.ascontiguousarray(dyb[r0:r1][:, wrows2[e]]))
        hq, hsf = _colwise_one_segment(hb[r0:r1])
        res["wgrad2"] = rel_err(got["wgrad2"][wst2[e]:wst2[e + 1]], oracle.gemm_nt(dq, dsf, hq, hsf))
        dq, dsf = _colwise_one_segment(np.ascontiguousarray(dhb[r0:r1][:, wrows1[e]]))
        xq, xsf = _colwise_one_segment(xb[src[r0:r1]])
        res["wgrad1"] = rel_err(got["wgrad1"][wst1[e]:wst1[e + 1]], oracle.gemm_nt(dq, dsf, xq, xsf))
        return res
    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        per_expert = list(ex.map(expert, range(E)))
    worst = {name: max(r[name] for r in per_expert) for name in per_expert[0]}
    print("six GEMMs, worst per-expert max|gpu - oracle| / rms(oracle):", worst)
    assert max(worst.values()) <= TOL, worst
