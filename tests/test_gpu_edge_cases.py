"""Degenerate and limit cases of the grouped GEMMs and quantizers against the oracle:
the largest expert count (E = 1024, most experts without tokens), every routed row in a single
expert, a single-token expert, and calls with nothing to do.  Both tile shapes (CTA pairs and
single CTAs) are exercised through the internal test entry."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, ROW_B, TOL, bits, check_dev_err, dev, np_, offsets, rel_err  # noqa: F401

pytestmark = pytest.mark.gpu


def _check_all_passes(dev, counts, N, K, ctas, seed):
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(seed)
    xp, w, dy = synth.randn_bf16((R, K), g), synth.randn_bf16((E * N, K), g), synth.randn_bf16((R, N), g, std=1e-2)
    err = mx.new_dev_err(dev)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err)
    qb = mx.quantize_alloc(w.to(dev), ROW_B, dev_err=err)
    C = torch.full((max(R, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    assert mx.testing_grouped_gemm(mx.MX_TESTING_FWD, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd,
                                   poffd, E, R, N, K, 0, C, err, ctas_per_mma=ctas) == 0
    qd = mx.quantize_alloc(dy.to(dev), mx.MX_COLWISE, offd, poffd, dev_err=err)
    qx = mx.quantize_alloc(xp.to(dev), COL_B, offd, poffd, dev_err=err)
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    assert mx.testing_grouped_gemm(mx.MX_TESTING_WGRAD, qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd,
                                   poffd, E, 0, N, K, qd["ld_col"], dW, err, ctas_per_mma=ctas) == 0
    check_dev_err(err)
    got, gdw = C.float().cpu().numpy().astype(np.float64), dW.cpu().numpy()
    oq, osf = oracle.quantize_rowwise(bits(xp))
    wq, wsf = oracle.quantize_rowwise(bits(w))
    ld = qd["ld_col"]
    dq, dsf = oracle.quantize_colwise_seg(bits(dy), off, poff, ld)
    xq, xsf = oracle.quantize_colwise_seg(bits(xp), off, poff, ld)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        p0, p1 = int(poff[e]), int(poff[e + 1])
        if r1 == r0:
            assert np.all(gdw[e] == 0.0), "expert %d without tokens must get a zero gradient" % e
            continue
        ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N])
        assert rel_err(got[r0:r1], ref) <= TOL, "fwd expert %d" % e
        ref = oracle.gemm_nt(dq[:, p0:p1], dsf[:, p0 // 32:p1 // 32], xq[:, p0:p1], xsf[:, p0 // 32:p1 // 32])
        assert rel_err(gdw[e].astype(np.float64), ref) <= TOL, "wgrad expert %d" % e


@pytest.mark.parametrize("ctas", [2, 1])
def test_largest_expert_count_mostly_empty(dev, ctas):
    # E = 1024 (the limit): 1000 experts without tokens, the rest 1..300 rows
    rng = np.random.default_rng(3)
    counts = np.zeros(1024, np.int64)
    busy = rng.choice(1024, 24, replace=False)
    counts[busy] = rng.integers(1, 300, 24)
    _check_all_passes(dev, counts.tolist(), 128, 128, ctas, 11)


@pytest.mark.parametrize("ctas", [2, 1])
def test_all_rows_in_one_expert(dev, ctas):
    # every routed row in expert 5 of 8 (a dense GEMM inside a grouped call), plus a
    # single-token expert next to it
    counts = [0, 0, 0, 0, 0, 1000, 1, 0]
    _check_all_passes(dev, counts, 256, 256, ctas, 12)


def test_calls_with_nothing_to_do(dev):
    # zero rows: the calls succeed and write nothing
    err = mx.new_dev_err(dev)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    q = torch.full((16,), 7, dtype=torch.uint8, device=dev)
    mx.mxfp8_quantize(x, 0, 64, mx.MX_ROWWISE, None, None, 0, 0, q, q, None, None, err)
    off = torch.zeros(3, dtype=torch.int32, device=dev)
    C = torch.full((1, 128), 3.0, dtype=torch.bfloat16, device=dev)
    mx.grouped_gemm_mxfp8_fwd(q, q, q, q, off, off, 2, 0, 128, 128, C, err)
    check_dev_err(err)
    assert torch.all(q == 7) and torch.all(C == 3.0)
