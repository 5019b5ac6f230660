"""The quantizers at full size, every output byte against the oracle.

* The 16384 x 7168 quantizer workload (log-normal row magnitudes, 0.1 % outliers at 1000x):
  rowwise, columnwise and both from one read, the whole tensor bit for bit; the same values
  as fp32 input (both forms, floor and ceiling scale rules).
* Quantize-on-gather on the MoE FFN routing (16384 tokens, top-8 of 32 experts, hidden 7168:
  131072 gathered rows): rowwise and columnwise codes and scales of every expert bit for bit.

The oracle is plain single-threaded C; these tests run independent oracle calls (row blocks,
experts) on a thread pool, since the C calls do not hold the Python lock."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, bits, check_dev_err, dev, np_, sf_x4_first  # noqa: F401

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


def _pool_map(fn, items):
    with ThreadPoolExecutor(THREADS) as ex:
        return list(ex.map(fn, items))


@pytest.mark.parametrize("mode", [mx.MX_ROWWISE, mx.MX_COLWISE, mx.MX_ROWWISE | mx.MX_COLWISE])
def test_quantizer_workload_whole_tensor(dev, mode):
    d = synth.quant(device="cuda")
    x = d["x"]
    rows, cols = x.shape
    out = mx.quantize_alloc(x, mode)
    torch.cuda.synchronize()
    xb = bits(x)
    kb = cols // 32
    if mode & mx.MX_ROWWISE:
        q = np_(out["q_row"])
        sf = oracle.sf_from_tcgen05(np_(out["sf_row"]), rows, kb)
        step = 1024

        def rowblock(r0):
            oq, osf = oracle.quantize_rowwise(xb[r0:r0 + step])
            return np.array_equal(q[r0:r0 + step], oq) and np.array_equal(sf[r0:r0 + step], osf)
        ok = _pool_map(rowblock, range(0, rows, step))
        assert all(ok), "rowwise row blocks differing from the oracle: %s" % [i for i, v in enumerate(ok) if not v]
    if mode & mx.MX_COLWISE:
        q = np_(out["q_col"])
        sf = oracle.sf_from_tcgen05(np_(out["sf_col"]), cols, rows // 32)
        step = 256

        def colblock(c0):
            sub = np.ascontiguousarray(xb[:, c0:c0 + step])
            cq, csf = oracle.quantize_colwise_seg(sub, [0, rows], [0, rows], rows)
            return np.array_equal(q[c0:c0 + step], cq) and np.array_equal(sf[c0:c0 + step], csf)
        ok = _pool_map(colblock, range(0, cols, step))
        assert all(ok), "columnwise blocks differing from the oracle: %s" % [i for i, v in enumerate(ok) if not v]


@pytest.mark.parametrize("rule", [oracle.RULE_FLOOR, oracle.RULE_RCEIL])
def test_quantizer_workload_fp32_whole_tensor(dev, rule):
    # the same 16384 x 7168 values as fp32 input (the pages' microbenchmark input type; the
    # fp32 kernel's full-tile path on every tile), both forms from one read, with a few values
    # below bf16 precision so that the fp32 bits matter
    d = synth.quant(device="cuda")
    x = d["x"].float()
    x[::97, ::89] *= 1.0 + 2.0 ** -12
    rows, cols = x.shape
    out = mx.quantize_alloc(x, mx.MX_ROWWISE | mx.MX_COLWISE,
                            scale_rule=mx.MX_SCALE_FLOOR if rule == oracle.RULE_FLOOR else mx.MX_SCALE_RCEIL)
    torch.cuda.synchronize()
    xh = x.cpu().numpy()
    q = np_(out["q_row"])
    sf = oracle.sf_from_tcgen05(np_(out["sf_row"]), rows, cols // 32)
    step = 1024

    def rowblock(r0):
        oq, osf = oracle.quantize_rowwise_ex(np.ascontiguousarray(xh[r0:r0 + step]), rule)
        return np.array_equal(q[r0:r0 + step], oq) and np.array_equal(sf[r0:r0 + step], osf)
    ok = _pool_map(rowblock, range(0, rows, step))
    assert all(ok), "rowwise row blocks differing from the oracle: %s" % [i for i, v in enumerate(ok) if not v]
    qc = np_(out["q_col"])
    ld = out["ld_col"]
    sfc = oracle.sf_from_tcgen05(np_(out["sf_col"]), cols, ld // 32)
    step = 256

    def colblock(c0):
        sub = np.ascontiguousarray(xh[:, c0:c0 + step])
        cq, csf = oracle.quantize_colwise_seg_ex(sub, [0, rows], [0, rows], rows, rule)
        return np.array_equal(qc[c0:c0 + step, :rows], cq) and np.array_equal(sfc[c0:c0 + step, : rows // 32], csf)
    ok = _pool_map(colblock, range(0, cols, step))
    assert all(ok), "columnwise blocks differing from the oracle: %s" % [i for i, v in enumerate(ok) if not v]


def test_gather_quantize_ffn_routing_every_byte(dev):
    # the layer's quantize-on-gather call (rowwise GEMM1 operand, columnwise wgrad1 operand in
    # the four-copy scale layout) on the full MoE FFN routing
    d = synth.ffn(device="cuda", with_weights=False)
    T, E, k, H = d["T"], d["E"], d["k"], d["hidden"]
    R = T * k
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(d["ids"], E, dev_err=err)
    pb = mx.mx_padded_rows_bound(R, E)
    q_row = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sf_row = torch.empty(mx.mx_sf_bytes(pb, H // 32), dtype=torch.uint8, device=dev)
    q_col = torch.empty(H, pb, dtype=torch.uint8, device=dev)
    sf_col = torch.empty(mx.mx_sf_bytes_x4(H, pb // 32), dtype=torch.uint8, device=dev)
    mx.mxfp8_gather_quantize(d["x"], T, H, mx.MX_ROWWISE | COL_B, pm["src_row"], pm["off"], pm["poff"], E, R, pb,
                             q_row, sf_row, q_col, sf_col, err)
    check_dev_err(err)
    p = oracle.permute(d["ids"].cpu().numpy(), E)
    for key in ("off", "poff"):
        assert np.array_equal(np_(pm[key]), p[key])
    off, poff, src = p["off"], p["poff"], p["src_row"]
    xb = bits(d["x"])
    gq, gcq = np_(q_row), np_(q_col)
    P = int(poff[-1])
    gsf = oracle.sf_from_tcgen05(np_(sf_row), P, H // 32)
    gcsf = oracle.sf_from_tcgen05(sf_x4_first(sf_col, pb // 128, P // 128), H, pb // 32)

    def expert(e):
        r0, r1 = int(off[e]), int(off[e + 1])
        p0, p1 = int(poff[e]), int(poff[e + 1])
        xg = oracle.gather_rows(xb, src[r0:r1])
        oq, osf = oracle.quantize_rowwise(xg)
        ok = np.array_equal(gq[r0:r1], oq) and np.array_equal(gsf[p0:p0 + (r1 - r0)], osf)
        ok &= bool(np.all(gsf[p0 + (r1 - r0):p1] == 0))                   # padding scale rows
        cq, csf = oracle.quantize_colwise_seg(xg, [0, r1 - r0], [0, p1 - p0], p1 - p0)
        ok &= np.array_equal(gcq[:, p0:p1], cq) and np.array_equal(gcsf[:, p0 // 32:p1 // 32], csf)
        return ok
    ok = _pool_map(expert, range(E))
    assert all(ok), "experts differing from the oracle: %s" % [e for e, v in enumerate(ok) if not v]
