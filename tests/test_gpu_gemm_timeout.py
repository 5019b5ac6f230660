"""The grouped GEMM's failure detector: every pipeline wait in the kernel is bounded, and a
wait that runs out sets MX_DEVERR_TIMEOUT, makes every role of the kernel leave and frees
the tensor memory, so the context stays usable.

The internal test entry withholds every operand copy, so the "stage full" barrier the MMA
issuer waits on is never armed, and sets a short wait limit (1 ms instead of 2 s).  Nothing
here can hang the GPU: every wait in the kernel is bounded by that limit (or by a fixed
limit for the final drains, which have nothing outstanding here).  After the failed call, a
normal call on the same stream must still return correct results."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import COL_B, ROW_B, TOL, bits, check_dev_err, dev, offsets, rel_err  # noqa: F401

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000   # 1 ms


@pytest.mark.parametrize("ctas", [2, 1])
@pytest.mark.parametrize("pass_", ["fwd", "wgrad"])
def test_withheld_operands_time_out_and_the_context_survives(dev, ctas, pass_):
    counts, N, K = [300, 0, 129, 77], 256, 384
    E = len(counts)
    off, poff = offsets(counts)
    R = int(off[-1])
    g = synth.generator(77 + ctas)
    xp = synth.randn_bf16((R, K), g)
    w = synth.randn_bf16((E * N, K), g)
    dy = synth.randn_bf16((R, N), g, std=1e-2)
    offd, poffd = torch.from_numpy(off).to(dev), torch.from_numpy(poff).to(dev)
    err0 = mx.new_dev_err(dev)
    if pass_ == "fwd":
        qa = mx.quantize_alloc(xp.to(dev), mx.MX_ROWWISE, offd, poffd, dev_err=err0)
        qb = mx.quantize_alloc(w.to(dev), ROW_B, dev_err=err0)
        args = (mx.MX_TESTING_FWD, qa["q_row"], qa["sf_row"], qb["q_row"], qb["sf_row"], offd, poffd, E, R, N, K, 0)
        out = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=dev)
    else:
        qd = mx.quantize_alloc(dy.to(dev), mx.MX_COLWISE, offd, poffd, dev_err=err0)
        qx = mx.quantize_alloc(xp.to(dev), COL_B, offd, poffd, dev_err=err0)
        args = (mx.MX_TESTING_WGRAD, qd["q_col"], qd["sf_col"], qx["q_col"], qx["sf_col"], offd, poffd, E, 0, N, K,
                qd["ld_col"])
        out = torch.full((E, N, K), float("nan"), dtype=torch.float32, device=dev)
    check_dev_err(err0)

    # 1. the failing call: returns MX_OK (the failure is asynchronous), then reports the timeout
    err = mx.new_dev_err(dev)
    st = mx.testing_grouped_gemm(*args, out, err, ctas_per_mma=ctas, wait_limit_ns=LIMIT_NS, withhold_operands=True)
    assert st == 0
    torch.cuda.synchronize()
    bitsv = int(err.item())
    assert bitsv & mx.MX_DEVERR_TIMEOUT, "no timeout reported (dev_err = %d)" % bitsv

    # 2. the same call without the withheld operands, on the same stream: correct results
    err2 = mx.new_dev_err(dev)
    assert mx.testing_grouped_gemm(*args, out, err2, ctas_per_mma=ctas) == 0
    check_dev_err(err2)
    got = out.float().cpu().numpy().astype(np.float64)
    if pass_ == "fwd":
        oq, osf = oracle.quantize_rowwise(bits(xp))
        wq, wsf = oracle.quantize_rowwise(bits(w))
        for e in range(E):
            r0, r1 = int(off[e]), int(off[e + 1])
            if r1 > r0:
                ref = oracle.gemm_nt(oq[r0:r1], osf[r0:r1], wq[e * N:(e + 1) * N], wsf[e * N:(e + 1) * N])
                assert rel_err(got[r0:r1], ref) <= TOL
    else:
        ld = args[-1]
        dq, dsf = oracle.quantize_colwise_seg(bits(dy), off, poff, ld)
        xq, xsf = oracle.quantize_colwise_seg(bits(xp), off, poff, ld)
        for e in range(E):
            p0, p1 = int(poff[e]), int(poff[e + 1])
            if p1 == p0:
                assert np.all(got[e] == 0.0)
                continue
            ref = oracle.gemm_nt(dq[:, p0:p1], dsf[:, p0 // 32:p1 // 32], xq[:, p0:p1], xsf[:, p0 // 32:p1 // 32])
            assert rel_err(got[e], ref) <= TOL


def test_testing_entry_rejects_bad_options(dev):
    z = torch.zeros(64, dtype=torch.uint8, device=dev)
    o = torch.tensor([0, 128], dtype=torch.int32, device=dev)
    err = mx.new_dev_err(dev)
    out = torch.empty(128, 128, dtype=torch.bfloat16, device=dev)
    assert mx.testing_grouped_gemm(3, z, z, z, z, o, o, 1, 128, 128, 128, 0, out, err) == -1       # unknown pass
    assert mx.testing_grouped_gemm(0, z, z, z, z, o, o, 1, 128, 128, 128, 0, out, err, ctas_per_mma=3) == -1
    assert mx.testing_grouped_gemm(0, z, z, z, z, o, o, 1, 128, 128, 128, 0, out, err, flags=4) == -1
