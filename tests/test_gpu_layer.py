"""A whole MoE FFN layer step (forward + backward) on the GPU vs the oracle composed from
the same definitions: permute, quantize, fp64 GEMMs over the dequantized operands, combine."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import synth
from mxfp8_block_scaled_rowwise_gb300.layer import MoEFFNStep
from gpu_util import TOL, bits, check_dev_err, dev, np_, rel_err  # noqa: F401

pytestmark = pytest.mark.gpu


def _val(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_round(v):
    return _val(oracle.to_bf16_bits(v).reshape(v.shape))


@pytest.mark.parametrize("T,E,k,H,I", [(512, 4, 2, 256, 128), (384, 8, 3, 384, 256)])
def test_layer_step(dev, T, E, k, H, I):
    g = synth.generator(900 + T)
    st = MoEFFNStep(T, E, k, H, I, device=dev)
    I2 = 2 * I
    logits = torch.randn(T, E, generator=g)
    ids = synth.topk_ids(logits, k)
    gate = torch.softmax(logits.gather(1, ids.long()), dim=1)
    x = synth.randn_bf16((T, H), g)
    w1 = synth.randn_bf16((E, I2, H), g)
    w2 = synth.randn_bf16((E, H, I), g)
    h = synth.randn_bf16((T * k, I), g)
    dout = synth.randn_bf16((T, H), g, std=1e-2)
    dh = synth.randn_bf16((T * k, I2), g, std=1e-2)
    for name, t in (("x", x), ("ids", ids), ("gate", gate), ("w1", w1), ("w2", w2), ("h", h), ("dout", dout),
                    ("dh", dh)):
        getattr(st, name).copy_(t.to(dev))
    st.step()
    check_dev_err(st.dev_err)

    p = oracle.permute(ids.numpy(), E)
    off, poff, src, dst = p["off"], p["poff"], p["src_row"], p["dst_of"]
    gn = gate.numpy()
    xb, hb, dhb = bits(x), bits(h), bits(dh)
    w1b, w2b = bits(w1).reshape(E * I2, H), bits(w2).reshape(E * H, I)
    # forward: GEMM1 (not part of out here: h stands in for SwiGLU), GEMM2, combine
    hq, hsf = oracle.quantize_rowwise(hb)
    w2q, w2sf = oracle.quantize_rowwise(w2b)
    Y = np.zeros((T * k, H))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            Y[r0:r1] = oracle.gemm_nt(hq[r0:r1], hsf[r0:r1], w2q[e * H:(e + 1) * H], w2sf[e * H:(e + 1) * H])
    Yb = oracle.to_bf16_bits(Y).reshape(Y.shape)
    out_ref = _val(oracle.combine_fwd(Yb, gn, dst))
    assert rel_err(_val(bits(st.out)), out_ref) <= TOL
    # GEMM1 output
    xg = oracle.gather_rows(xb, src)
    aq, asf = oracle.quantize_rowwise(xg)
    w1q, w1sf = oracle.quantize_rowwise(w1b)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            ref = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], w1q[e * I2:(e + 1) * I2], w1sf[e * I2:(e + 1) * I2])
            assert rel_err(_val(bits(st.out1[r0:r1])), ref) <= TOL
    # backward: combine backward (dY bit-exact: it does not depend on Y), dgate, wgrad2, dgrad1, wgrad1
    dYb, dgate_ref = oracle.combine_bwd(bits(dout), Yb, gn, dst)
    assert np.array_equal(bits(st.dy), dYb)
    assert rel_err(np_(st.dgate).astype(np.float64), dgate_ref) <= TOL
    ld = st.pb
    dyc, dycsf = oracle.quantize_colwise_seg(dYb, off, poff, ld)
    hc, hcsf = oracle.quantize_colwise_seg(hb, off, poff, ld)
    dhq, dhsf = oracle.quantize_rowwise(dhb)
    seg = np.arange(0, (E + 1) * I2, I2, dtype=np.int32)
    w1c, w1csf = oracle.quantize_colwise_seg(w1b, seg, seg, E * I2)
    dhc, dhcsf = oracle.quantize_colwise_seg(dhb, off, poff, ld)
    xc, xcsf = oracle.quantize_colwise_seg(xg, off, poff, ld)
    dXr = np.zeros((T * k, H))
    for e in range(E):
        p0, p1 = int(poff[e]), int(poff[e + 1])
        r0, r1 = int(off[e]), int(off[e + 1])
        dw2 = oracle.gemm_nt(dyc[:, p0:p1], dycsf[:, p0 // 32:p1 // 32], hc[:, p0:p1], hcsf[:, p0 // 32:p1 // 32])
        dw1 = oracle.gemm_nt(dhc[:, p0:p1], dhcsf[:, p0 // 32:p1 // 32], xc[:, p0:p1], xcsf[:, p0 // 32:p1 // 32])
        if p1 == p0:
            assert np.all(np_(st.dw2[e]) == 0) and np.all(np_(st.dw1[e]) == 0)
            continue
        assert rel_err(np_(st.dw2[e]).astype(np.float64), dw2) <= TOL
        assert rel_err(np_(st.dw1[e]).astype(np.float64), dw1) <= TOL
        dXr[r0:r1] = oracle.gemm_nt(dhq[r0:r1], dhsf[r0:r1], w1c[:, e * I2:(e + 1) * I2],
                                    w1csf[:, e * I2 // 32:(e + 1) * I2 // 32])
    dx_ref = _val(oracle.combine_fwd(oracle.to_bf16_bits(dXr).reshape(dXr.shape), np.ones((T, k), np.float32), dst))
    assert rel_err(_val(bits(st.dx)), dx_ref) <= TOL
