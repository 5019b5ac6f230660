"""A whole MoE FFN layer step (forward + backward) on the GPU vs the oracle composed from
the same definitions: permute, quantize, fp64 GEMMs over the dequantized operands, combine.

The SwiGLU value that decides each E4M3 code of h and dH is an fp32 number on both sides,
but formed by different arithmetic (the kernel's fp32 special-function path, the oracle's
fp64 rounded once), so a value within a few fp32 ulps of an E4M3 rounding boundary may take
the neighbouring code (test_gpu_swiglu.py bounds how often).  One such code at a block
maximum moves a whole output row of the next GEMM by a step of up to 1/8 of that block's
largest value.  Every output downstream of those codes is therefore held, element by
element, to the per-stage bound plus the largest effect one E4M3 step of one of its
SwiGLU inputs can have (computed from the oracle's own operands), and, as a whole, to a
relative Frobenius error of TOL."""
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


def _deq(q, sf):
    """Dequantized MXFP8 values; sf holds one scale byte per 32 consecutive elements of a row."""
    v = oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape)
    return v * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=1))[:, : q.shape[1]]


def _step(q, sf):
    """One E4M3 step at each code (2^(e-3) for a normal magnitude 2^e.., 2^-9 below 2^-6), times its scale."""
    v = np.abs(oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape))
    st = np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3)
    return st * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=1))[:, : q.shape[1]]


def _close(got, ref, n, allow):
    """Per element: n x TOL x rms plus the one-step allowance; as a whole: relative Frobenius <= TOL."""
    rms = float(np.sqrt(np.mean(np.square(ref))))
    assert np.all(np.abs(got - ref) <= n * TOL * rms + allow), float(np.max(np.abs(got - ref) - allow) / rms)
    assert np.linalg.norm(got - ref) <= TOL * np.linalg.norm(ref)


@pytest.mark.parametrize("T,E,k,H,I", [(512, 4, 2, 256, 128), (384, 8, 3, 384, 256)])
def test_layer_step(dev, T, E, k, H, I):
    # every reference is built by the oracle from the layer's own inputs only.  An output that
    # lies n quantized GEMM stages downstream of the inputs is held to n x the per-GEMM bound
    # (each stage's own rounding adds up to TOL x rms, and the two sides re-quantize slightly
    # different upstream values); single-GEMM parity on identical operands is held to TOL in
    # test_gpu_gemm.py.
    g = synth.generator(900 + T)
    st = MoEFFNStep(T, E, k, H, I, device=dev)
    I2 = 2 * I
    logits = torch.randn(T, E, generator=g)
    ids = synth.topk_ids(logits, k)
    gate = torch.softmax(logits.gather(1, ids.long()), dim=1)
    x = synth.randn_bf16((T, H), g)
    w1 = synth.randn_bf16((E, I2, H), g, std=H ** -0.5)
    w2 = synth.randn_bf16((E, H, I), g, std=I ** -0.5)
    dout = synth.randn_bf16((T, H), g, std=1e-2)
    for name, t in (("x", x), ("ids", ids), ("gate", gate), ("w1", w1), ("w2", w2), ("dout", dout)):
        getattr(st, name).copy_(t.to(dev))
    st.step()
    check_dev_err(st.dev_err)

    p = oracle.permute(ids.numpy(), E)
    off, poff, src, dst = p["off"], p["poff"], p["src_row"], p["dst_of"]
    gn = gate.numpy()
    xb = bits(x)
    w1b, w2b = bits(w1).reshape(E * I2, H), bits(w2).reshape(E * H, I)
    R = T * k
    ld = st.pb

    def grouped(aq, asf, bq, bsf, n):                      # rows grouped by expert, B per expert [n x K]
        out = np.zeros((R, n))
        for e in range(E):
            r0, r1 = int(off[e]), int(off[e + 1])
            if r1 > r0:
                out[r0:r1] = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], bq[e * n:(e + 1) * n], bsf[e * n:(e + 1) * n])
        return out

    def bf(v):
        return oracle.to_bf16_bits(v).reshape(v.shape)

    # forward: gather + quantize x, GEMM1, SwiGLU -> fp32 h, quantize, GEMM2, combine
    xg = oracle.gather_rows(xb, src)
    aq, asf = oracle.quantize_rowwise(xg)
    w1q, w1sf = oracle.quantize_rowwise(w1b)
    a1 = bf(grouped(aq, asf, w1q, w1sf, I2))                  # GEMM1 output, bf16 bits
    assert rel_err(_val(bits(st.out1)), _val(a1)) <= TOL
    h32 = oracle.swiglu_fwd(a1)
    hq, hsf = oracle.quantize_rowwise_ex(h32)
    w2q, w2sf = oracle.quantize_rowwise(w2b)
    Yb = bf(grouped(hq, hsf, w2q, w2sf, H))
    expert_of = np.repeat(np.arange(E), np.diff(off))          # expert of each routed row
    w2max = np.abs(_deq(w2q, w2sf)).reshape(E, H, I).max(axis=2)  # [E x H]: max_i |W2[e][j, i]|
    a_out2 = _step(hq, hsf).max(axis=1)[:, None] * w2max[expert_of]
    _close(_val(bits(st.out2)), _val(Yb), 2, a_out2)
    out_ref = _val(oracle.combine_fwd(Yb, gn, dst))
    _close(_val(bits(st.out)), out_ref, 2, np.einsum("tj,tjh->th", gn.astype(np.float64), a_out2[dst]))
    # backward: combine backward, dgrad2, SwiGLU backward, dgrad1 + un-permute, both wgrads
    dYb, dgate_ref = oracle.combine_bwd(bits(dout), Yb, gn, dst)
    assert np.array_equal(bits(st.dy), dYb)       # gate * dOut: independent of Y, exact
    a_dgate = np.einsum("th,tjh->tj", np.abs(_val(bits(dout))), a_out2[dst])
    _close(np_(st.dgate).astype(np.float64), dgate_ref, 2, a_dgate)
    dyq, dysf = oracle.quantize_rowwise(dYb)
    seg2 = np.arange(0, (E + 1) * H, H, dtype=np.int32)
    w2c, w2csf = oracle.quantize_colwise_seg(w2b, seg2, seg2, E * H)
    dh_in = np.zeros((R, I))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            dh_in[r0:r1] = oracle.gemm_nt(dyq[r0:r1], dysf[r0:r1], w2c[:, e * H:(e + 1) * H],
                                          w2csf[:, e * H // 32:(e + 1) * H // 32])
    dh_b = bf(dh_in)
    assert rel_err(_val(bits(st.dh_in)), _val(dh_b)) <= TOL
    dH32 = oracle.swiglu_bwd(dh_b, a1)
    dhq, dhsf = oracle.quantize_rowwise_ex(dH32)
    seg1 = np.arange(0, (E + 1) * I2, I2, dtype=np.int32)
    w1c, w1csf = oracle.quantize_colwise_seg(w1b, seg1, seg1, E * I2)
    dXr = np.zeros((R, H))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            dXr[r0:r1] = oracle.gemm_nt(dhq[r0:r1], dhsf[r0:r1], w1c[:, e * I2:(e + 1) * I2],
                                        w1csf[:, e * I2 // 32:(e + 1) * I2 // 32])
    dx_ref = _val(oracle.combine_fwd(bf(dXr), np.ones((T, k), np.float32), dst))
    w1max = np.abs(_deq(w1c, w1csf)).reshape(H, E, I2).max(axis=2).T    # [E x H]: max_i |W1[e][i, j]|
    a_dxr = _step(dhq, dhsf).max(axis=1)[:, None] * w1max[expert_of]
    _close(_val(bits(st.dx)), dx_ref, 3, a_dxr[dst].sum(axis=1))
    dyc, dycsf = oracle.quantize_colwise_seg(dYb, off, poff, ld)
    hc, hcsf = oracle.quantize_colwise_seg_ex(h32, off, poff, ld)
    dhc, dhcsf = oracle.quantize_colwise_seg_ex(dH32, off, poff, ld)
    xc, xcsf = oracle.quantize_colwise_seg(xg, off, poff, ld)
    for e in range(E):
        p0, p1 = int(poff[e]), int(poff[e + 1])
        if p1 == p0:
            assert np.all(np_(st.dw2[e]) == 0) and np.all(np_(st.dw1[e]) == 0)
            continue
        s0, s1 = p0 // 32, p1 // 32
        dw2 = oracle.gemm_nt(dyc[:, p0:p1], dycsf[:, s0:s1], hc[:, p0:p1], hcsf[:, s0:s1])
        dw1 = oracle.gemm_nt(dhc[:, p0:p1], dhcsf[:, s0:s1], xc[:, p0:p1], xcsf[:, s0:s1])
        a_dw2 = np.abs(_deq(dyc[:, p0:p1], dycsf[:, s0:s1])).max(axis=1)[:, None] * \
            _step(hc[:, p0:p1], hcsf[:, s0:s1]).max(axis=1)[None, :]
        a_dw1 = _step(dhc[:, p0:p1], dhcsf[:, s0:s1]).max(axis=1)[:, None] * \
            np.abs(_deq(xc[:, p0:p1], xcsf[:, s0:s1])).max(axis=1)[None, :]
        _close(np_(st.dw2[e]).astype(np.float64), dw2, 2, a_dw2)
        _close(np_(st.dw1[e]).astype(np.float64), dw1, 3, a_dw1)
