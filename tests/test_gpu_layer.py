"""A whole MoE FFN layer step (forward + backward, layer.MoEFFNStep) on the GPU vs the oracle
composed from the same definitions: permute, quantize, fp64 GEMMs over the dequantized
operands, SwiGLU, combine.

The layer's inputs are chosen so that most stages are exact and can be held bit for bit:
activations, weights and the output gradient are small integers times powers of two, and the
routing weights are powers of two.  Then every quantization of them is exact, GEMM1 and the
dgrad of the down projection are exact sums (fp32 in tensor memory and fp64 in the oracle give
the same number), and the combine backward is exact.  Each stage is compared with the oracle
on the oracle's own upstream values:

  bit for bit      permutation, GEMM1 output, combine backward dY (and its quantized forms,
                   also when formed on the fly from dOut), dgrad2 output
  near-tie rule    the SwiGLU codes and scales of h and dH (both forms): a difference only where
                   the kernel's fp32 SwiGLU error bound explains it (near_tie)
  one GEMM stage   GEMM2, dgrad1 and both wgrads: max|gpu - oracle| <= 2e-2 x rms(oracle), plus,
                   per element, exactly the change that the explained SwiGLU code differences
                   make through that GEMM (zero where no such difference feeds the element)
                   and, for the bf16 outputs, their own final rounding (2^-9 |oracle|): the
                   power-of-two routing weights spread the rows' magnitudes over 16x, so the
                   largest outputs lie far enough above the rms for one bf16 rounding to
                   exceed 2e-2 x rms
  linear maps      combine forward, dgate and the un-permute sum of dx: the bound of their
                   input carried through the map, plus one bf16 / fp32 rounding"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300.layer import MoEFFNStep
from gpu_util import TOL, bits, check_dev_err, dev, np_, sf_x4_first  # noqa: F401
from swiglu_check import check_swiglu_outputs

pytestmark = pytest.mark.gpu


def _val(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _deq(q, sf):
    """Dequantized MXFP8 values; sf holds one scale byte per 32 consecutive elements of a row."""
    v = oracle.e4m3_decode(q.reshape(-1)).reshape(q.shape)
    return v * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=1))[:, : q.shape[1]]


def _grid(rng, shape, step):
    return torch.from_numpy((rng.integers(-3, 4, size=shape) * step).astype(np.float32)).to(torch.bfloat16)


def _within(got, ref, bound, what):
    excess = np.abs(got - ref) - bound
    assert np.all(excess <= 0), "%s: %d elements beyond the bound, worst by %.3g (rms %.3g)" % (
        what, int((excess > 0).sum()), float(excess.max()), float(np.sqrt(np.mean(ref ** 2))))


@pytest.mark.parametrize("fuse_dy", [True, False])
@pytest.mark.parametrize("T,E,k,H,I", [(512, 4, 2, 256, 128), (384, 8, 3, 384, 256)])
def test_layer_step(dev, T, E, k, H, I, fuse_dy):
    rng = np.random.default_rng(900 + T)
    st = MoEFFNStep(T, E, k, H, I, device=dev, fuse_dy=fuse_dy)
    I2, R = 2 * I, T * k
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32))
    ids = torch.sort(logits, dim=1, descending=True, stable=True).indices[:, :k].to(torch.int32).contiguous()
    gate = torch.from_numpy(np.exp2(-rng.integers(1, 5, size=(T, k))).astype(np.float32))
    x = _grid(rng, (T, H), 2.0 ** -3)
    w1 = _grid(rng, (E, I2, H), 2.0 ** -4)
    w2 = _grid(rng, (E, H, I), 2.0 ** -4)
    dout = _grid(rng, (T, H), 2.0 ** -10)
    for name, t in (("x", x), ("ids", ids), ("gate", gate), ("w1", w1), ("w2", w2), ("dout", dout)):
        getattr(st, name).copy_(t.to(dev))
    st.step()
    check_dev_err(st.dev_err)

    p = oracle.permute(ids.numpy(), E)
    off, poff, src, dst = p["off"], p["poff"], p["src_row"], p["dst_of"]
    for key in ("off", "poff"):
        assert np.array_equal(np_(getattr(st, key)), p[key])
    assert np.array_equal(np_(st.src_row)[:R], src)
    gn = gate.numpy().astype(np.float64)
    xb = bits(x)
    w1b, w2b = bits(w1).reshape(E * I2, H), bits(w2).reshape(E * H, I)
    counts = np.diff(off)
    expert_of = np.repeat(np.arange(E), counts)
    rows_pad = np.concatenate([np.arange(poff[e], poff[e] + counts[e]) for e in range(E)]).astype(np.int64)
    P, ld = int(poff[-1]), st.pb

    def grouped(aq, asf, bq, bsf, n):                      # rows grouped by expert, B per expert [n x K]
        out = np.zeros((R, n))
        for e in range(E):
            r0, r1 = int(off[e]), int(off[e + 1])
            if r1 > r0:
                out[r0:r1] = oracle.gemm_nt(aq[r0:r1], asf[r0:r1], bq[e * n:(e + 1) * n], bsf[e * n:(e + 1) * n])
        return out

    def bf(v):
        return oracle.to_bf16_bits(v).reshape(v.shape)

    def rows_form(q_dev, sf_dev, cols):                    # the kernel's rowwise codes and scales
        sf = oracle.sf_from_tcgen05(np_(sf_dev), max(P, 1), cols // 32)[rows_pad]
        return np_(q_dev)[:R], sf

    def cols_form(q_dev, sf_dev, cols):                    # the kernel's columnwise ones (four-copy scales)
        return np_(q_dev)[:, :P], oracle.sf_from_tcgen05(sf_x4_first(sf_dev, ld // 128, P // 128), cols,
                                                         ld // 32)[:, : P // 32]

    # ---- forward: gather + quantize x, GEMM1 (exact), SwiGLU -> h codes, GEMM2, combine
    xg = oracle.gather_rows(xb, src)
    aq, asf = oracle.quantize_rowwise(xg)
    w1q, w1sf = oracle.quantize_rowwise(w1b)
    a1 = grouped(aq, asf, w1q, w1sf, I2)
    assert np.all(a1 * 2.0 ** 7 == np.round(a1 * 2.0 ** 7))           # an exact sum on the 2^-7 grid
    a1b = bf(a1)
    assert np.array_equal(bits(st.out1)[:R], a1b), "GEMM1 output differs from the oracle"
    check_swiglu_outputs(False, a1b, None, off, poff, st.h_q, st.h_sf, st.hc_q, st.hc_sf, x4=(False, True))
    h32 = oracle.swiglu_fwd(a1b)
    hq, hsf = oracle.quantize_rowwise_ex(h32)
    dh_row = _deq(*rows_form(st.h_q, st.h_sf, I)) - _deq(hq, hsf)     # explained near-tie differences only
    w2q, w2sf = oracle.quantize_rowwise(w2b)
    w2d = np.abs(_deq(w2q, w2sf)).reshape(E, H, I)
    Y = grouped(hq, hsf, w2q, w2sf, H)
    allow_y = np.zeros((R, H))
    for r, i in zip(*np.nonzero(dh_row)):
        allow_y[r] += abs(dh_row[r, i]) * w2d[expert_of[r], :, i]
    bound_y = TOL * np.sqrt(np.mean(Y ** 2)) + 2.0 ** -9 * np.abs(Y) + allow_y
    _within(_val(bits(st.out2)[:R]), Y, bound_y, "GEMM2 output")
    Yb = bf(Y)
    out_ref = _val(oracle.combine_fwd(Yb, gate.numpy(), dst))
    bound_out = np.einsum("tj,tjh->th", gn, bound_y[dst] + 2.0 ** -8 * np.abs(_val(Yb))[dst]) + \
        2.0 ** -8 * np.abs(out_ref)
    _within(_val(bits(st.out)), out_ref, bound_out, "combined output")

    # ---- backward: combine backward (exact dY), dgrad2 (exact), SwiGLU backward -> dH codes,
    #      dgrad1 + un-permute, both weight gradients
    dYb, dgate_ref = oracle.combine_bwd(bits(dout), Yb, gate.numpy(), dst)
    if not fuse_dy:
        assert np.array_equal(bits(st.dy)[:R], dYb[:R]), "combine backward dY differs from the oracle"
    # dY's operand forms, byte for byte (with fuse_dy they are formed from dOut on the fly)
    dyq_o, dysf_o = oracle.quantize_rowwise(dYb)
    gq, gsf = rows_form(st.dy_q, st.dy_sf, H)
    assert np.array_equal(gq, dyq_o) and np.array_equal(gsf, dysf_o), "rowwise dY operand differs"
    dyc_o, dycsf_o = oracle.quantize_colwise_seg(dYb, off, poff, ld)
    assert np.array_equal(np_(st.dyc_q)[:, :P], dyc_o[:, :P])
    assert np.array_equal(oracle.sf_from_tcgen05(np_(st.dyc_sf), H, ld // 32)[:, : P // 32], dycsf_o[:, : P // 32])
    dov = np.abs(_val(bits(dout)))
    bound_dgate = np.einsum("th,tjh->tj", dov, bound_y[dst] + 2.0 ** -8 * np.abs(_val(Yb))[dst]) + \
        H * 2.0 ** -24 * np.einsum("th,tjh->tj", dov, np.abs(_val(Yb))[dst])    # fp32 sum of H products
    _within(np_(st.dgate).astype(np.float64), dgate_ref, bound_dgate, "dgate")
    dyq, dysf = dyq_o, dysf_o
    seg2 = np.arange(0, (E + 1) * H, H, dtype=np.int32)
    w2c, w2csf = oracle.quantize_colwise_seg(w2b, seg2, seg2, E * H)
    dh_in = np.zeros((R, I))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            dh_in[r0:r1] = oracle.gemm_nt(dyq[r0:r1], dysf[r0:r1], w2c[:, e * H:(e + 1) * H],
                                          w2csf[:, e * H // 32:(e + 1) * H // 32])
    dh_b = bf(dh_in)
    assert np.array_equal(bits(st.dh_in)[:R], dh_b), "dgrad2 output differs from the oracle"
    check_swiglu_outputs(True, a1b, dh_b, off, poff, st.dh_q, st.dh_sf, st.dhc_q, st.dhc_sf, x4=(False, False))
    dH32 = oracle.swiglu_bwd(dh_b, a1b)
    dhq, dhsf = oracle.quantize_rowwise_ex(dH32)
    d_dh_row = _deq(*rows_form(st.dh_q, st.dh_sf, I2)) - _deq(dhq, dhsf)
    seg1 = np.arange(0, (E + 1) * I2, I2, dtype=np.int32)
    w1c, w1csf = oracle.quantize_colwise_seg(w1b, seg1, seg1, E * I2)
    w1d = np.abs(_deq(w1q, w1sf)).reshape(E, I2, H)
    dXr = np.zeros((R, H))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            dXr[r0:r1] = oracle.gemm_nt(dhq[r0:r1], dhsf[r0:r1], w1c[:, e * I2:(e + 1) * I2],
                                        w1csf[:, e * I2 // 32:(e + 1) * I2 // 32])
    allow_dx = np.zeros((R, H))
    for r, i in zip(*np.nonzero(d_dh_row)):
        allow_dx[r] += abs(d_dh_row[r, i]) * w1d[expert_of[r], i, :]
    bound_dxr = TOL * np.sqrt(np.mean(dXr ** 2)) + 2.0 ** -9 * np.abs(dXr) + allow_dx
    _within(_val(bits(st.dx_routed)[:R]), dXr, bound_dxr, "dgrad1 output")
    dXrb = bf(dXr)
    dx_ref = _val(oracle.combine_fwd(dXrb, np.ones((T, k), np.float32), dst))
    bound_dx = (bound_dxr + 2.0 ** -8 * np.abs(_val(dXrb)))[dst].sum(axis=1) + 2.0 ** -8 * np.abs(dx_ref)
    _within(_val(bits(st.dx)), dx_ref, bound_dx, "input gradient")

    # weight gradients: contraction over each expert's tokens (columnwise operands)
    dyc, dycsf = oracle.quantize_colwise_seg(dYb, off, poff, ld)
    hc, hcsf = oracle.quantize_colwise_seg_ex(h32, off, poff, ld)
    dhc, dhcsf = oracle.quantize_colwise_seg_ex(dH32, off, poff, ld)
    xc, xcsf = oracle.quantize_colwise_seg(xg, off, poff, ld)
    d_hc = _deq(*cols_form(st.hc_q, st.hc_sf, I)) - _deq(hc[:, :P], hcsf[:, : P // 32])
    gq, gs = np_(st.dhc_q)[:, :P], oracle.sf_from_tcgen05(np_(st.dhc_sf), I2, ld // 32)[:, : P // 32]
    d_dhc = _deq(gq, gs) - _deq(dhc[:, :P], dhcsf[:, : P // 32])
    dyd = np.abs(_deq(dyc[:, :P], dycsf[:, : P // 32]))                # [H x P]
    xd = np.abs(_deq(xc[:, :P], xcsf[:, : P // 32]))                    # [H x P]
    for e in range(E):
        p0, p1 = int(poff[e]), int(poff[e + 1])
        if p1 == p0:
            assert np.all(np_(st.dw2[e]) == 0) and np.all(np_(st.dw1[e]) == 0)
            continue
        s0, s1 = p0 // 32, p1 // 32
        dw2 = oracle.gemm_nt(dyc[:, p0:p1], dycsf[:, s0:s1], hc[:, p0:p1], hcsf[:, s0:s1])
        dw1 = oracle.gemm_nt(dhc[:, p0:p1], dhcsf[:, s0:s1], xc[:, p0:p1], xcsf[:, s0:s1])
        allow2 = dyd[:, p0:p1] @ np.abs(d_hc[:, p0:p1]).T                # [H x I]
        allow1 = np.abs(d_dhc[:, p0:p1]) @ xd[:, p0:p1].T                 # [I2 x H]
        _within(np_(st.dw2[e]).astype(np.float64), dw2, TOL * np.sqrt(np.mean(dw2 ** 2)) + allow2,
                "dW2 of expert %d" % e)
        _within(np_(st.dw1[e]).astype(np.float64), dw1, TOL * np.sqrt(np.mean(dw1 ** 2)) + allow1,
                "dW1 of expert %d" % e)
