"""GPU combine (unpermute / weighted merge) forward and backward vs the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import bits, check_dev_err, dev, np_  # noqa: F401

pytestmark = pytest.mark.gpu


def _val(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(name):
    g = synth.generator(55)
    if name == "tiny":
        T, E, k, H = 512, 4, 1, 256
        ids = synth.uniform_ids(T, E, k, g)
    elif name == "ffn_slice":
        T, E, k, H = 1024, 32, 8, 7168
        ids = synth.topk_ids(torch.randn(T, E, generator=g), k)
    else:
        d = synth.skewed(with_weights=False)
        T, E, k, H, ids = 1024, d["E"], d["k"], 512, d["ids"][:1024].contiguous()
    R = T * k
    Y = synth.randn_bf16((R, H), g)
    gate = torch.softmax(torch.randn(T, k, generator=g), dim=1).to(torch.float32)
    dOut = synth.randn_bf16((T, H), g, std=1e-2)
    return T, E, k, H, ids, Y, gate, dOut


@pytest.mark.parametrize("name", ["tiny", "ffn_slice", "skewed"])
def test_combine_fwd_bwd(dev, name):
    T, E, k, H, ids, Y, gate, dOut = _case(name)
    R = T * k
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(ids.to(dev), E, dev_err=err)
    dst = pm["dst_of"][: T * k].view(T, k).contiguous()
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    mx.moe_combine_fwd(Y.to(dev), gate.to(dev), dst, T, k, H, R, out, err)
    dY = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=dev)
    dgate = torch.empty(T, k, dtype=torch.float32, device=dev)
    mx.moe_combine_bwd(dOut.to(dev), Y.to(dev), gate.to(dev), dst, T, k, H, R, dY, dgate, err)
    check_dev_err(err)
    p = oracle.permute(ids.numpy(), E)
    Yb, dOb, gn = bits(Y), bits(dOut), gate.numpy()
    # forward: fp32 accumulation of k products, then bf16 -> one bf16 ulp plus accumulation error
    ref = _val(oracle.combine_fwd(Yb, gn, p["dst_of"]))
    got = _val(bits(out))
    mag = np.zeros_like(ref)
    for j in range(k):
        mag += np.abs(gn[:, j:j + 1].astype(np.float64)) * np.abs(_val(Yb[p["dst_of"][:, j]]))
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -20 * mag)
    # backward: dY is a single rounded product -> bit-exact; dgate within fp32 summation error
    rdY, rdg = oracle.combine_bwd(dOb, Yb, gn, p["dst_of"])
    assert np.array_equal(bits(dY), rdY)
    mag_g = np.zeros((T, k))
    for j in range(k):
        mag_g[:, j] = np.sum(np.abs(_val(dOb)) * np.abs(_val(Yb[p["dst_of"][:, j]])), axis=1)
    assert np.all(np.abs(np_(dgate).astype(np.float64) - rdg) <= H * 2.0 ** -23 * mag_g + 1e-30)


def test_combine_unit_gates_is_unpermute_sum(dev):
    T, E, k, H, ids, Y, gate, dOut = _case("ffn_slice")
    R = T * k
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(ids.to(dev), E, dev_err=err)
    dst = pm["dst_of"][: T * k].view(T, k).contiguous()
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    mx.moe_combine_fwd(Y.to(dev), None, dst, T, k, H, R, out, err)
    check_dev_err(err)
    p = oracle.permute(ids.numpy(), E)
    ref = _val(oracle.combine_fwd(bits(Y), np.ones((T, k), np.float32), p["dst_of"]))
    got = _val(bits(out))
    mag = sum(np.abs(_val(bits(Y))[p["dst_of"][:, j]]) for j in range(k))
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -20 * mag)


def test_combine_drops_out_of_range_rows(dev):
    T, k, H, R = 4, 2, 64, 8
    Y = synth.randn_bf16((R, H), synth.generator(2)).to(dev)
    gate = torch.ones(T, k, dtype=torch.float32, device=dev)
    dst = torch.tensor([[0, 1], [2, 99], [-1, 3], [4, 5]], dtype=torch.int32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    err = mx.new_dev_err(dev)
    mx.moe_combine_fwd(Y, gate, dst, T, k, H, R, out, err)
    torch.cuda.synchronize()
    assert int(err.item()) & mx.MX_DEVERR_BAD_SEGMENTS
    assert torch.equal(out[1], Y[2]) and torch.equal(out[2], Y[3])


@pytest.mark.parametrize("name", ["ffn_slice", "skewed"])
def test_combine_bwd_without_dy_and_the_scaled_gather_quantize(dev, name):
    # moe_combine_bwd_ex without dY: the same dgate bytes, plus the routing weight of every
    # routed row; mxfp8_gather_quantize_ex of dOut with those weights as row scales gives, byte
    # for byte, the oracle's quantization of the combine backward's dY (rowwise and columnwise)
    T, E, k, H, ids, Y, gate, dOut = _case(name)
    R = T * k
    err = mx.new_dev_err(dev)
    pm = mx.permute_alloc(ids.to(dev), E, dev_err=err)
    dst = pm["dst_of"][: T * k].view(T, k).contiguous()
    dY = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    dgate = torch.empty(T, k, dtype=torch.float32, device=dev)
    mx.moe_combine_bwd(dOut.to(dev), Y.to(dev), gate.to(dev), dst, T, k, H, R, dY, dgate, err)
    dgate2 = torch.empty(T, k, dtype=torch.float32, device=dev)
    rows = torch.full((R,), float("nan"), dtype=torch.float32, device=dev)
    mx.moe_combine_bwd_ex(dOut.to(dev), Y.to(dev), gate.to(dev), dst, T, k, H, R, None, dgate2, rows, err)
    pb = mx.mx_padded_rows_bound(R, E)
    q_row = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sf_row = torch.empty(mx.mx_sf_bytes(pb, H // 32), dtype=torch.uint8, device=dev)
    q_col = torch.empty(H, pb, dtype=torch.uint8, device=dev)
    sf_col = torch.empty(mx.mx_sf_bytes(H, pb // 32), dtype=torch.uint8, device=dev)
    mx.mxfp8_gather_quantize_ex(dOut.to(dev), T, H, mx.MX_ROWWISE | mx.MX_COLWISE, pm["src_row"], rows, pm["off"],
                                pm["poff"], E, R, pb, q_row, sf_row, q_col, sf_col, err)
    check_dev_err(err)
    assert torch.equal(dgate.view(torch.int32), dgate2.view(torch.int32))
    p = oracle.permute(ids.numpy(), E)
    gn = gate.numpy()
    want_rows = np.empty(R, np.float32)
    want_rows[p["dst_of"].reshape(-1)] = gn.reshape(-1)
    assert np.array_equal(np_(rows), want_rows)
    rdY, _ = oracle.combine_bwd(bits(dOut), bits(Y), gn, p["dst_of"])
    oq, osf = oracle.quantize_rowwise(rdY)
    assert np.array_equal(np_(q_row), oq)
    want = oracle.sf_to_tcgen05(oracle.place_sf_rows(osf, p["off"], p["poff"]))
    assert np.array_equal(np_(sf_row)[: want.size], want)
    P = int(p["poff"][-1])
    cq, csf = oracle.quantize_colwise_seg(rdY, p["off"], p["poff"], pb)
    assert np.array_equal(np_(q_col)[:, :P], cq[:, :P])
    got = oracle.sf_from_tcgen05(np_(sf_col), H, pb // 32)
    assert np.array_equal(got[:, : P // 32], csf[:, : P // 32])
