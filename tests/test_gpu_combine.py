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
