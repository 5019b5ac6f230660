"""GPU permutation vs the CPU oracle: bit-exact counts, offsets, indices and gathered bytes."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import bits, check_dev_err, dev, np_  # noqa: F401

pytestmark = pytest.mark.gpu


def _compare(ids_np, E, pm):
    p = oracle.permute(ids_np, E)
    R = int(p["off"][-1])
    for key in ("counts", "off", "poff"):
        assert np.array_equal(np_(pm[key]), p[key]), key
    assert np.array_equal(np_(pm["src_row"])[:R], p["src_row"])
    assert np.array_equal(np_(pm["dst_of"])[: ids_np.size], p["dst_of"].reshape(-1))
    return p


def _ids_cases():
    g = synth.generator(77)
    yield "tiny_top1", synth.uniform_ids(512, 4, 1, g), 4
    yield "random_small", synth.uniform_ids(37, 5, 2, g), 5
    yield "ffn_top8_of_32", synth.ffn(with_weights=False)["ids"], 32
    yield "skewed_zipf_128", synth.skewed(with_weights=False)["ids"], 128
    yield "single_expert", torch.zeros(1000, 1, dtype=torch.int32), 1
    yield "ragged_tail_chunk", synth.uniform_ids(2049, 16, 3, g), 16
    yield "E1024", synth.uniform_ids(3000, 1024, 8, g), 1024
    # one chunk of at most 2048 slots takes the single-launch path: the largest expert count,
    # exactly one full chunk, and one slot over it (two chunks)
    yield "E1024_one_chunk", synth.uniform_ids(200, 1024, 8, g), 1024
    yield "full_one_chunk", synth.uniform_ids(256, 32, 8, g), 32
    yield "one_chunk_plus_one", synth.uniform_ids(683, 64, 3, g), 64


@pytest.mark.parametrize("name,ids,E", list(_ids_cases()), ids=lambda v: v if isinstance(v, str) else "")
def test_index_permutation(dev, name, ids, E):
    pm = mx.permute_alloc(ids.to(dev), E)
    check_dev_err(pm["dev_err"])
    _compare(ids.numpy(), E, pm)


def test_skewed_has_empty_and_ragged_experts():
    ids = synth.skewed(with_weights=False)["ids"].numpy()
    counts = np.bincount(ids.reshape(-1), minlength=128)
    assert (counts == 0).sum() >= 3 and np.any(counts % 128 != 0)


def test_invalid_ids_flagged(dev):
    ids = torch.tensor([[0, 5], [-1, 1], [1, 0]], dtype=torch.int32)
    pm = mx.permute_alloc(ids.to(dev), 2)
    torch.cuda.synchronize()
    assert int(pm["dev_err"].item()) & mx.MX_DEVERR_BAD_EXPERT_ID
    p = _compare(ids.numpy(), 2, pm)
    assert np.all(np_(pm["src_row"])[int(p["off"][-1]):6] == -1)


def test_empty_input(dev):
    ids = torch.empty(0, 4, dtype=torch.int32)
    pm = mx.permute_alloc(ids.to(dev), 8)
    check_dev_err(pm["dev_err"])
    assert np.all(np_(pm["counts"]) == 0) and np.all(np_(pm["off"]) == 0) and np.all(np_(pm["poff"]) == 0)


@pytest.mark.parametrize("T,K,E,k", [(512, 256, 4, 1), (300, 96, 7, 3), (4096, 4096, 128, 8)])
def test_gather_quantized_rows(dev, T, K, E, k):
    g = synth.generator(T + K)
    x = synth.randn_bf16((T, K), g)
    ids = synth.uniform_ids(T, E, k, g) if E != 128 else synth.skewed(with_weights=False)["ids"]
    xd = x.to(dev)
    qx = mx.quantize_alloc(xd, mx.MX_ROWWISE)
    pm = mx.permute_alloc(ids.to(dev), E, qx["q_row"], qx["sf_row"])
    check_dev_err(pm["dev_err"])
    p = _compare(ids.numpy(), E, pm)
    oq, osf = oracle.quantize_rowwise(bits(x))
    R = int(p["off"][-1])
    assert np.array_equal(np_(pm["q"])[:R], oracle.gather_rows(oq, p["src_row"]))
    want = oracle.sf_to_tcgen05(oracle.place_sf_rows(oracle.gather_rows(osf, p["src_row"]), p["off"], p["poff"]))
    assert np.array_equal(np_(pm["sf"])[: want.size], want)


def test_gather_bf16_rows(dev):
    g = synth.generator(5)
    x = synth.randn_bf16((700, 192), g)
    ids = synth.uniform_ids(700, 9, 2, g)
    pm = mx.permute_alloc(ids.to(dev), 9)
    R = 1400
    out = torch.empty(R, 192, dtype=torch.bfloat16, device=dev)
    mx.moe_gather_rows(x.to(dev), 192 * 2, pm["src_row"], R, out)
    torch.cuda.synchronize()
    p = oracle.permute(ids.numpy(), 9)
    assert np.array_equal(bits(out.cpu()), oracle.gather_rows(bits(x), p["src_row"]))
