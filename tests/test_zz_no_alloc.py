"""moe_permute_noalloc -- the permutation for callers that cannot allocate device memory.

Such callers (a fixed memory plan owned by someone else, or a region where cudaMalloc's
implicit device synchronization is not allowed) get the same result as moe_permute, with
the scratch taken from a fixed array inside the library instead of a caller workspace.
Every result is checked against the CPU oracle (counts, offsets, indices, gathered codes and
scales) and against moe_permute, on calls that follow each other and share that array.
This file is collected last so that a run stopping at the first failure has already run
every other test."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import bits, dev, np_  # noqa: F401

pytestmark = pytest.mark.gpu

SCRATCH = 1 << 20   # bytes of the library's fixed array


def _noalloc(ids, E, q_in=None, sf_in=None):
    T, k = ids.shape
    d = ids.device
    R = T * k
    out = dict(counts=torch.full((E,), -7, dtype=torch.int32, device=d),
               off=torch.full((E + 1,), -7, dtype=torch.int32, device=d),
               poff=torch.full((E + 1,), -7, dtype=torch.int32, device=d),
               src_row=torch.full((max(R, 1),), -7, dtype=torch.int32, device=d),
               dst_of=torch.full((max(R, 1),), -7, dtype=torch.int32, device=d),
               dev_err=torch.zeros(1, dtype=torch.int32, device=d))
    K = 0
    q_out = sf_out = None
    if q_in is not None:
        K = q_in.shape[1]
        q_out = torch.zeros(max(R, 1), K, dtype=torch.uint8, device=d)
        sf_out = torch.zeros(mx.mx_sf_bytes(mx.mx_padded_rows_bound(R, E), K // 32), dtype=torch.uint8, device=d)
    mx.moe_permute_noalloc(ids, T, k, E, out["counts"], out["off"], out["poff"], out["src_row"], out["dst_of"],
                           q_in, sf_in, K, q_out, sf_out, out["dev_err"])
    out.update(q=q_out, sf=sf_out)
    return out


def _against_oracle(got, ids_np, E, x_bits=None):
    """Every output of the call against the oracle's permutation (and its gather of the
    oracle's own rowwise quantization of x); returns the oracle's permutation."""
    p = oracle.permute(ids_np, E)
    R = int(p["off"][-1])
    n = ids_np.size
    for key in ("counts", "off", "poff"):
        assert np.array_equal(np_(got[key]), p[key]), key
    src = np_(got["src_row"])
    assert np.array_equal(src[:R], p["src_row"])
    assert np.all(src[R:n] == -1), "src_row entries past off[E] must be -1"
    assert np.array_equal(np_(got["dst_of"])[:n], p["dst_of"].reshape(-1))
    if x_bits is not None:
        oq, osf = oracle.quantize_rowwise(x_bits)
        assert np.array_equal(np_(got["q"])[:R], oracle.gather_rows(oq, p["src_row"]))
        want = oracle.sf_to_tcgen05(oracle.place_sf_rows(oracle.gather_rows(osf, p["src_row"]), p["off"], p["poff"]))
        assert np.array_equal(np_(got["sf"])[: want.size], want)
    return p


def _same_as_workspace_call(got, ref, R):
    for key in ("counts", "off", "poff"):
        assert np.array_equal(np_(got[key]), np_(ref[key])), key
    assert np.array_equal(np_(got["src_row"])[:R], np_(ref["src_row"])[:R])
    assert np.array_equal(np_(got["dst_of"])[:R], np_(ref["dst_of"])[:R])


def test_noalloc_matches_oracle_and_moe_permute_on_two_calls_in_a_row(dev):
    # two different problems back to back: the second call must not see the first's scratch
    g = synth.generator(4242)
    cases = [(synth.ffn(with_weights=False)["ids"], 32, 512), (synth.uniform_ids(3001, 128, 8, g), 128, 256)]
    for ids, E, K in cases:
        T, k = ids.shape
        x = synth.randn_bf16((T, K), g)
        idsd = ids.to(dev)
        qx = mx.quantize_alloc(x.to(dev), mx.MX_ROWWISE)
        got = _noalloc(idsd, E, qx["q_row"], qx["sf_row"])
        ref = mx.permute_alloc(idsd, E, qx["q_row"], qx["sf_row"])
        torch.cuda.synchronize()
        assert int(got["dev_err"].item()) == 0 and int(ref["dev_err"].item()) == 0
        _against_oracle(got, ids.numpy(), E, bits(x))
        _same_as_workspace_call(got, ref, T * k)


def test_noalloc_at_its_size_limit(dev):
    # scratch = 8 * ceil(T*k / 2048) * E + 16 bytes: ceil(T*k / 2048) * E = 131070 fills the
    # 1 MiB array exactly (E = 510 experts, T*k = 257 * 2048 routed slots) and is accepted ...
    E, k = 510, 8
    T = 257 * 2048 // k
    assert mx.moe_permute_workspace_bytes(T, k, E) == SCRATCH
    ids = torch.randint(0, E, (T, k), dtype=torch.int32, generator=synth.generator(99))
    got = _noalloc(ids.to(dev), E)
    torch.cuda.synchronize()
    assert int(got["dev_err"].item()) == 0
    _against_oracle(got, ids.numpy(), E)
    # ... while one routed slot more needs another 2048-slot chunk and is refused before any launch
    lib = mx.load()
    d = torch.zeros(16, dtype=torch.int32, device=dev)
    p = d.data_ptr()
    assert mx.moe_permute_workspace_bytes(T * k + 1, 1, E) > SCRATCH
    st = lib.moe_permute_noalloc(p, T * k + 1, 1, E, p, p, p, p, p, None, None, 0, None, None, p, None)
    assert st == -6 and lib.mx_status_str(st) == b"MX_ERR_TOO_LARGE"


def test_noalloc_flags_invalid_ids(dev):
    # ids outside [0, E): the slot is dropped (dst_of = -1), src_row is -1 past off[E], and the
    # device error word says so -- while the shared array carries the previous call's contents
    g = synth.generator(31)
    ids = synth.uniform_ids(999, 12, 3, g)
    flat = ids.view(-1)
    flat[torch.randint(0, flat.numel(), (40,), generator=g)] = 12
    flat[torch.randint(0, flat.numel(), (25,), generator=g)] = -3
    got = _noalloc(ids.to(dev), 12)
    torch.cuda.synchronize()
    assert int(got["dev_err"].item()) & mx.MX_DEVERR_BAD_EXPERT_ID
    p = _against_oracle(got, ids.numpy(), 12)
    assert p["bad"] > 0 and int(p["off"][-1]) < ids.numel()


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    T, k, E = 1 << 20, 8, 1024       # needs 2 * 4096 * 1024 * 4 bytes of scratch, far over 1 MiB
    assert mx.moe_permute_workspace_bytes(T, k, E) > SCRATCH
    lib = mx.load()
    d = torch.zeros(16, dtype=torch.int32, device=dev)
    p = d.data_ptr()
    st = lib.moe_permute_noalloc(p, T, k, E, p, p, p, p, p, None, None, 0, None, None, p, None)
    assert st == -6 and lib.mx_status_str(st) == b"MX_ERR_TOO_LARGE"
