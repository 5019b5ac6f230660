"""moe_permute_noalloc -- the permutation for callers that cannot allocate device memory.

Such callers (a fixed memory plan owned by someone else, or a region where
cudaMalloc's implicit device synchronization is not allowed) get the same result as
moe_permute, with the scratch taken from a fixed array inside the library instead
of a caller workspace.  This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth
from gpu_util import dev, np_  # noqa: F401

pytestmark = pytest.mark.gpu


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


def _same(a, b, R, nsf=None):
    for key in ("counts", "off", "poff"):
        assert np.array_equal(np_(a[key]), np_(b[key])), key
    assert np.array_equal(np_(a["src_row"])[:R], np_(b["src_row"])[:R])
    assert np.array_equal(np_(a["dst_of"])[:R], np_(b["dst_of"])[:R])
    if a.get("q") is not None:
        rows = int(np_(a["off"])[-1])
        assert np.array_equal(np_(a["q"])[:rows], np_(b["q"])[:rows])
        P = int(np_(a["poff"])[-1])
        n = mx.mx_sf_bytes(P, a["q"].shape[1] // 32)
        assert np.array_equal(np_(a["sf"])[:n], np_(b["sf"])[:n])


def test_noalloc_matches_moe_permute_on_two_calls_in_a_row(dev):
    # two different problems back to back: the second call must not see the first's scratch
    g = synth.generator(4242)
    cases = [(synth.ffn(with_weights=False)["ids"], 32, 512), (synth.uniform_ids(3001, 128, 8, g), 128, 256)]
    for ids, E, K in cases:
        ids = ids.to(dev)
        T, k = ids.shape
        x = synth.randn_bf16((T, K), g).to(dev)
        qx = mx.quantize_alloc(x, mx.MX_ROWWISE)
        ref = mx.permute_alloc(ids, E, qx["q_row"], qx["sf_row"])
        got = _noalloc(ids, E, qx["q_row"], qx["sf_row"])
        torch.cuda.synchronize()
        assert int(got["dev_err"].item()) == 0 and int(ref["dev_err"].item()) == 0
        _same(got, ref, T * k)


def test_noalloc_rejects_problems_beyond_its_scratch(dev):
    T, k, E = 1 << 20, 8, 1024       # needs 2 * 4096 * 1024 * 4 bytes of scratch, far over 1 MiB
    assert mx.moe_permute_workspace_bytes(T, k, E) > (1 << 20)
    lib = mx.load()
    d = torch.zeros(16, dtype=torch.int32, device=dev)
    p = d.data_ptr()
    st = lib.moe_permute_noalloc(p, T, k, E, p, p, p, p, p, None, None, 0, None, None, p, None)
    assert st == -6 and lib.mx_status_str(st) == b"MX_ERR_TOO_LARGE"
