"""Shared helpers of the GPU parity tests (marshalling only; no method arithmetic)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_rowwise_gb300 import binding as mx
from mxfp8_block_scaled_rowwise_gb300 import synth

TOL = 2e-2   # max|gpu - oracle| <= TOL * rms(oracle) for GEMM outputs
# quantize modes of the grouped GEMMs' B operands: scales in the four-copy layout
ROW_B = mx.MX_ROWWISE | mx.MX_ROWWISE_X4
COL_B = mx.MX_COLWISE | mx.MX_COLWISE_X4


@pytest.fixture(scope="session")
def dev():
    from mxfp8_block_scaled_rowwise_gb300 import _build
    _build.build()
    oracle.build()
    mx.load()
    return torch.device("cuda:0")


def bits(t):
    return synth.bf16_bits(t)


def from_bits(b: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def np_(t):
    return t.detach().cpu().numpy()


def offsets(counts):
    counts = np.asarray(counts, np.int64)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    return off, poff


def rel_err(got, ref):
    rms = float(np.sqrt(np.mean(np.square(ref)))) if ref.size else 0.0
    if rms == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref))) / rms


def check_dev_err(err):
    torch.cuda.synchronize()
    v = int(err.item())
    assert v == 0, "device error bits %d" % v


def sf_x4_first(buf, groups=None, used_groups=None) -> np.ndarray:
    """A scale array in the four-copy layout (each 512-byte atom stored four times) as the
    plain tensor-core atom layout, after checking that the four copies are identical.
    groups / used_groups: atoms per 128-row block and how many of them the call wrote (a
    columnwise array over padded positions is written only up to poff[E]); unwritten atoms
    are not checked."""
    a = np_(buf).reshape(-1, 4, 512)
    chk = a if groups is None else a.reshape(-1, groups, 4, 512)[:, :used_groups]
    assert np.array_equal(chk, np.broadcast_to(chk[..., :1, :], chk.shape)), "the four copies of a scale atom differ"
    return np.ascontiguousarray(a[:, 0]).reshape(-1)
