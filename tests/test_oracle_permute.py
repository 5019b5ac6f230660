"""Pins of the oracle's token permutation -- CPU only."""
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _brute(ids, E):
    T, k = ids.shape
    pairs = sorted(((int(ids[t, j]), t * k + j) for t in range(T) for j in range(k) if 0 <= ids[t, j] < E))
    counts = np.bincount([e for e, _ in pairs], minlength=E)[:E]
    src_row = np.array([i // k for _, i in pairs], np.int32)
    dst_of = np.full(T * k, -1, np.int32)
    for r, (_, i) in enumerate(pairs):
        dst_of[i] = r
    return counts, src_row, dst_of.reshape(T, k)


def test_golden_small():
    vals = {}
    with open(os.path.join(GOLDEN, "permute_small.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                key, *rest = ln.split()
                vals[key] = np.array([int(v) for v in rest], np.int32)
    E, k = int(vals["E"][0]), int(vals["k"][0])
    ids = vals["ids"].reshape(-1, k)
    p = oracle.permute(ids, E)
    for key in ("counts", "off", "poff", "src_row"):
        assert np.array_equal(p[key], vals[key]), key
    assert np.array_equal(p["dst_of"].reshape(-1), vals["dst_of"])


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (37, 2, 5, 1), (300, 8, 32, 2), (1000, 4, 128, 3), (64, 8, 8, 4)])
def test_against_brute_sort(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] if k <= E else rng.integers(0, E, k) for _ in range(T)]).astype(np.int32)
    p = oracle.permute(ids, E)
    counts, src_row, dst_of = _brute(ids, E)
    assert np.array_equal(p["counts"], counts)
    assert np.array_equal(p["src_row"], src_row)
    assert np.array_equal(p["dst_of"], dst_of)
    # invariants
    assert p["off"][-1] == T * k and np.all(np.diff(p["off"]) == counts)
    assert np.all(np.diff(p["poff"]) == (counts + 127) // 128 * 128)
    assert np.all(p["poff"] % 128 == 0)
    flat = p["dst_of"].reshape(-1)
    assert np.array_equal(np.sort(flat), np.arange(T * k))
    assert np.all(p["src_row"][flat] == np.arange(T * k) // k)


def test_invalid_ids_are_dropped():
    ids = np.array([[0, 5], [-1, 1], [1, 0]], np.int32)
    p = oracle.permute(ids, 2)
    assert p["bad"] == 2
    assert list(p["counts"]) == [2, 2]
    assert p["dst_of"][0, 1] == -1 and p["dst_of"][1, 0] == -1
    assert list(p["src_row"]) == [0, 2, 1, 2]


def test_gather_rows():
    src = np.arange(5 * 7, dtype=np.uint8).reshape(5, 7)
    out = oracle.gather_rows(src, [4, 0, 0, 2])
    assert np.array_equal(out, src[[4, 0, 0, 2]])
