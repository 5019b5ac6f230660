"""The fused SwiGLU kernels' quantized outputs against the oracle, with differences allowed only
where near_tie explains them (shared by the standalone and the GEMM-epilogue SwiGLU tests)."""
import numpy as np

import oracle
from gpu_util import np_, sf_x4_first
from near_tie import check_blocks, swiglu_bounds


def _vals(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def check_swiglu_outputs(bwd, a_bits, dh_bits, off, poff, q_row, sf_row, q_col, sf_col, x4=(False, False)):
    """The kernel's rowwise and columnwise outputs (device tensors) against the oracle's SwiGLU
    of the same inputs, differences only where explained by the kernel's error bound."""
    counts = np.diff(off)
    E = len(counts)
    R, I2 = a_bits.shape
    I = I2 // 2
    cols = 2 * I if bwd else I
    g, u = _vals(a_bits[:, :I]), _vals(a_bits[:, I:])
    if bwd:
        ref32 = oracle.swiglu_bwd(dh_bits, a_bits)
        b_dg, b_du = swiglu_bounds(g, u, _vals(dh_bits))
        bound = np.concatenate([b_dg, b_du], axis=1)
    else:
        ref32 = oracle.swiglu_fwd(a_bits)
        bound = swiglu_bounds(g, u)
    v = ref32.astype(np.float64)
    P = int(poff[-1])
    pb = q_col.shape[1]
    srow = sf_x4_first(sf_row) if x4[0] else np_(sf_row)
    scol = sf_x4_first(sf_col, pb // 128, -(-P // 128)) if x4[1] else np_(sf_col)
    rows_pad = np.concatenate([np.arange(poff[e], poff[e] + counts[e]) for e in range(E)]).astype(np.int64)
    sf_rm = oracle.sf_from_tcgen05(srow, max(P, 1), cols // 32)
    n_row = check_blocks(v, bound, np_(q_row)[:R], sf_rm[rows_pad])
    vc = np.zeros((cols, P))
    bc = np.zeros((cols, P))
    vc[:, rows_pad] = v.T
    bc[:, rows_pad] = bound.T
    got_sf = oracle.sf_from_tcgen05(scol, cols, pb // 32)
    n_col = check_blocks(vc, bc, np_(q_col)[:, :P], got_sf[:, : P // 32])
    return n_row, n_col
