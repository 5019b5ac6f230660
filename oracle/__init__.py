"""CPU oracle for the MXFP8 MoE hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product path.

The arithmetic lives in ``mx_oracle.c`` (plain C, double precision).  This
module only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  Every function names the passage it follows; see the C file for the
definitions and the list of pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmxoracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile mx_oracle.c into libmxoracle.so with gcc (no fast-math, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int32
        sig = {
            "orc_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e8m0_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_e4m3_encode_brute": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_check_encoders": (i64, [ctypes.c_int, ctypes.c_int, P, P]),
            "orc_e4m3_encode_array": (None, [P, i64, P]),
            "orc_e4m3_decode_array": (None, [P, i64, P]),
            "orc_mx_block": (ctypes.c_uint8, [P, ctypes.c_int, P]),
            "orc_quantize_rowwise": (None, [P, i64, i64, P, P]),
            "orc_quantize_colwise_seg": (None, [P, i64, i64, P, P, ctypes.c_int, i64, P, P]),
            "orc_place_sf_rows": (None, [P, i64, P, P, ctypes.c_int, P]),
            "orc_sf_to_tcgen05": (None, [P, i64, i64, P]),
            "orc_sf_from_tcgen05": (None, [P, i64, i64, P]),
            "orc_permute": (i64, [P, i64, ctypes.c_int, ctypes.c_int, P, P, P, P, P]),
            "orc_gather_rows": (None, [P, i64, P, i64, P]),
            "orc_gemm_nt": (None, [i64, i64, i64, P, i64, P, i64, P, i64, P, i64, P, i64]),
            "orc_double_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_combine_fwd": (None, [P, P, P, i64, ctypes.c_int, i64, P]),
            "orc_swiglu_fwd": (None, [P, i64, i64, P]),
            "orc_swiglu_bwd": (None, [P, P, i64, i64, P]),
            "orc_mx_block_rule": (ctypes.c_uint8, [P, ctypes.c_int, P, ctypes.c_int]),
            "orc_quantize_rowwise_ex": (None, [P, ctypes.c_int, i64, i64, ctypes.c_int, P, P]),
            "orc_quantize_colwise_seg_ex": (None, [P, ctypes.c_int, i64, i64, P, P, ctypes.c_int, i64, ctypes.c_int,
                                                   P, P]),
            "orc_combine_bwd": (None, [P, P, P, P, i64, ctypes.c_int, i64, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _ = i32
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- element formats --------------------------------------------------------

def e4m3_encode(v) -> np.ndarray:
    v = _c(v, np.float64).reshape(-1)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def e4m3_encode_brute(v) -> np.ndarray:
    v = _c(v, np.float64).reshape(-1)
    return np.array([lib().orc_e4m3_encode_brute(float(x)) for x in v], np.uint8)


def e4m3_decode(c) -> np.ndarray:
    c = _c(c, np.uint8).reshape(-1)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e8m0_decode(b: int) -> float:
    return lib().orc_e8m0_decode(int(b))


def bf16_to_double(h) -> np.ndarray:
    h = _c(h, np.uint16).reshape(-1)
    return np.array([lib().orc_bf16_to_double(int(x)) for x in h], np.float64)


def check_encoders(shift_lo: int, shift_hi: int):
    fb = ctypes.c_int32(0)
    fs = ctypes.c_int32(0)
    bad = lib().orc_check_encoders(shift_lo, shift_hi, ctypes.byref(fb), ctypes.byref(fs))
    return int(bad), int(fb.value), int(fs.value)


def mx_block(x) -> tuple[int, np.ndarray]:
    """One MX block (<= 32 values, given as doubles): returns (scale byte, E4M3 codes)."""
    x = _c(x, np.float64).reshape(-1)
    assert x.size <= 32
    q = np.empty(x.size, np.uint8)
    b = lib().orc_mx_block(_p(x), int(x.size), _p(q))
    return int(b), q


# --- quantization -------------------------------------------------------------

def quantize_rowwise(x_bits: np.ndarray):
    """Rowwise MX quantization of bf16 bits [rows, cols] -> (q [rows, cols], sf row-major [rows, cols/32])."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    assert cols % 32 == 0
    q = np.empty((rows, cols), np.uint8)
    sf = np.empty((rows, cols // 32), np.uint8)
    lib().orc_quantize_rowwise(_p(x), rows, cols, _p(q), _p(sf))
    return q, sf


def quantize_colwise_seg(x_bits: np.ndarray, off, poff, ld: int):
    """Columnwise MX quantization over segments -> (q [cols, ld], sf row-major [cols, ld/32]).

    Positions at or past poff[-1] are left as 0 in the returned arrays."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    off = _c(off, np.int32)
    poff = _c(poff, np.int32)
    nseg = off.size - 1
    assert ld % 128 == 0 and ld >= int(poff[-1])
    q = np.zeros((cols, ld), np.uint8)
    sf = np.zeros((cols, ld // 32), np.uint8)
    lib().orc_quantize_colwise_seg(_p(x), rows, cols, _p(off), _p(poff), nseg, ld, _p(q), _p(sf))
    return q, sf


def place_sf_rows(sf_dense: np.ndarray, off, poff):
    sf_dense = _c(sf_dense, np.uint8)
    kb = sf_dense.shape[1]
    off = _c(off, np.int32)
    poff = _c(poff, np.int32)
    out = np.zeros((int(poff[-1]), kb), np.uint8)
    lib().orc_place_sf_rows(_p(sf_dense), kb, _p(off), _p(poff), off.size - 1, _p(out))
    return out


def sf_to_tcgen05(sf_rm: np.ndarray) -> np.ndarray:
    sf_rm = _c(sf_rm, np.uint8)
    rows, kb = sf_rm.shape
    n = ((rows + 127) // 128 * 128) * ((kb + 3) // 4 * 4)
    out = np.empty(n, np.uint8)
    lib().orc_sf_to_tcgen05(_p(sf_rm), rows, kb, _p(out))
    return out


def sf_from_tcgen05(sf_sw: np.ndarray, rows: int, kb: int) -> np.ndarray:
    sf_sw = _c(sf_sw, np.uint8).reshape(-1)
    assert sf_sw.size >= ((rows + 127) // 128 * 128) * ((kb + 3) // 4 * 4)
    out = np.empty((rows, kb), np.uint8)
    lib().orc_sf_from_tcgen05(_p(sf_sw), rows, kb, _p(out))
    return out


# --- permutation --------------------------------------------------------------

def permute(ids: np.ndarray, E: int):
    """Stable counting sort of routed (token, slot) pairs by expert."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    poff = np.empty(E + 1, np.int32)
    n_valid = T * k  # upper bound; trimmed below
    src_row = np.full(max(n_valid, 1), -1, np.int32)
    dst_of = np.empty(T * k, np.int32)
    bad = lib().orc_permute(_p(ids), T, k, E, _p(counts), _p(off), _p(poff), _p(src_row), _p(dst_of))
    return dict(counts=counts, off=off, poff=poff, src_row=src_row[: int(off[-1])].copy(),
                dst_of=dst_of.reshape(T, k), bad=int(bad))


def gather_rows(src: np.ndarray, src_row) -> np.ndarray:
    src = np.ascontiguousarray(src)
    src_row = _c(src_row, np.int32)
    row_bytes = src.strides[0]
    R = src_row.size
    out = np.empty((R,) + src.shape[1:], src.dtype)
    lib().orc_gather_rows(_p(src), row_bytes, _p(src_row), R, _p(out))
    return out


# --- GEMM ---------------------------------------------------------------------

def gemm_nt(qa: np.ndarray, sfa: np.ndarray, qb: np.ndarray, sfb: np.ndarray) -> np.ndarray:
    """fp64 C[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k]; operands are [rows, K] codes with
    row-major scale arrays [rows, K/32]."""
    qa = _c(qa, np.uint8)
    qb = _c(qb, np.uint8)
    sfa = _c(sfa, np.uint8)
    sfb = _c(sfb, np.uint8)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % 32 == 0
    assert sfa.shape == (M, K // 32) and sfb.shape == (N, K // 32)
    c = np.empty((M, N), np.float64)
    lib().orc_gemm_nt(M, N, K, _p(qa), K, _p(sfa), K // 32, _p(qb), K, _p(sfb), K // 32, _p(c), N)
    return c


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float64).reshape(-1)
    return np.array([lib().orc_double_to_bf16(float(x)) for x in v], np.uint16)


# --- combine (unpermute) ------------------------------------------------------

def combine_fwd(Y_bits: np.ndarray, gate: np.ndarray, dst_of: np.ndarray) -> np.ndarray:
    """out[t] = bf16(sum_j gate[t][j] * Y[dst_of[t][j]]) as bf16 bits [T, H]."""
    Y = _c(Y_bits, np.uint16)
    gate = _c(gate, np.float32)
    dst_of = _c(dst_of, np.int32)
    T, k = gate.shape
    H = Y.shape[1]
    out = np.empty((T, H), np.uint16)
    lib().orc_combine_fwd(_p(Y), _p(gate), _p(dst_of), T, k, H, _p(out))
    return out


def combine_bwd(dOut_bits: np.ndarray, Y_bits: np.ndarray, gate: np.ndarray, dst_of: np.ndarray):
    """(dY bf16 bits [R, H] for the routed rows, dgate float64 [T, k]); rows of dY that no
    (t, j) maps to are left as 0."""
    dOut = _c(dOut_bits, np.uint16)
    Y = _c(Y_bits, np.uint16)
    gate = _c(gate, np.float32)
    dst_of = _c(dst_of, np.int32)
    T, k = gate.shape
    H = Y.shape[1]
    dY = np.zeros(Y.shape, np.uint16)
    dgate = np.empty((T, k), np.float64)
    lib().orc_combine_bwd(_p(dOut), _p(Y), _p(gate), _p(dst_of), T, k, H, _p(dY), _p(dgate))
    return dY, dgate


# --- scale-rule / input-type variants ----------------------------------------
RULE_FLOOR, RULE_RCEIL = 0, 1


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return 0
    if x.dtype == np.float32:
        return 1
    raise TypeError("bf16 bits (uint16) or float32 expected")


def mx_block_rule(x, rule: int):
    x = _c(x, np.float64).reshape(-1)
    q = np.empty(x.size, np.uint8)
    b = lib().orc_mx_block_rule(_p(x), int(x.size), _p(q), int(rule))
    return int(b), q


def quantize_rowwise_ex(x: np.ndarray, rule: int = RULE_FLOOR):
    """Rowwise MX quantization of bf16 bits (uint16) or float32 [rows, cols]."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sf = np.empty((rows, cols // 32), np.uint8)
    lib().orc_quantize_rowwise_ex(_p(x), _dtype_code(x), rows, cols, int(rule), _p(q), _p(sf))
    return q, sf


def quantize_colwise_seg_ex(x: np.ndarray, off, poff, ld: int, rule: int = RULE_FLOOR):
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    off = _c(off, np.int32)
    poff = _c(poff, np.int32)
    q = np.zeros((cols, ld), np.uint8)
    sf = np.zeros((cols, ld // 32), np.uint8)
    lib().orc_quantize_colwise_seg_ex(_p(x), _dtype_code(x), rows, cols, _p(off), _p(poff), off.size - 1, ld,
                                      int(rule), _p(q), _p(sf))
    return q, sf


# --- SwiGLU (the fused quantizing kernels' elementwise step) -------------------

def swiglu_fwd(a_bits: np.ndarray) -> np.ndarray:
    """h = silu(gate) * up in double, rounded once to fp32; a = [gate | up] bf16 bits [R, 2I]."""
    a = _c(a_bits, np.uint16)
    R, I2 = a.shape
    h = np.empty((R, I2 // 2), np.float32)
    lib().orc_swiglu_fwd(_p(a), R, I2 // 2, _p(h))
    return h


def swiglu_bwd(dh_bits: np.ndarray, a_bits: np.ndarray) -> np.ndarray:
    """[dgate | dup] fp32 [R, 2I] for output gradient dh bf16 bits [R, I]."""
    a = _c(a_bits, np.uint16)
    dh = _c(dh_bits, np.uint16)
    R, I2 = a.shape
    out = np.empty((R, I2), np.float32)
    lib().orc_swiglu_bwd(_p(dh), _p(a), R, I2 // 2, _p(out))
    return out
